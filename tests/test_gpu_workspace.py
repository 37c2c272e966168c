"""One workspace shared by attention calls of different sizes.

include/kivi.h promises that every decode or multi-query call leaves its workspace
all zero again (split tickets reset, merged partial records cleared), so a caller can
keep one buffer for calls whose sequence counts, kv-head counts and query counts
differ. These tests run a small call, then larger ones, on one buffer, check every
output against the oracle and check that the buffer is all zero after each call.
"""
import numpy as np
import pytest
import torch

import bit_asymmetric_kv_kivi_gb300 as kivi
import oracle
import synth
from gpu_util import ATTN_TOL, configs, dev_tensor, record_error

pytestmark = pytest.mark.gpu


def _cache(nseq, hq, h, lengths, dtype, seed):
    wl = synth.Workload("ws", nseq, hq, h, 128, tuple(lengths), dtype, seed=seed)
    kcfg, ocfg = configs(2, dtype, hq, h)
    cap = (max(lengths) // 32 + 2) * 32
    cache = kivi.KVCache(kcfg, nseq, cap)
    refs = []
    ks, vs = [], []
    for b in range(nseq):
        K, V = wl.kv_seq(b, 0, lengths[b])
        ks.append(dev_tensor(K, dtype))
        vs.append(dev_tensor(V, dtype))
        ref = oracle.SeqCache(ocfg, cap)
        assert ref.append(K, V) == oracle.OK
        refs.append(ref)
    cache.append(ks, vs)
    return wl, cache, refs


def _check_decode(wl, cache, refs, ws):
    cache._ws = ws
    q = wl.query(0)
    out = cache.decode(dev_tensor(q, wl.dtype), softmax_scale=wl.softmax_scale).cpu().numpy()
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    assert int(torch.count_nonzero(ws).item()) == 0, "workspace not all zero after the call"
    err = max(float(np.max(np.abs(out[b] - refs[b].decode(q[b], wl.softmax_scale)))) for b in range(cache.nseq))
    record_error(err)
    assert err <= ATTN_TOL, err


def _check_multi(wl, cache, refs, ws, nq):
    cache._ws = ws
    qm = np.stack([wl.query(1 + i) for i in range(nq)], axis=1)          # [nseq][nq][Hq][D]
    out = cache.decode_multi(dev_tensor(qm, wl.dtype), softmax_scale=wl.softmax_scale).cpu().numpy()
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    assert int(torch.count_nonzero(ws).item()) == 0, "workspace not all zero after the call"
    err = max(float(np.max(np.abs(out[b] - refs[b].decode_multi(qm[b], wl.softmax_scale))))
              for b in range(cache.nseq))
    record_error(err)
    assert err <= ATTN_TOL, err


@pytest.mark.parametrize("g_small,g_large", [(4, 4), (4, 8), (1, 6)])
def test_small_then_larger_calls_share_one_workspace(g_small, g_large):
    small = _cache(2, 2 * g_small, 2, (3000, 700), "f16", seed=91)
    large = _cache(6, 8 * g_large, 8, (5000, 129, 2600, 40, 9000, 1200), "f16", seed=92)
    need = max(small[1].cfg.decode_workspace_bytes(2, small[1].max_len),
               large[1].cfg.decode_workspace_bytes(6, large[1].max_len),
               large[1].cfg.decode_multi_workspace_bytes(6, 2, large[1].max_len),
               small[1].cfg.decode_multi_workspace_bytes(2, 3, small[1].max_len))
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    for _ in range(2):
        _check_decode(*small, ws)           # fewer sequences and kv heads: records end early
        _check_decode(*large, ws)           # more streams: tickets reach past the small call's tickets
        _check_multi(*large, ws, 2)
        _check_multi(*small, ws, 3)
