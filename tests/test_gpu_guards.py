"""Guard bands around every buffer the kernels write.

compute-sanitizer is not open on this pool, so out-of-bounds writes are caught the plain
way: every device buffer of a small cache (codes, scales, zeros and residual rings of each
sequence, kv_len, the status word, the attention output and the workspace) is a view into a
larger allocation whose margins hold a sentinel byte pattern. Prefill (the multi-launch
append), decode steps across a flush (the one-launch append), decode attention at query
groups 4, 8 and 6 (the persistent kernel, its eight-head form, the multi-query kernel) and
multi-query attention run on it; after each call every margin must still hold the sentinel
and the outputs must match the oracle.
"""
import numpy as np
import pytest
import torch

import bit_asymmetric_kv_kivi_gb300 as kivi
import oracle
import synth
from gpu_util import ATTN_TOL, configs, dev_tensor, record_error

pytestmark = pytest.mark.gpu

GUARD = 256          # bytes of sentinel on each side (keeps every view 256-byte aligned)
SENTINEL = 0xA5


class Guarded:
    """Device buffers carved out of one uint8 allocation, each with sentinel margins."""

    def __init__(self):
        self.regions = []    # (backing tensor, nbytes)

    def alloc(self, shape, dtype):
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        pad = (-nbytes) % 16
        back = torch.full((GUARD + nbytes + pad + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.regions.append((back, nbytes + pad))
        view = back[GUARD:GUARD + nbytes].view(dtype).view(shape)
        view.zero_()
        return view

    def check(self, what):
        torch.cuda.synchronize()
        for i, (back, n) in enumerate(self.regions):
            lo, hi = back[:GUARD], back[GUARD + n:]
            assert bool((lo == SENTINEL).all()), f"{what}: bytes before buffer {i} changed"
            assert bool((hi == SENTINEL).all()), f"{what}: bytes after buffer {i} changed"


def _guarded_cache(cfg, nseq, cap, g):
    """A KVCache whose buffers, kv_len and status are guarded views."""
    cache = kivi.KVCache(cfg, nseq, cap)
    H, D, G = cfg.num_kv_heads, cfg.head_dim, cfg.group
    shapes = {"k_codes": ((H, cap, cfg.k_row_bytes), torch.uint8), "k_scale": ((H, cap // G, D), torch.int16),
              "k_zero": ((H, cap // G, D), torch.int16), "v_codes": ((H, cap, cfg.v_row_bytes), torch.uint8),
              "v_scale": ((H, cap, D // G), torch.int16), "v_zero": ((H, cap, D // G), torch.int16),
              "k_res": ((H, cfg.ring, D), cfg.torch_dtype), "v_res": ((H, cfg.ring, D), cfg.torch_dtype)}
    rec = np.zeros((nseq, kivi.SEQ_STRUCT_BYTES // 8), dtype=np.uint64)
    for b in range(nseq):
        for i, name in enumerate(kivi.SEQ_FIELDS):
            shape, dt = shapes[name]
            rec[b, i] = g.alloc(shape, dt).data_ptr()
        rec[b, 8] = np.uint64(cap)
    cache.seqs = torch.from_numpy(rec.view(np.uint8).reshape(-1)).to("cuda")
    cache.kv_len = g.alloc((nseq,), torch.int32)
    cache.status = g.alloc((1,), torch.int32)
    return cache


@pytest.mark.parametrize("bits", [2, 4])
def test_no_write_outside_any_buffer(bits):
    nseq, H, D = 2, 2, 128
    lengths = (300, 161)
    steps = 40                                            # crosses one flush of each sequence
    cap = 512
    wl = synth.Workload("guards", nseq, 8 * H, H, D, lengths, "f16", seed=95, bits=bits)
    g = Guarded()
    caches, refs = {}, {}
    for gq in (4, 8, 6):
        kcfg, ocfg = configs(bits, "f16", gq * H, H)
        cache = _guarded_cache(kcfg, nseq, cap, g)
        ks, vs, rs = [], [], []
        for b in range(nseq):
            K, V = wl.kv_seq(b, 0, lengths[b])
            ks.append(dev_tensor(K, "f16"))
            vs.append(dev_tensor(V, "f16"))
            r = oracle.SeqCache(ocfg, cap)
            assert r.append(K, V) == oracle.OK
            rs.append(r)
        cache.append(ks, vs)                               # prefill: the multi-launch append
        g.check(f"prefill g={gq}")
        for s in range(steps):                             # decode steps: the one-launch append
            kn, vn = [], []
            for b in range(nseq):
                K, V = wl.kv_seq(b, lengths[b] + s, 1)
                kn.append(dev_tensor(K, "f16"))
                vn.append(dev_tensor(V, "f16"))
                assert rs[b].append(K, V) == oracle.OK
            cache.append(kn, vn)
        g.check(f"decode steps g={gq}")
        assert int(cache.status.item()) == 0
        caches[gq], refs[gq] = (cache, kcfg), rs
    for gq, (cache, kcfg) in caches.items():
        hq = gq * H
        need = max(kcfg.decode_workspace_bytes(nseq, cache.max_len),
                   kcfg.decode_multi_workspace_bytes(nseq, 2 if gq <= 8 else 1, cache.max_len))
        cache._ws = g.alloc((need,), torch.uint8)
        q = np.stack([wl.query(0)[b][:hq] for b in range(nseq)])
        out = g.alloc((nseq, hq, D), torch.float32)
        cache.decode(dev_tensor(q, "f16"), out=out, softmax_scale=wl.softmax_scale)
        g.check(f"decode attention g={gq}")
        got = out.cpu().numpy()
        for b in range(nseq):
            err = float(np.max(np.abs(got[b] - refs[gq][b].decode(q[b], wl.softmax_scale))))
            record_error(err)
            assert err <= ATTN_TOL, err
        nq = 2 if gq * 2 <= 32 else 1
        qm = np.stack([np.stack([wl.query(1 + i)[b][:hq] for i in range(nq)]) for b in range(nseq)])
        outm = g.alloc((nseq, nq, hq, D), torch.float32)
        cache.decode_multi(dev_tensor(qm, "f16"), out=outm, softmax_scale=wl.softmax_scale)
        g.check(f"multi-query attention g={gq}")
        gotm = outm.cpu().numpy()
        for b in range(nseq):
            err = float(np.max(np.abs(gotm[b] - refs[gq][b].decode_multi(qm[b], wl.softmax_scale))))
            record_error(err)
            assert err <= ATTN_TOL, err
        assert int(cache.status.item()) == 0
