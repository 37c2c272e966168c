"""GPU parity of the paged layout (kivi.h: packed groups in a shared pool of 32-token
pages behind per-sequence block tables). The same appends on a contiguous and a paged
cache (pages handed out in a random order, spare pages filled with a sentinel) must give
the same packed state, gathered through the tables, bit for bit, and the same decode
output bit for bit, which the oracle checks to 2e-3; no page outside the tables is
written."""
import numpy as np
import pytest
import torch

import bit_asymmetric_kv_kivi_gb300 as kivi
import oracle
import synth
from gpu_util import ATTN_TOL, assert_state_equal, configs, dev_tensor, record_error

pytestmark = pytest.mark.gpu


def pair(kcfg, nseq, cap, spare=5):
    cont = kivi.KVCache(kcfg, nseq, cap)
    paged = kivi.KVCache(kcfg, nseq, cap, paged=True, page_seed=nseq + cap, spare_pages=spare)
    for name in ("k_codes", "v_codes"):
        getattr(paged, name).fill_(0xAB)
    for name in ("k_scale", "k_zero", "v_scale", "v_zero"):
        getattr(paged, name).fill_(-21555)          # 0xABCD
    return cont, paged


def spare_pages(cache):
    used = set(cache.block_tables.cpu().numpy().ravel().tolist())
    return [p for p in range(cache.k_codes.shape[0]) if p not in used]


def assert_spares_untouched(cache):
    for p in spare_pages(cache):
        assert torch.all(cache.k_codes[p] == 0xAB) and torch.all(cache.v_codes[p] == 0xAB)
        assert torch.all(cache.k_scale[p] == -21555) and torch.all(cache.v_zero[p] == -21555)


def assert_same_state(a, b, nseq):
    for s in range(nseq):
        x, y = a.seq_numpy(s), b.seq_numpy(s)
        L = x["kv_len"]
        assert L == y["kv_len"]
        P = (max(L - 128, 0) // 32) * 32
        for name in ("k_codes", "v_codes", "v_scale", "v_zero"):
            assert np.array_equal(x[name][:, :P], y[name][:, :P]), (s, name)
        for name in ("k_scale", "k_zero"):
            assert np.array_equal(x[name][:, :P // 32], y[name][:, :P // 32]), (s, name)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("g", [4, 8])
def test_paged_equals_contiguous(bits, dtype, g):
    H = 2
    lengths = (0, 1, 160, 161, 700, 2000)
    wl = synth.Workload("paged", len(lengths), g * H, H, 128, lengths, dtype, seed=40 + g)
    kcfg, ocfg = configs(bits, dtype, g * H, H)
    cap = 2048
    cont, paged = pair(kcfg, wl.batch, cap)
    refs = []
    ks, vs = [], []
    for b, L in enumerate(lengths):
        K, V = wl.kv_seq(b, 0, L)
        ks.append(dev_tensor(K, dtype))
        vs.append(dev_tensor(V, dtype))
        r = oracle.SeqCache(ocfg, cap)
        assert r.append(K, V) == oracle.OK
        refs.append(r)
    cont.append(ks, vs)
    paged.append(ks, vs)
    torch.cuda.synchronize()
    assert int(paged.status.item()) == 0
    assert_same_state(cont, paged, wl.batch)
    for b in (3, 4, 5):
        assert_state_equal(paged, b, refs[b])
    assert_spares_untouched(paged)
    # streaming: 40 one-token steps (one flush boundary for every sequence), decode each time
    for s in range(40):
        kn, vn = [], []
        for b, L in enumerate(lengths):
            K, V = wl.kv_seq(b, L + s, 1)
            kn.append(dev_tensor(K, dtype))
            vn.append(dev_tensor(V, dtype))
            if b in (3, 5):
                assert refs[b].append(K, V) == oracle.OK
        cont.append(kn, vn)
        paged.append(kn, vn)
        q = wl.query(s)
        qd = dev_tensor(q, dtype)
        oc = cont.decode(qd, softmax_scale=wl.softmax_scale).cpu().numpy()
        op = paged.decode(qd, softmax_scale=wl.softmax_scale).cpu().numpy()
        assert np.array_equal(oc, op), s
        if s % 13 == 0 or s == 39:
            for b in (3, 5):
                err = float(np.max(np.abs(op[b] - refs[b].decode(q[b], wl.softmax_scale))))
                record_error(err)
                assert err <= ATTN_TOL, err
    torch.cuda.synchronize()
    assert int(paged.status.item()) == 0
    assert_same_state(cont, paged, wl.batch)
    assert_spares_untouched(paged)
