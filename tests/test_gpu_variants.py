"""GPU parity of the configuration variants: G = 64 with R = 64 or 128 (the config
example in "KV-Cache Quantization: I Ran the Experiments So You Don't Have To",
section "Component 4"), and key and value code widths set apart (k_bits != v_bits).
Codec and cache state bit-exact against the oracle, decode attention within 2e-3 for
every query group (tensor-core kernel for 1, 2, 4; CUDA-core kernel for 8), and the
paged layout with 64-token pages equal to the contiguous one."""
import numpy as np
import pytest
import torch

import bit_asymmetric_kv_kivi_gb300 as kivi
import oracle
import synth
from gpu_util import ATTN_TOL, assert_state_equal, configs, dev_tensor, host_bits, record_error

pytestmark = pytest.mark.gpu

# (k_bits, v_bits, G, R)
VARIANTS = [(2, 2, 64, 64), (4, 4, 64, 64), (2, 4, 32, 128), (4, 2, 32, 64), (2, 4, 64, 128), (4, 2, 64, 64)]
IDS = [f"k{kb}v{vb}-G{G}-R{R}" for kb, vb, G, R in VARIANTS]


def edge_lengths(G, R):
    """Lengths around every boundary of the packed / residual split for (G, R)."""
    base = {0, 1, 31, 32, 33, G - 1, G, G + 1, R - 1, R, R + 1, R + G - 1, R + G, R + G + 1,
            R + 2 * G - 1, R + 2 * G, R + 2 * G + 1, 1000, 1000 + G // 2}
    return tuple(sorted(x for x in base if x >= 0))


@pytest.mark.parametrize("kb,vb", [(2, 4), (4, 2)])
@pytest.mark.parametrize("G", [32, 64])
def test_codec_widths_apart(kb, vb, G):
    """kivi_quant_keys codes at k_bits and kivi_quant_values at v_bits, bit-exact."""
    rng = np.random.default_rng(70 + kb + G)
    S, T, D = 2, 3 * G, 128
    kcfg, ocfg = configs(2, "bf16", 1, 1, D, G=G, kb=kb, vb=vb)
    x = rng.standard_normal((S, T, D))
    x[:, :, :3] *= 20
    xb = synth.to_dtype_bits(x, "bf16")
    codes, scale, zero = kivi.quant_keys(kcfg, dev_tensor(xb, "bf16"))
    rc, rs, rz = oracle.quant_keys(ocfg, xb)
    assert codes.shape[-1] == D * kb // 8
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
    np.testing.assert_array_equal(host_bits(scale), rs)
    np.testing.assert_array_equal(host_bits(zero), rz)
    codes, scale, zero = kivi.quant_values(kcfg, dev_tensor(xb, "bf16"))
    rc, rs, rz = oracle.quant_values(ocfg, xb)
    assert codes.shape[-1] == D * vb // 8
    np.testing.assert_array_equal(codes.cpu().numpy(), rc)
    np.testing.assert_array_equal(host_bits(scale), rs)
    np.testing.assert_array_equal(host_bits(zero), rz)


@pytest.mark.parametrize("kb,vb,G,R", VARIANTS, ids=IDS)
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_then_streaming_bitexact(kb, vb, G, R, dtype):
    """A varlen prefill at every edge length, then one-token and chunked appends across
    several flushes, the packed state compared with the oracle after each append."""
    H = 2
    lengths = edge_lengths(G, R)
    wl = synth.Workload("variants", len(lengths), 2 * H, H, 128, lengths, dtype, seed=80 + kb + 3 * vb + G + R)
    kcfg, ocfg = configs(2, dtype, 2 * H, H, G=G, R=R, kb=kb, vb=vb)
    cap = 2048
    cache = kivi.KVCache(kcfg, wl.batch, cap)
    refs, ks, vs = [], [], []
    for b, L in enumerate(lengths):
        K, V = wl.kv_seq(b, 0, L)
        ks.append(dev_tensor(K, dtype))
        vs.append(dev_tensor(V, dtype))
        r = oracle.SeqCache(ocfg, cap)
        assert r.append(K, V) == oracle.OK
        refs.append(r)
    cache.append(ks, vs)
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    for b in range(wl.batch):
        assert_state_equal(cache, b, refs[b])
    rng = np.random.default_rng(G + R)
    pos = list(lengths)
    for step in range(G + 5 + 12):               # at most 1032 + G + 5 + 12 (G + 8) tokens: within cap
        n = [1 if step < G + 5 else int(rng.integers(0, G + 9)) for _ in range(wl.batch)]
        kn, vn = [], []
        for b in range(wl.batch):
            K, V = wl.kv_seq(b, pos[b], n[b])
            kn.append(dev_tensor(K, dtype))
            vn.append(dev_tensor(V, dtype))
            assert refs[b].append(K, V) == oracle.OK
            pos[b] += n[b]
        cache.append(kn, vn)
        if step % 16 == 0 or step >= G + 5:
            torch.cuda.synchronize()
            for b in (0, 7, wl.batch - 1):
                assert_state_equal(cache, b, refs[b])
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    for b in range(wl.batch):
        assert_state_equal(cache, b, refs[b])


@pytest.mark.parametrize("kb,vb,G,R", VARIANTS, ids=IDS)
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_decode_edge_lengths(kb, vb, G, R, g):
    dtype = ("f16", "bf16")[(VARIANTS.index((kb, vb, G, R)) + g) % 2]
    H = 2
    lengths = edge_lengths(G, R)
    wl = synth.Workload("variants", len(lengths), g * H, H, 128, lengths, dtype, seed=90 + g + kb + 3 * vb + G)
    kcfg, ocfg = configs(2, dtype, g * H, H, G=G, R=R, kb=kb, vb=vb)
    cap = 1024
    cache = kivi.KVCache(kcfg, wl.batch, cap)
    refs, ks, vs = [], [], []
    for b, L in enumerate(lengths):
        K, V = wl.kv_seq(b, 0, L)
        ks.append(dev_tensor(K, dtype))
        vs.append(dev_tensor(V, dtype))
        r = oracle.SeqCache(ocfg, cap)
        assert r.append(K, V) == oracle.OK
        refs.append(r)
    cache.append(ks, vs)
    q = wl.query(0)
    out = cache.decode(dev_tensor(q, dtype), softmax_scale=wl.softmax_scale).cpu().numpy()
    assert int(cache.status.item()) == 0
    worst = 0.0
    for b, r in enumerate(refs):
        worst = max(worst, float(np.max(np.abs(out[b] - r.decode(q[b], wl.softmax_scale)))))
    record_error(worst)
    assert worst <= ATTN_TOL, worst
    assert np.all(out[lengths.index(0)] == 0)


@pytest.mark.parametrize("kb,vb,G,R", [(2, 2, 64, 64), (4, 2, 64, 128)])
@pytest.mark.parametrize("g", [4, 8])
def test_paged_64_token_pages(kb, vb, G, R, g):
    """Paged layout with G-token pages in a random order: the same packed state and the
    same decode output as the contiguous layout, bit for bit; spare pages untouched."""
    dtype, H = "f16", 2
    lengths = (0, 1, 2 * G + R, 700, 1500)
    wl = synth.Workload("paged", len(lengths), g * H, H, 128, lengths, dtype, seed=60 + g + G)
    kcfg, ocfg = configs(2, dtype, g * H, H, G=G, R=R, kb=kb, vb=vb)
    cap = 2048
    cont = kivi.KVCache(kcfg, wl.batch, cap)
    paged = kivi.KVCache(kcfg, wl.batch, cap, paged=True, page_seed=7, spare_pages=3)
    for name in ("k_codes", "v_codes"):
        getattr(paged, name).fill_(0xAB)
    ks, vs, refs = [], [], []
    for b, L in enumerate(lengths):
        K, V = wl.kv_seq(b, 0, L)
        ks.append(dev_tensor(K, dtype))
        vs.append(dev_tensor(V, dtype))
        r = oracle.SeqCache(ocfg, cap)
        assert r.append(K, V) == oracle.OK
        refs.append(r)
    cont.append(ks, vs)
    paged.append(ks, vs)
    for s in range(G + 3):
        kn, vn = [], []
        for b, L in enumerate(lengths):
            K, V = wl.kv_seq(b, L + s, 1)
            kn.append(dev_tensor(K, dtype))
            vn.append(dev_tensor(V, dtype))
            assert refs[b].append(K, V) == oracle.OK
        cont.append(kn, vn)
        paged.append(kn, vn)
    torch.cuda.synchronize()
    assert int(paged.status.item()) == 0
    for b in range(wl.batch):
        assert_state_equal(paged, b, refs[b])
    used = set(paged.block_tables.cpu().numpy().ravel().tolist())
    for p in range(paged.k_codes.shape[0]):
        if p not in used:
            assert torch.all(paged.k_codes[p] == 0xAB) and torch.all(paged.v_codes[p] == 0xAB)
    q = wl.query(1)
    qd = dev_tensor(q, dtype)
    oc = cont.decode(qd, softmax_scale=wl.softmax_scale).cpu().numpy()
    op = paged.decode(qd, softmax_scale=wl.softmax_scale).cpu().numpy()
    assert np.array_equal(oc, op)
    worst = max(float(np.max(np.abs(op[b] - refs[b].decode(q[b], wl.softmax_scale)))) for b in range(wl.batch))
    record_error(worst)
    assert worst <= ATTN_TOL, worst
