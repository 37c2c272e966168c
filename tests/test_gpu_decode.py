"""GPU parity of kivi_decode_attn against the oracle's fp64 attention over the
same cache: max |out - oracle| <= 2e-3 over every output element, for both code
widths, both dtypes, GQA groups 1/2/4/8, the length edge cases of the packed /
residual split, varlen batches and the split-K combine."""
import math

import numpy as np
import pytest
import torch

import bit_asymmetric_kv_kivi_gb300 as kivi
import oracle
import synth
from gpu_util import ATTN_TOL, assert_state_equal, configs, dev_tensor, record_error

pytestmark = pytest.mark.gpu


def build(wl: synth.Workload, bits: int, cap: int):
    """Library and oracle caches of workload `wl` (every sequence prefilled to its length)."""
    kcfg, ocfg = configs(bits, wl.dtype, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.residual)
    cache = kivi.KVCache(kcfg, wl.batch, cap)
    refs, ks, vs = [], [], []
    for b in range(wl.batch):
        K, V = wl.kv_seq(b, 0, wl.lengths[b])
        ks.append(dev_tensor(K, wl.dtype))
        vs.append(dev_tensor(V, wl.dtype))
        r = oracle.SeqCache(ocfg, cap)
        assert r.append(K, V) == oracle.OK
        refs.append(r)
    cache.append(ks, vs)
    return cache, refs


def check_decode(wl, cache, refs, step=0, max_kv_len=None, heads=None):
    q = wl.query(step)
    out = cache.decode(dev_tensor(q, wl.dtype), softmax_scale=wl.softmax_scale, max_kv_len=max_kv_len)
    out = out.cpu().numpy()
    assert int(cache.status.item()) == 0
    worst = 0.0
    for b, r in enumerate(refs):
        if heads is None:
            want = r.decode(q[b], wl.softmax_scale)
            err = np.max(np.abs(out[b] - want))
        else:
            want = r.decode(q[b], wl.softmax_scale, heads[0], heads[1])
            err = np.max(np.abs(out[b, heads[0]:heads[0] + heads[1]] - want[heads[0]:heads[0] + heads[1]]))
        worst = max(worst, float(err))
    record_error(worst)
    assert worst <= ATTN_TOL, worst
    return out, worst


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_decode_edge_lengths(bits, dtype, g):
    """One batch holding the edge lengths of the packed/residual split."""
    lengths = (1, 5, 31, 32, 33, 127, 128, 129, 159, 160, 161, 191, 300, 1000)
    H = 2
    wl = synth.Workload("edges", len(lengths), H * g, H, 128, lengths, dtype, bits=bits,
                        seed=500 + g + bits)
    cache, refs = build(wl, bits, 1024)
    for b, r in enumerate(refs):
        assert_state_equal(cache, b, r)
    check_decode(wl, cache, refs)


def test_decode_empty_sequence_gives_zeros():
    wl = synth.Workload("empty", 3, 4, 2, 128, (0, 200, 0), "f16", seed=7)
    cache, refs = build(wl, 2, 256)
    out, _ = check_decode(wl, cache, refs)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_split_count_invariance(dtype):
    """The same sequences give the same attention however the work is cut: alone, next
    to each other, or behind other sequences that move the CTA boundaries (query group
    4, persistent schedule); and with different split sizes (query group 8, whose split
    size follows max_kv_len). Agreement to 1e-4: the f16 hi+lo operands carry ~22 bits with an
    absolute floor of 2^-25 on subnormal low parts, and each part's running max changes
    which terms sit at that floor."""
    lens = (9000, 5000)
    base = synth.Workload("splits", 2, 8, 2, 128, lens, dtype, seed=8)
    kcfg, ocfg = configs(2, dtype, 8, 2)
    kv = [base.kv_seq(i, 0, lens[i]) for i in range(2)]
    refs = []
    for K, V in kv:
        r = oracle.SeqCache(ocfg, 20000)
        assert r.append(K, V) == oracle.OK
        refs.append(r)
    q0 = base.query(0)
    outs = []
    for pad in ((), (3000,), (700, 20000, 64)):
        padw = synth.Workload("pad", max(len(pad), 1), 8, 2, 128, pad or (1,), dtype, seed=9)
        kvp = [padw.kv_seq(i, 0, pad[i]) for i in range(len(pad))] + kv
        cache = kivi.KVCache(kcfg, len(kvp), 20000)
        cache.append([dev_tensor(K, dtype) for K, _ in kvp], [dev_tensor(V, dtype) for _, V in kvp])
        q = np.concatenate([padw.query(0)[:len(pad)], q0]) if pad else q0
        out = cache.decode(dev_tensor(q, dtype), softmax_scale=base.softmax_scale).cpu().numpy()[len(pad):]
        assert int(cache.status.item()) == 0
        for i, r in enumerate(refs):
            err = float(np.max(np.abs(out[i] - r.decode(q0[i], base.softmax_scale))))
            record_error(err)
            assert err <= ATTN_TOL, err
        outs.append(out)
    assert np.max(np.abs(outs[0] - outs[1])) <= 1e-4 and np.max(np.abs(outs[0] - outs[2])) <= 1e-4
    wl = synth.Workload("splits8", 2, 16, 2, 128, lens, dtype, seed=8)
    cache, refs = build(wl, 2, 9024)
    a, _ = check_decode(wl, cache, refs, max_kv_len=9000)          # 1280-token splits
    b, _ = check_decode(wl, cache, refs, max_kv_len=400000)        # 4096-token splits
    c, _ = check_decode(wl, cache, refs, max_kv_len=24000)         # 3072-token splits
    assert np.max(np.abs(a - b)) <= 1e-4 and np.max(np.abs(a - c)) <= 1e-4


def test_gqa_equals_repeated_mha():
    """Hq/Hkv = 4 over a cache equals MHA over the same cache with each kv head repeated 4 times."""
    wl = synth.Workload("gqa", 2, 8, 2, 128, (700, 450), "f16", seed=9)
    cache, refs = build(wl, 2, 640)
    q = dev_tensor(wl.query(0), "f16")
    out_gqa = cache.decode(q, softmax_scale=wl.softmax_scale)
    kcfg = kivi.Config(bits=2, num_q_heads=8, num_kv_heads=8, dtype=kivi.F16)
    mha = kivi.KVCache(kcfg, 2, 640)
    ks, vs = [], []
    for b in range(2):
        K, V = wl.kv_seq(b, 0, wl.lengths[b])
        ks.append(dev_tensor(np.repeat(K, 4, axis=0), "f16"))
        vs.append(dev_tensor(np.repeat(V, 4, axis=0), "f16"))
    mha.append(ks, vs)
    out_mha = mha.decode(q, softmax_scale=wl.softmax_scale)
    # the same arithmetic per head, up to the power-of-two q prescale chosen per CTA
    assert float((out_gqa - out_mha).abs().max()) <= 2e-5


def test_bad_length_gives_nan_and_status():
    wl = synth.Workload("bad", 2, 2, 1, 128, (300, 100), "f16", seed=10)
    cache, refs = build(wl, 2, 256)
    q = dev_tensor(wl.query(0), "f16")
    out = cache.decode(q, softmax_scale=wl.softmax_scale, max_kv_len=200).cpu().numpy()
    assert int(cache.status.item()) == kivi.ERR_LENGTH
    assert np.all(np.isnan(out[0]))
    want = refs[1].decode(wl.query(0)[1], wl.softmax_scale)
    assert np.max(np.abs(out[1] - want)) <= ATTN_TOL


def test_workload_tiny_decode():
    """Workload 0 (one sequence, one head, 1024 tokens: 28 key groups + 128 residual)."""
    wl = synth.workload(0)
    cache, refs = build(wl, 2, 1024)
    assert oracle.n_packed(refs[0].cfg, 1024) == 896
    assert_state_equal(cache, 0, refs[0])
    check_decode(wl, cache, refs)


def test_workload_llama2_7b_mha():
    """Workload 1 at full size: 8 sequences, 32 heads (MHA), 4096 tokens, fp16."""
    wl = synth.workload(1)
    cache, refs = build(wl, 2, 4096)
    for b in (0, 7):
        assert_state_equal(cache, b, refs[b])
    check_decode(wl, cache, refs)


@pytest.mark.parametrize("g", [1, 4, 8])
@pytest.mark.parametrize("shape", ["short", "one_long"])
def test_many_streams_persistent_schedule(g, shape):
    """Hundreds of sequences (more than one per scan thread) of mixed lengths: empty ones,
    residual-only ones, a few groups; in "one_long" also one 20000-token sequence, so
    that one stream spans many CTAs while single CTAs hold many short streams (with a
    query group of 8, two streams of four heads per kv head)."""
    rng = np.random.default_rng(900 + g)
    n = 300
    lengths = rng.integers(0, 700, size=n)
    lengths[rng.random(n) < 0.1] = 0
    short = rng.random(n) < 0.2
    lengths[short] = rng.integers(1, 160, size=int(short.sum()))          # residual-only
    lengths[:6] = (0, 1, 159, 160, 161, 192)
    if shape == "one_long":
        lengths[137] = 20000
    H = 2
    wl = synth.Workload("streams", n, g * H, H, 128, tuple(int(x) for x in lengths), "f16", seed=31 + g)
    cap = ((int(lengths.max()) + 31) // 32) * 32
    cache, refs = build(wl, 2, cap)
    out, _ = check_decode(wl, cache, refs)
    assert np.all(out[lengths == 0] == 0)


@pytest.mark.parametrize("g", [3, 5, 6, 16, 32])
@pytest.mark.parametrize("bits", [2, 4])
def test_decode_any_query_group(g, bits):
    """Query groups other than 1, 2, 4 (up to 32) run on the multi-query kernel with one
    query, its virtual heads padded to whole warps of four."""
    lengths = (0, 1, 33, 160, 161, 700, 3000)
    H = 2
    dtype = "bf16" if g % 2 else "f16"
    wl = synth.Workload("anyg", len(lengths), H * g, H, 128, lengths, dtype, bits=bits, seed=700 + g + bits)
    cache, refs = build(wl, bits, 3008)
    out, _ = check_decode(wl, cache, refs)
    assert np.all(out[0] == 0)
