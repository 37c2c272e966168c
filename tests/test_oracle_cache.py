"""Pins for the oracle's cache (append + group flush) and its decode attention.

Checks against things other than the oracle itself:
  * the flush schedule against its closed form n_packed(L) = G*floor(max(L-R,0)/G);
  * streaming one token at a time == one bulk append == random chunks (bit-exact);
  * the packed history against the codec entry points run on the same tokens;
  * the residual ring against the raw inputs (slot p mod (R+G));
  * attention against torch.nn.functional.scaled_dot_product_attention in fp64:
    on caches with L <= R (nothing quantized), and on planted-grid caches (every
    packed token decodes exactly), with GQA head mapping;
  * closed-form special cases: L = 1 gives v, identical keys give the mean of V.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from synth import bits_to_f32, to_dtype_bits, workload
from test_oracle_codec import planted_codes


def _rand_kv(rng, H, n, D, dtype="f16"):
    K = rng.standard_normal((H, n, D))
    K[:, :, :3] *= 20
    V = rng.standard_normal((H, n, D))
    V[:, rng.random(n) < 0.03, :] *= 10
    return to_dtype_bits(K, dtype), to_dtype_bits(V, dtype)


# (k_bits, v_bits, G, R): the default setting, the config example of "KV-Cache
# Quantization: I Ran the Experiments So You Don't Have To", section "Component 4"
# (G = R = 64), and mixed widths
VARIANTS = [(2, 2, 32, 128), (4, 4, 32, 128), (2, 2, 64, 64), (4, 2, 32, 64), (2, 4, 64, 128)]


@pytest.mark.parametrize("G,R", [(32, 128), (64, 64), (32, 64), (64, 128)])
def test_flush_schedule_closed_form(oracle_lib, G, R):
    cfg = oracle.Cfg(num_kv_heads=1, head_dim=64, group=G, residual=R)
    rng = np.random.default_rng(1 + G + R)
    s = oracle.SeqCache(cfg, 1024)
    L = 0
    while L < 900:
        n = int(rng.integers(0, 70))
        K, V = _rand_kv(rng, 1, n, 64)
        assert s.append(K, V) == oracle.OK
        L += n
        assert s.L == L
        want = G * (max(L - R, 0) // G)
        assert oracle.n_packed(cfg, L) == want
        r = L - want
        assert (r == L) if L < R else (R <= r <= R + G - 1)


@pytest.mark.parametrize("kb,vb,G,R", VARIANTS)
def test_nothing_packed_beyond_n_packed(oracle_lib, kb, vb, G, R):
    """Groups are packed exactly when the residual reaches R+G: after every append the
    packed buffers hold nothing past n_packed(L) (they keep a sentinel there)."""
    cfg = oracle.Cfg(k_bits=kb, v_bits=vb, num_kv_heads=2, head_dim=64, group=G, residual=R)
    rng = np.random.default_rng(30 + kb + 3 * vb + G + R)
    s = oracle.SeqCache(cfg, 512)
    for name in ("k_codes", "v_codes"):
        getattr(s, name)[...] = 0xAB
    for name in ("k_scale", "k_zero", "v_scale", "v_zero"):
        getattr(s, name)[...] = 0xABCD
    L = 0
    for n in [100, 27, 1, 1, 1, 3, 30, 31, 32, 33, 1, 64, 5, 40] + [1] * 100:
        K, V = _rand_kv(rng, 2, n, 64)
        assert s.append(K, V) == oracle.OK
        L += n
        P = oracle.n_packed(cfg, L)
        assert np.all(s.k_codes[:, P:] == 0xAB) and np.all(s.v_codes[:, P:] == 0xAB)
        assert np.all(s.k_scale[:, P // G:] == 0xABCD) and np.all(s.v_scale[:, P:] == 0xABCD)
        assert not np.all(s.k_codes[:, :P] == 0xAB) or P == 0


@pytest.mark.parametrize("kb,vb,G,R", VARIANTS)
def test_streaming_equals_bulk(oracle_lib, kb, vb, G, R):
    cfg = oracle.Cfg(k_bits=kb, v_bits=vb, num_q_heads=4, num_kv_heads=2, head_dim=64, group=G, residual=R)
    rng = np.random.default_rng(2 + kb + 3 * vb + G + R)
    n = 517
    K, V = _rand_kv(rng, 2, n, 64)
    bulk = oracle.SeqCache(cfg, 512)
    assert bulk.append(K, V) == oracle.OK
    one = oracle.SeqCache(cfg, 512)
    for t in range(n):
        assert one.append(K[:, t:t + 1], V[:, t:t + 1]) == oracle.OK
    chunks = oracle.SeqCache(cfg, 512)
    t = 0
    while t < n:
        m = int(rng.integers(1, 100))
        assert chunks.append(K[:, t:t + m], V[:, t:t + m]) == oracle.OK
        t += min(m, n - t)
    for other in (one, chunks):
        for name in ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero", "k_res", "v_res"):
            assert np.array_equal(getattr(bulk, name), getattr(other, name)), name


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
@pytest.mark.parametrize("kb,vb,G,R", [(2, 2, 32, 128), (2, 4, 64, 64), (4, 2, 64, 128)])
def test_packed_history_matches_codec_and_ring_holds_inputs(oracle_lib, dtype, kb, vb, G, R):
    dt = oracle.BF16 if dtype == "bf16" else oracle.F16
    cfg = oracle.Cfg(k_bits=kb, v_bits=vb, num_q_heads=2, num_kv_heads=2, head_dim=64, dtype=dt, group=G,
                     residual=R)
    rng = np.random.default_rng(5 + G + R)
    n = 450
    K, V = _rand_kv(rng, 2, n, 64, dtype)
    s = oracle.SeqCache(cfg, 384)
    assert s.append(K, V) == oracle.OK
    P = oracle.n_packed(cfg, n)
    assert P == G * ((n - R) // G)
    kc, ks, kz = oracle.quant_keys(cfg, np.ascontiguousarray(K[:, :P]))
    vc, vs, vz = oracle.quant_values(cfg, np.ascontiguousarray(V[:, :P]))
    assert kc.shape[-1] == 64 * kb // 8 and vc.shape[-1] == 64 * vb // 8
    assert np.array_equal(s.k_codes[:, :P], kc) and np.array_equal(s.v_codes[:, :P], vc)
    assert np.array_equal(s.k_scale[:, :P // G], ks) and np.array_equal(s.k_zero[:, :P // G], kz)
    assert np.array_equal(s.v_scale[:, :P], vs) and np.array_equal(s.v_zero[:, :P], vz)
    for p in range(P, n):
        assert np.array_equal(s.k_res[:, p % cfg.ring], K[:, p])
        assert np.array_equal(s.v_res[:, p % cfg.ring], V[:, p])


def test_capacity_overflow_leaves_sequence_unchanged(oracle_lib):
    cfg = oracle.Cfg(num_kv_heads=1, head_dim=32)
    rng = np.random.default_rng(6)
    s = oracle.SeqCache(cfg, 64)
    K, V = _rand_kv(rng, 1, 200, 32)
    assert s.append(K, V) == oracle.OK                       # 64 packed + 136 residual
    before = {k: getattr(s, k).copy() for k in ("k_codes", "k_res", "v_res", "kv_len")}
    K2, V2 = _rand_kv(rng, 1, 30, 32)                          # would need 96 packed
    assert s.append(K2, V2) == oracle.ERR_CAPACITY
    for k, v in before.items():
        assert np.array_equal(getattr(s, k), v)


def _sdpa(q, K, V, scale, g):
    """torch SDPA in fp64: q [Hq][D], K, V [Hkv][L][D] -> [Hq][D]."""
    qt = torch.from_numpy(q)[None, :, None, :]
    Kt = torch.from_numpy(K).repeat_interleave(g, dim=0)[None]
    Vt = torch.from_numpy(V).repeat_interleave(g, dim=0)[None]
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, scale=scale)
    return o[0, :, 0, :].numpy()


@pytest.mark.parametrize("L", [1, 37, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_attention_unquantized_matches_sdpa(oracle_lib, L, dtype):
    dt = oracle.BF16 if dtype == "bf16" else oracle.F16
    cfg = oracle.Cfg(num_q_heads=8, num_kv_heads=2, head_dim=64, dtype=dt)
    rng = np.random.default_rng(7 + L)
    K, V = _rand_kv(rng, 2, L, 64, dtype)
    s = oracle.SeqCache(cfg, 64)
    assert s.append(K, V) == oracle.OK and oracle.n_packed(cfg, L) == 0
    q = to_dtype_bits(rng.standard_normal((8, 64)), dtype)
    scale = 1 / math.sqrt(64)
    got = s.decode(q, scale)
    f = lambda b: bits_to_f32(b, dtype).astype(np.float64)
    want = _sdpa(f(q), f(K), f(V), scale, 4)
    assert np.max(np.abs(got - want)) < 1e-12
    if L == 1:
        assert np.array_equal(got, np.repeat(f(V)[:, 0], 4, axis=0))


@pytest.mark.parametrize("kb,vb,G,R", VARIANTS)
def test_attention_planted_cache_matches_sdpa(oracle_lib, kb, vb, G, R):
    """Packed tokens built on exact grids decode without error, so the oracle's
    attention over packed + residual tokens must equal exact attention. Keys and
    values use their own code widths (codes 0 and qmax planted in every group)."""
    D, H, g = 128, 2, 4
    cfg = oracle.Cfg(k_bits=kb, v_bits=vb, num_q_heads=H * g, num_kv_heads=H, head_dim=D, group=G, residual=R)
    kq, vq = (1 << kb) - 1, (1 << vb) - 1
    rng = np.random.default_rng(8 + kb + 3 * vb + G + R)
    L = 333                                  # e.g. 192 packed (6 groups of 32) + 141 residual
    P = oracle.n_packed(cfg, L)
    assert P == G * ((L - R) // G) and P > 0
    # keys: per (head, group, channel) a power-of-two scale and zero; codes use 0 and qmax
    sk = np.ldexp(1.0, rng.integers(-4, 0, size=(H, L // G + 1, D)))
    zk = rng.integers(-16, 16, size=sk.shape) * sk
    ck = planted_codes(rng, (H, L // G + 1, G, D), kq, axis=2).reshape(H, -1, D)[:, :L]
    K = np.repeat(zk, G, axis=1)[:, :L] + ck * np.repeat(sk, G, axis=1)[:, :L]
    # values: per (head, token, channel group)
    sv = np.ldexp(1.0, rng.integers(-4, 0, size=(H, L, D // G)))
    zv = rng.integers(-16, 16, size=sv.shape) * sv
    cv = planted_codes(rng, (H, L, D // G, G), vq, axis=3).reshape(H, L, D)
    V = np.repeat(zv, G, axis=2) + cv * np.repeat(sv, G, axis=2)
    Kb, Vb = to_dtype_bits(K, "f16"), to_dtype_bits(V, "f16")
    s = oracle.SeqCache(cfg, 256)
    assert s.append(Kb, Vb) == oracle.OK
    q = to_dtype_bits(rng.standard_normal((H * g, D)), "f16")
    scale = 1 / math.sqrt(D)
    got = s.decode(q, scale)
    want = _sdpa(bits_to_f32(q, "f16").astype(np.float64), K, V, scale, g)
    assert np.max(np.abs(got - want)) < 1e-12


def test_attention_identical_keys_is_mean_of_values(oracle_lib):
    D = 64
    cfg = oracle.Cfg(num_q_heads=1, num_kv_heads=1, head_dim=D)
    rng = np.random.default_rng(9)
    L = 300
    k = rng.standard_normal(D)
    K = np.repeat(k[None, None, :], L, axis=1)
    # values on exact grids (see the planted test) so that they decode exactly
    sv = np.ldexp(1.0, rng.integers(-3, 0, size=(1, L, D // 32)))
    cv = planted_codes(rng, (1, L, D // 32, 32), 3, axis=3).reshape(1, L, D)
    V = cv * np.repeat(sv, 32, axis=2)
    s = oracle.SeqCache(cfg, 256)
    assert s.append(to_dtype_bits(K, "f16"), to_dtype_bits(V, "f16")) == oracle.OK
    got = s.decode(to_dtype_bits(rng.standard_normal((1, D)), "f16"), 0.125)
    assert np.max(np.abs(got[0] - V[0].mean(axis=0))) < 1e-12


def test_attention_empty_sequence_is_zero(oracle_lib):
    cfg = oracle.Cfg(num_q_heads=2, num_kv_heads=1, head_dim=32)
    s = oracle.SeqCache(cfg, 32)
    out = s.decode(np.zeros((2, 32), np.uint16), 0.1)
    assert np.all(out == 0.0)


def test_workload_tiny_state(oracle_lib):
    """The tiny decode workload ends with 896 packed tokens (28 key groups) and 128 residual."""
    wl = workload(0)
    cfg = oracle.Cfg(num_q_heads=1, num_kv_heads=1)
    s = oracle.SeqCache(cfg, 1024)
    K, V = wl.kv_seq(0, 0, 1024)
    assert s.append(K, V) == oracle.OK
    assert oracle.n_packed(cfg, s.L) == 896 and s.L - 896 == 128
