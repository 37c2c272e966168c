"""Pins for the oracle's multi-query attention (the n_query newest tokens of a
sequence, each attending causally to the tokens up to its own position): checked
against torch's scaled_dot_product_attention in fp64 with an explicit causal mask on
caches whose packed tokens decode exactly (planted grids), with GQA, at both code
widths and both group sizes."""
import math

import numpy as np
import pytest
import torch

import oracle
from synth import bits_to_f32, to_dtype_bits
from test_oracle_codec import planted_codes


def planted_cache(rng, cfg, L):
    """K, V [Hkv][L][D] on exact grids of the cache's groups (every packed token decodes
    exactly) and the oracle cache holding them."""
    H, D, G = cfg.num_kv_heads, cfg.head_dim, cfg.group
    kq, vq = (1 << cfg.k_bits) - 1, (1 << cfg.v_bits) - 1
    ng = L // G + 1
    sk = np.ldexp(1.0, rng.integers(-4, 0, size=(H, ng, D)))
    zk = rng.integers(-16, 16, size=sk.shape) * sk
    ck = planted_codes(rng, (H, ng, G, D), kq, axis=2).reshape(H, -1, D)[:, :L]
    K = np.repeat(zk, G, axis=1)[:, :L] + ck * np.repeat(sk, G, axis=1)[:, :L]
    sv = np.ldexp(1.0, rng.integers(-4, 0, size=(H, L, D // G)))
    zv = rng.integers(-16, 16, size=sv.shape) * sv
    cv = planted_codes(rng, (H, L, D // G, G), vq, axis=3).reshape(H, L, D)
    V = np.repeat(zv, G, axis=2) + cv * np.repeat(sv, G, axis=2)
    cap = G * ((L + G - 1) // G)
    s = oracle.SeqCache(cfg, cap)
    assert s.append(to_dtype_bits(K, "f16"), to_dtype_bits(V, "f16")) == oracle.OK
    return K, V, s


def causal_sdpa(q, K, V, scale, g):
    """q [nq][Hq][D] at the nq newest positions, K, V [Hkv][L][D] -> [nq][Hq][D], fp64."""
    nq, L = q.shape[0], K.shape[1]
    qt = torch.from_numpy(q).permute(1, 0, 2)[None]                  # [1][Hq][nq][D]
    Kt = torch.from_numpy(K).repeat_interleave(g, dim=0)[None]
    Vt = torch.from_numpy(V).repeat_interleave(g, dim=0)[None]
    pos = torch.arange(L - nq, L)[:, None]
    mask = torch.arange(L)[None, :] <= pos                             # [nq][L]
    o = torch.nn.functional.scaled_dot_product_attention(qt, Kt, Vt, attn_mask=mask, scale=scale)
    return o[0].permute(1, 0, 2).numpy()


@pytest.mark.parametrize("kb,vb,G,R", [(2, 2, 32, 128), (4, 2, 64, 64), (2, 4, 32, 64)])
@pytest.mark.parametrize("g", [1, 4])
@pytest.mark.parametrize("nq", [1, 3, 16])
def test_multi_query_matches_causal_sdpa(oracle_lib, kb, vb, G, R, g, nq):
    D, H = 64, 2
    cfg = oracle.Cfg(k_bits=kb, v_bits=vb, group=G, residual=R, num_q_heads=g * H, num_kv_heads=H, head_dim=D)
    rng = np.random.default_rng(1000 + kb + 3 * vb + G + R + g + nq)
    L = 301
    K, V, s = planted_cache(rng, cfg, L)
    assert oracle.n_packed(cfg, L) > 0
    qb = to_dtype_bits(rng.standard_normal((nq, g * H, D)), "f16")
    scale = 1 / math.sqrt(D)
    got = s.decode_multi(qb, scale)
    want = causal_sdpa(bits_to_f32(qb, "f16").astype(np.float64), K, V, scale, g)
    assert np.max(np.abs(got - want)) < 1e-12
    # the newest query sees every token: it is decode attention
    assert np.max(np.abs(got[-1] - s.decode(qb[-1], scale))) < 1e-12


def test_multi_query_all_residual_and_length_errors(oracle_lib):
    """A sequence shorter than R (nothing packed): the causal mask alone decides; the first
    query of a sequence holding exactly n_query tokens sees only token 0. L < n_query is an
    argument error."""
    D, H, nq = 64, 1, 5
    cfg = oracle.Cfg(num_q_heads=2, num_kv_heads=H, head_dim=D)
    rng = np.random.default_rng(7)
    K = rng.standard_normal((H, nq, D))
    V = rng.standard_normal((H, nq, D))
    s = oracle.SeqCache(cfg, 32)
    assert s.append(to_dtype_bits(K, "f16"), to_dtype_bits(V, "f16")) == oracle.OK
    qb = to_dtype_bits(rng.standard_normal((nq, 2, D)), "f16")
    got = s.decode_multi(qb, 0.125)
    Vf = bits_to_f32(to_dtype_bits(V, "f16"), "f16").astype(np.float64)
    assert np.array_equal(got[0], np.repeat(Vf[:, 0], 2, axis=0))
    Kf = bits_to_f32(to_dtype_bits(K, "f16"), "f16").astype(np.float64)
    want = causal_sdpa(bits_to_f32(qb, "f16").astype(np.float64), Kf, Vf, 0.125, 2)
    assert np.max(np.abs(got - want)) < 1e-12
    with pytest.raises(ValueError):
        s.decode_multi(to_dtype_bits(np.zeros((nq + 1, 2, D)), "f16"), 0.125)
