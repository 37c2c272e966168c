"""The premise of the asymmetric scheme on the synthetic outlier-structured caches, through
the oracle's quantizers (CPU): keys carry fixed outlier channels, so quantizing them per
channel ("KV-Cache Quantization: I Ran the Experiments So You Don't Have To", Component 2,
Figure 4: per-channel key 0.623 vs per-token key 0.786 at 2 bits) gives lower score error
than per token; values carry burst tokens, so per-token values give lower output error
than per-channel ones; KIVI's pairing is the best of the four at both widths. Also the
reference numbers for the GPU study (tests/test_gpu_study.py)."""
import numpy as np
import pytest

import oracle
import synth
from test_oracle_codec import unpack

SCHEMES = {
    "uniform, K and V per-token": ("token", "token"),
    "uniform, K and V per-channel": ("channel", "channel"),
    "KIVI: K per-channel, V per-token": ("channel", "token"),
    "K per-token, V per-channel": ("token", "channel"),
}


def f16(b):
    return np.asarray(b, np.uint16).view(np.float16).astype(np.float64)


def dequant(cfg, xb, axis):
    G = cfg.group
    if axis == "channel":
        codes, s, z = oracle.quant_keys(cfg, xb)
        s, z = np.repeat(f16(s), G, axis=1), np.repeat(f16(z), G, axis=1)
    else:
        codes, s, z = oracle.quant_values(cfg, xb)
        s, z = np.repeat(f16(s), G, axis=2), np.repeat(f16(z), G, axis=2)
    return unpack(codes, cfg.bits, cfg.head_dim) * s + z


def softmax(x):
    e = np.exp(x - x.max(axis=-1, keepdims=True))
    return e / e.sum(axis=-1, keepdims=True)


def study(workload=1, seqs=1, T=512, bits_list=(2, 4), group=32):
    wl = synth.workload(workload)
    H, D = wl.num_kv_heads, wl.head_dim
    Kb = np.stack([wl.keys(b, h, 0, T) for b in range(seqs) for h in range(H)])
    Vb = np.stack([wl.values(b, h, 0, T) for b in range(seqs) for h in range(H)])
    K, V = synth.bits_to_f32(Kb, wl.dtype).astype(np.float64), synth.bits_to_f32(Vb, wl.dtype).astype(np.float64)
    qa = synth.bits_to_f32(wl.query(0), wl.dtype).astype(np.float64)
    g = wl.num_q_heads // H
    q = np.stack([qa[b, h * g] for b in range(seqs) for h in range(H)])
    s = np.einsum("sd,std->st", q, K) * wl.softmax_scale
    p = softmax(s)
    o = np.einsum("st,std->sd", p, V)
    rows = {}
    for bits in bits_list:
        cfg = oracle.Cfg(bits=bits, head_dim=D, dtype=oracle.BF16 if wl.dtype == "bf16" else oracle.F16, group=group)
        deq = {("k", a): dequant(cfg, Kb, a) for a in ("token", "channel")}
        deq.update({("v", a): dequant(cfg, Vb, a) for a in ("token", "channel")})
        for name, (ka, va) in SCHEMES.items():
            sq = np.einsum("sd,std->st", q, deq[("k", ka)]) * wl.softmax_scale
            pq = softmax(sq)
            oq = np.einsum("st,std->sd", pq, deq[("v", va)])
            rows[(name, bits)] = (float(np.mean(np.linalg.norm(sq - s, axis=-1) / np.linalg.norm(s, axis=-1))),
                                  float(np.mean(0.5 * np.abs(pq - p).sum(axis=-1))),
                                  float(np.mean(np.linalg.norm(oq - o, axis=-1) / np.linalg.norm(o, axis=-1))))
    return rows


@pytest.mark.parametrize("workload", [1, 2])
def test_asymmetric_scheme_wins_on_outlier_structure(workload):
    rows = study(workload, seqs=1, T=512)
    for bits in (2, 4):
        kivi_ = rows[("KIVI: K per-channel, V per-token", bits)]
        tok_k = rows[("uniform, K and V per-token", bits)]
        wrong = rows[("K per-token, V per-channel", bits)]
        chan = rows[("uniform, K and V per-channel", bits)]
        # keys: per-channel beats per-token on the scores (outlier channels)
        assert kivi_[0] < tok_k[0] and chan[0] < wrong[0], (bits, kivi_, tok_k)
        # values: per-token beats per-channel on the output, with the same keys (burst tokens)
        assert kivi_[2] < chan[2] and tok_k[2] < wrong[2], (bits, kivi_, chan)
        # KIVI's pairing is the best of the four, and 4 bits beat 2 bits
        assert kivi_[2] == min(rows[(n, bits)][2] for n in SCHEMES)
    assert rows[("KIVI: K per-channel, V per-token", 4)][2] < rows[("KIVI: K per-channel, V per-token", 2)][2]
