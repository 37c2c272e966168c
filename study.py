"""Attention error of four quantization axes on a synthetic outlier-structured cache.

An analysis script that sits beside bench.py: it drives the library's codec entry
points with the seeded generators of synth/ and is not part of the library package.

The comparison of "KV-Cache Quantization: I Ran the Experiments So You Don't Have To",
Component 2 (Figure 4): keys and values each quantized along the tokens of a channel
("per-channel": this library's key quantizer, kivi_quant_keys) or along the channels of a
token ("per-token": the value quantizer, kivi_quant_values), at 2 and 4 bits, then
attention recomputed from the dequantized cache (c * s + z) against the unquantized one.
Every quantization runs through the library's own entry points on the GPU; the errors are
computed in fp64. The page does not define its error; here three are reported per query
head and averaged: relative L2 error of the scores, total variation of the softmax
probabilities, and relative L2 error of the attention output.

    python study.py --workload 1 --seqs 2
"""
from __future__ import annotations

import argparse
import json

import numpy as np
import torch

import synth
from bit_asymmetric_kv_kivi_gb300 import BF16, F16, Config, GROUP, quant_keys, quant_values

SCHEMES = {
    "uniform, K and V per-token": ("token", "token"),
    "uniform, K and V per-channel": ("channel", "channel"),
    "KIVI: K per-channel, V per-token": ("channel", "token"),
    "K per-token, V per-channel": ("token", "channel"),
}


def unpack(codes: torch.Tensor, bits: int, D: int) -> torch.Tensor:
    """[..., D * bits / 8] u8 -> [..., D] integer codes: channel d in byte d*bits/8 at bit (d mod 8/bits)*bits."""
    d = torch.arange(D, device=codes.device)
    byte = codes[..., (d * bits) // 8].to(torch.int32)
    return (byte >> ((d * bits) % 8).to(torch.int32)) & ((1 << bits) - 1)


def f16(x: torch.Tensor) -> torch.Tensor:
    return x.view(torch.float16).to(torch.float64)


def dequant(cfg: Config, x: torch.Tensor, axis: str) -> torch.Tensor:
    """Quantize x [S][T][D] (cfg dtype, T a multiple of 32) along `axis` with the library and
    return c * s + z in fp64."""
    S, T, D = x.shape
    if axis == "channel":
        codes, scale, zero = quant_keys(cfg, x)
        s = f16(scale).repeat_interleave(cfg.group, dim=1)               # [S][T][D]
        z = f16(zero).repeat_interleave(cfg.group, dim=1)
    else:
        codes, scale, zero = quant_values(cfg, x)
        s = f16(scale).repeat_interleave(cfg.group, dim=2)               # [S][T][D]
        z = f16(zero).repeat_interleave(cfg.group, dim=2)
    return unpack(codes, cfg.bits, D).to(torch.float64) * s + z


def attention_errors(q, K, V, Kq, Vq, scale):
    """q [S][D], K, V, Kq, Vq [S][T][D] fp64 -> mean over S of (score rel. L2, prob. TV, output rel. L2)."""
    s = torch.einsum("sd,std->st", q, K) * scale
    sq = torch.einsum("sd,std->st", q, Kq) * scale
    p, pq = torch.softmax(s, dim=-1), torch.softmax(sq, dim=-1)
    o, oq = torch.einsum("st,std->sd", p, V), torch.einsum("st,std->sd", pq, Vq)
    e_s = (torch.linalg.norm(sq - s, dim=-1) / torch.linalg.norm(s, dim=-1)).mean()
    e_p = (0.5 * (pq - p).abs().sum(dim=-1)).mean()
    e_o = (torch.linalg.norm(oq - o, dim=-1) / torch.linalg.norm(o, dim=-1)).mean()
    return float(e_s), float(e_p), float(e_o)


def run(workload: int = 1, seqs: int = 2, tokens: int | None = None, bits_list=(2, 4), device="cuda",
        group: int = GROUP):
    """One row per (scheme, bits): the three mean errors over `seqs` sequences x every kv
    head (one decode query per head: the first query head of its group), with groups of
    `group` tokens (keys) or channels (values)."""
    wl = synth.workload(workload)
    T = (min(tokens or wl.lengths[0], wl.lengths[0]) // group) * group
    H, D = wl.num_kv_heads, wl.head_dim
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
    K = torch.stack([synth.torch_kv_head_major(wl, b, h, 0, T, "k", device) for b in range(seqs) for h in range(H)])
    V = torch.stack([synth.torch_kv_head_major(wl, b, h, 0, T, "v", device) for b in range(seqs) for h in range(H)])
    q_all = torch.from_numpy(wl.query(0).view(np.int16)).view(tdt)          # [B][Hq][D]
    g = wl.num_q_heads // H
    q = torch.stack([q_all[b, h * g] for b in range(seqs) for h in range(H)]).to(device).to(torch.float64)
    K64, V64 = K.to(torch.float64), V.to(torch.float64)
    rows = []
    for bits in bits_list:
        cfg = Config(bits=bits, head_dim=D, num_q_heads=1, num_kv_heads=1, dtype=BF16 if wl.dtype == "bf16" else F16,
                     group=group)
        deq = {("k", a): dequant(cfg, K, a) for a in ("token", "channel")}
        deq.update({("v", a): dequant(cfg, V, a) for a in ("token", "channel")})
        for name, (ka, va) in SCHEMES.items():
            e = attention_errors(q, K64, V64, deq[("k", ka)], deq[("v", va)], wl.softmax_scale)
            rows.append({"scheme": name, "bits": bits, "score_rel_l2": e[0], "prob_tv": e[1], "out_rel_l2": e[2]})
    return {"workload": wl.name, "sequences": seqs, "tokens": T, "kv_heads": H, "group": group, "rows": rows}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--workload", type=int, default=1)
    ap.add_argument("--seqs", type=int, default=2)
    ap.add_argument("--tokens", type=int, default=0)
    ap.add_argument("--group", type=int, default=GROUP, help="G: 32 or 64")
    args = ap.parse_args()
    res = run(args.workload, args.seqs, args.tokens or None, group=args.group)
    print(f"{res['workload']}: {res['sequences']} sequences x {res['kv_heads']} kv heads x {res['tokens']} tokens, "
          f"G = {res['group']}")
    print(f"{'scheme':34s} bits  score rel.L2  prob. TV  output rel.L2")
    for r in res["rows"]:
        print(f"{r['scheme']:34s} {r['bits']:4d}  {r['score_rel_l2']:12.4f}  {r['prob_tv']:8.4f}  {r['out_rel_l2']:13.4f}")
    print(json.dumps(res))


if __name__ == "__main__":
    main()
