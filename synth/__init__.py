"""Seeded synthetic inputs for the KIVI workloads.

Shared by the tests, the oracle runs and the benchmark. This module holds no
quantization and no attention arithmetic: it only draws keys, values and
queries with the shapes and structure of the workloads (fixed outlier key
channels per kv head, value "burst" tokens), as bit patterns of the storage
dtype.

Generator. Every element has a counter (seed, tensor id, index). A uniform is
``splitmix64(seed * A + tensor_id * B + index) >> 11`` scaled by 2^-53
(splitmix64 as published by Steele, Lea and Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014). A standard normal is
Box-Muller over the uniforms of counters 2i and 2i+1, in fp64. Values are
then rounded to fp32 and from fp32 to the storage dtype (round to nearest,
ties to even). Because every element depends only on its own counter, any
slice (one sequence, one head, a token range) can be drawn on its own, on the
CPU (numpy) or on the GPU (torch), and the two agree up to the last-ulp
behaviour of log/cos in fp64.

Element counters:
  K[b, h, t, d]   tensor 1, index ((b*Hkv + h) << 20 | t) * D + d
  V[b, h, t, d]   tensor 2, same index
  outlier perm    tensor 3, index h*D + i            (Fisher-Yates per kv head)
  burst token     tensor 4, index b << 20 | t        (Bernoulli per (b, t))
  q[step, b, hq]  tensor 5, index ((step*B + b)*Hq + hq)*D + d
  length L_b      tensor 6, index b                  (log-uniform)
Token counters leave room for 2^20 positions per (b, h).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

_M64 = (1 << 64) - 1
_A = 0x9E3779B97F4A7C15
_B = 0xD1B54A32D192ED03
T_K, T_V, T_PERM, T_BURST, T_Q, T_LEN = 1, 2, 3, 4, 5, 6
TOKEN_BITS = 20


def _splitmix64(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z += np.uint64(0x9E3779B97F4A7C15)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return z


def _base(seed: int, tensor: int) -> np.uint64:
    return np.uint64((seed * _A + tensor * _B) & _M64)


def uniform(seed: int, tensor: int, index: np.ndarray) -> np.ndarray:
    """U[0,1) in fp64 for the given uint64 counters."""
    idx = np.asarray(index, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = _splitmix64(idx + _base(seed, tensor))
    return (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def normal(seed: int, tensor: int, index: np.ndarray) -> np.ndarray:
    """N(0,1) in fp64 by Box-Muller over counters 2i and 2i+1."""
    idx = np.asarray(index, dtype=np.uint64)
    u1 = uniform(seed, tensor, idx * np.uint64(2))
    u2 = uniform(seed, tensor, idx * np.uint64(2) + np.uint64(1))
    return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * math.pi * u2)


def to_dtype_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 -> fp32 (RN) -> storage dtype (RN-even); returns uint16 bit patterns."""
    x32 = np.asarray(x, dtype=np.float32)
    if dtype == "f16":
        return x32.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x32.view(np.uint32).astype(np.uint64)
        upper = u >> np.uint64(16)
        rem = u & np.uint64(0xFFFF)
        up = (rem > 0x8000) | ((rem == 0x8000) & ((upper & np.uint64(1)) == 1))
        return (upper + up.astype(np.uint64)).astype(np.uint16)
    raise ValueError(dtype)


def bits_to_f32(bits: np.ndarray, dtype: str) -> np.ndarray:
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclass(frozen=True)
class Workload:
    """One synthetic KIVI workload (shapes, distributions and seed)."""
    name: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    lengths: tuple            # tokens per sequence before any decode step
    dtype: str = "f16"        # storage dtype of K, V, q
    bits: int = 2
    group: int = 32
    residual: int = 128
    k_outliers: int = 4       # outlier key channels per kv head
    k_outlier_scale: float = 20.0
    v_burst_frac: float = 0.02
    v_burst_scale: float = 10.0
    steps: int = 0            # decode steps (streaming workload)
    seed: int = 1000
    extra: dict = field(default_factory=dict, compare=False, hash=False)

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    def outlier_channels(self, h: int) -> np.ndarray:
        """The fixed outlier channels of kv head h: the first k of a seeded Fisher-Yates shuffle."""
        D = self.head_dim
        u = uniform(self.seed, T_PERM, np.arange(h * D, (h + 1) * D, dtype=np.uint64))
        perm = list(range(D))
        for i in range(D - 1, 0, -1):
            j = int(u[i] * (i + 1))
            perm[i], perm[j] = perm[j], perm[i]
        return np.array(sorted(perm[: self.k_outliers]), dtype=np.int64)

    def burst_mask(self, b: int, t0: int, n: int) -> np.ndarray:
        idx = (np.uint64(b) << np.uint64(TOKEN_BITS)) + np.arange(t0, t0 + n, dtype=np.uint64)
        return uniform(self.seed, T_BURST, idx) < self.v_burst_frac

    def _kv_index(self, b: int, h: int, t0: int, n: int) -> np.ndarray:
        D = self.head_dim
        row = ((np.uint64(b * self.num_kv_heads + h) << np.uint64(TOKEN_BITS))
               + np.arange(t0, t0 + n, dtype=np.uint64))
        return (row[:, None] * np.uint64(D) + np.arange(D, dtype=np.uint64)[None, :])

    def keys_f64(self, b: int, h: int, t0: int, n: int) -> np.ndarray:
        k = normal(self.seed, T_K, self._kv_index(b, h, t0, n))
        k[:, self.outlier_channels(h)] *= self.k_outlier_scale
        return k

    def values_f64(self, b: int, h: int, t0: int, n: int) -> np.ndarray:
        v = normal(self.seed, T_V, self._kv_index(b, h, t0, n))
        v[self.burst_mask(b, t0, n)] *= self.v_burst_scale
        return v

    def keys(self, b: int, h: int, t0: int, n: int) -> np.ndarray:
        """[n][D] uint16 patterns of K[b, h, t0:t0+n, :]."""
        return to_dtype_bits(self.keys_f64(b, h, t0, n), self.dtype)

    def values(self, b: int, h: int, t0: int, n: int) -> np.ndarray:
        return to_dtype_bits(self.values_f64(b, h, t0, n), self.dtype)

    def kv_seq(self, b: int, t0: int, n: int):
        """K, V of sequence b for all kv heads: two [Hkv][n][D] uint16 arrays."""
        K = np.stack([self.keys(b, h, t0, n) for h in range(self.num_kv_heads)])
        V = np.stack([self.values(b, h, t0, n) for h in range(self.num_kv_heads)])
        return K, V

    def query(self, step: int = 0, b: int | None = None) -> np.ndarray:
        """q [B][Hq][D] (or [Hq][D] for one sequence) uint16 patterns for a decode step."""
        B, Hq, D = self.batch, self.num_q_heads, self.head_dim
        bs = range(B) if b is None else [b]
        idx = np.stack([((np.uint64(step * B + bb) * np.uint64(Hq) + np.arange(Hq, dtype=np.uint64))[:, None]
                         * np.uint64(D) + np.arange(D, dtype=np.uint64)[None, :]) for bb in bs])
        q = to_dtype_bits(normal(self.seed, T_Q, idx), self.dtype)
        return q if b is None else q[0]

    def replace(self, **kw) -> "Workload":
        d = {f: getattr(self, f) for f in self.__dataclass_fields__}
        d.update(kw)
        return Workload(**d)


def varlen_lengths(seed: int, batch: int, lo: int = 1024, hi: int = 131072) -> tuple:
    """L_b = floor(lo * (hi/lo)^u), u ~ U[0,1) per sequence, clamped to [lo, hi]."""
    u = uniform(seed, T_LEN, np.arange(batch, dtype=np.uint64))
    L = np.floor(lo * np.power(hi / lo, u)).astype(np.int64)
    return tuple(int(x) for x in np.clip(L, lo, hi))


def workload(index: int) -> Workload:
    """The five workloads of the KIVI decode path, by index.

    0 tiny decode: 1 seq, 1/1 heads, 1024 tokens, fp16, 4 outlier channels x20, 2% bursts x10
    1 Llama-2-7B layer: 8 seqs, 32/32 heads, 4096 tokens, fp16, 8 outlier channels x15, 2% bursts x10
    2 Llama-3-8B GQA decode: 64 seqs, 32/8 heads, 32768 tokens, bf16, 4 x20, 1% x10
    3 streaming: 16 seqs, 32/8 heads, 16384-token prefill then 512 decode steps, fp16, 4 x20, 1% x10
    4 long varlen (Mistral-7B shape): 32 seqs, 32/8 heads, log-uniform [1024, 131072], fp16, 4 x20, 1% x10
    """
    seed = 1000 + index
    if index == 0:
        return Workload("tiny-decode", 1, 1, 1, 128, (1024,), "f16", k_outliers=4, k_outlier_scale=20.0,
                        v_burst_frac=0.02, seed=seed)
    if index == 1:
        return Workload("llama2-7b-mha", 8, 32, 32, 128, (4096,) * 8, "f16", k_outliers=8,
                        k_outlier_scale=15.0, v_burst_frac=0.02, seed=seed)
    if index == 2:
        return Workload("llama3-8b-gqa", 64, 32, 8, 128, (32768,) * 64, "bf16", k_outliers=4,
                        k_outlier_scale=20.0, v_burst_frac=0.01, seed=seed)
    if index == 3:
        return Workload("streaming-append", 16, 32, 8, 128, (16384,) * 16, "f16", k_outliers=4,
                        k_outlier_scale=20.0, v_burst_frac=0.01, steps=512, seed=seed)
    if index == 4:
        return Workload("long-varlen", 32, 32, 8, 128, varlen_lengths(seed, 32), "f16", k_outliers=4,
                        k_outlier_scale=20.0, v_burst_frac=0.01, seed=seed)
    raise ValueError(index)


# ---------------------------------------------------------------- GPU drawing (torch)
def _torch_splitmix64(z):
    import torch
    # uint64 arithmetic in int64 tensors: + and * wrap mod 2^64; right shifts are
    # made logical with a mask.
    def srl(x, k):
        return (x >> k) & ((1 << (64 - k)) - 1)
    z = z + torch.tensor(_to_i64(0x9E3779B97F4A7C15), dtype=torch.int64, device=z.device)
    z = (z ^ srl(z, 30)) * torch.tensor(_to_i64(0xBF58476D1CE4E5B9), dtype=torch.int64, device=z.device)
    z = (z ^ srl(z, 27)) * torch.tensor(_to_i64(0x94D049BB133111EB), dtype=torch.int64, device=z.device)
    return z ^ srl(z, 31)


def _to_i64(u: int) -> int:
    u &= _M64
    return u - (1 << 64) if u >= (1 << 63) else u


def torch_normal(seed: int, tensor: int, index):
    """The same counters as `normal`, drawn with torch on index's device (int64 counters)."""
    import torch
    base = torch.tensor(_to_i64(int(_base(seed, tensor))), dtype=torch.int64, device=index.device)

    def u(ix):
        z = _torch_splitmix64(ix + base)
        return ((z >> 11) & ((1 << 53) - 1)).to(torch.float64) * (1.0 / 9007199254740992.0)

    u1 = u(index * 2)
    u2 = u(index * 2 + 1)
    return torch.sqrt(-2.0 * torch.log1p(-u1)) * torch.cos(2.0 * math.pi * u2)


def torch_kv_head_major(wl: Workload, b: int, h: int, t0: int, n: int, which: str, device):
    """K or V[b, h, t0:t0+n, :] as a torch tensor of wl.dtype on `device` (same counters as numpy)."""
    import torch
    D = wl.head_dim
    row = ((b * wl.num_kv_heads + h) << TOKEN_BITS) + torch.arange(t0, t0 + n, dtype=torch.int64, device=device)
    idx = row[:, None] * D + torch.arange(D, dtype=torch.int64, device=device)[None, :]
    x = torch_normal(wl.seed, T_K if which == "k" else T_V, idx)
    if which == "k":
        ch = torch.as_tensor(wl.outlier_channels(h), device=device)
        x[:, ch] *= wl.k_outlier_scale
    else:
        mask = torch.as_tensor(wl.burst_mask(b, t0, n), device=device)
        x[mask] *= wl.v_burst_scale
    tdt = torch.float16 if wl.dtype == "f16" else torch.bfloat16
    return x.to(torch.float32).to(tdt)
