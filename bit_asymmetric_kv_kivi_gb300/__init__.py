"""GB300-native KIVI KV-cache library: the Python binding of the C ABI in include/kivi.h.

This module only marshals arguments (tensor pointers, sizes, the current CUDA
stream) into libkivi.so; every step of the codec, the append/flush and the
decode attention runs in the library's CUDA kernels. PyTorch is used for
device memory and streams.

The library is built in-tree by ``__graft_entry__.build()`` (or
``python -m bit_asymmetric_kv_kivi_gb300._build``). Loading it needs no GPU, so
sizes and argument validation work on any host; compute calls raise
``RuntimeError`` when no CUDA device is present and ``ImportError``-style
``RuntimeError`` when the library has not been built. There is no CPU path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libkivi.so")

F16, BF16 = 0, 1
OK, ERR_ARG, ERR_UNSUPPORTED, ERR_CAPACITY, ERR_WORKSPACE, ERR_CUDA, ERR_LENGTH = range(7)
GROUP = 32          # the default G

_TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16}


class KiviError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


class _Cfg(ctypes.Structure):
    _fields_ = [("k_bits", ctypes.c_int32), ("v_bits", ctypes.c_int32), ("group", ctypes.c_int32),
                ("residual", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("dtype", ctypes.c_int32)]


SEQ_FIELDS = ("k_codes", "k_scale", "k_zero", "v_codes", "v_scale", "v_zero", "k_res", "v_res")
SEQ_STRUCT_BYTES = 8 * 8 + 2 * 4 + 8   # eight pointers, cap_tokens, flags, block_table
SEQ_PAGED = 1

_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libkivi.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libkivi.so is not built ({LIB_PATH}); run __graft_entry__.build()")
            L = ctypes.CDLL(LIB_PATH)
            P, I32, CFG = ctypes.c_void_p, ctypes.c_int32, ctypes.POINTER(_Cfg)
            for name in ("kivi_quant_keys", "kivi_quant_values"):
                fn = getattr(L, name)
                fn.argtypes = [CFG, I32, I32, P, P, P, P, P]
                fn.restype = I32
            L.kivi_append_flush.argtypes = [CFG, I32, P, P, P, P, P, I32, P, P]
            L.kivi_append_flush.restype = I32
            L.kivi_decode_attn.argtypes = [CFG, I32, P, P, P, P, ctypes.c_float, I32, P, ctypes.c_size_t, P, P]
            L.kivi_decode_attn.restype = I32
            L.kivi_decode_workspace_bytes.argtypes = [CFG, I32, I32]
            L.kivi_decode_workspace_bytes.restype = ctypes.c_size_t
            L.kivi_decode_multi_attn.argtypes = [CFG, I32, P, P, I32, P, P, ctypes.c_float, I32, P, ctypes.c_size_t,
                                                 P, P]
            L.kivi_decode_multi_attn.restype = I32
            L.kivi_decode_multi_workspace_bytes.argtypes = [CFG, I32, I32, I32]
            L.kivi_decode_multi_workspace_bytes.restype = ctypes.c_size_t
            L.kivi_seq_buffer_bytes.argtypes = [CFG, I32, ctypes.POINTER(ctypes.c_size_t)]
            L.kivi_seq_buffer_bytes.restype = I32
            L.kivi_seq_bytes.argtypes = [CFG, I32]
            L.kivi_seq_bytes.restype = ctypes.c_int64
            L.kivi_n_packed.argtypes = [CFG, ctypes.c_int64]
            L.kivi_n_packed.restype = ctypes.c_int64
            L.kivi_kv_bytes_plain.argtypes = [I32, I32, I32, I32, ctypes.c_int64, ctypes.c_int64]
            L.kivi_kv_bytes_plain.restype = ctypes.c_int64
            L.kivi_status_string.argtypes = [I32]
            L.kivi_status_string.restype = ctypes.c_char_p
            L.kivi_abi_version.argtypes = []
            L.kivi_abi_version.restype = I32
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().kivi_status_string(int(status)).decode()


def kv_bytes_plain(layers: int, num_kv_heads: int, head_dim: int, bits: int, tokens: int, batch: int = 1) -> int:
    """KV-cache bytes with no quantization metadata (kivi_kv_bytes_plain); -1 on bad input."""
    return int(lib().kivi_kv_bytes_plain(layers, num_kv_heads, head_dim, bits, tokens, batch))


def _check(status: int, where: str) -> None:
    if status != OK:
        raise KiviError(status, where)


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _require_cuda(t: torch.Tensor, name: str) -> None:
    if not torch.cuda.is_available():
        raise RuntimeError("KIVI kernels need a CUDA device; there is no CPU path")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _ptr(t: torch.Tensor | None) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


@dataclass(frozen=True)
class Config:
    """A KIVI configuration (mirrors kivi_cfg). `bits` sets both code widths; k_bits and
    v_bits, when given, set the key and value widths apart."""
    bits: int = 2
    head_dim: int = 128
    num_q_heads: int = 1
    num_kv_heads: int = 1
    dtype: int = F16
    residual: int = 128
    group: int = GROUP
    k_bits: int | None = None
    v_bits: int | None = None

    def __post_init__(self):
        if self.k_bits is None:
            object.__setattr__(self, "k_bits", self.bits)
        if self.v_bits is None:
            object.__setattr__(self, "v_bits", self.bits)

    def c(self) -> _Cfg:
        return _Cfg(self.k_bits, self.v_bits, self.group, self.residual, self.head_dim, self.num_q_heads,
                    self.num_kv_heads, self.dtype)

    @property
    def torch_dtype(self) -> torch.dtype:
        return _TORCH_DTYPE[self.dtype]

    @property
    def k_row_bytes(self) -> int:
        return self.head_dim * self.k_bits // 8

    @property
    def v_row_bytes(self) -> int:
        return self.head_dim * self.v_bits // 8

    @property
    def ring(self) -> int:
        return self.residual + self.group

    def n_packed(self, kv_len: int) -> int:
        return int(lib().kivi_n_packed(self.c(), kv_len))

    def seq_buffer_bytes(self, cap_tokens: int) -> list[int]:
        arr = (ctypes.c_size_t * 8)()
        _check(lib().kivi_seq_buffer_bytes(self.c(), cap_tokens, arr), "kivi_seq_buffer_bytes")
        return list(arr)

    def seq_bytes(self, cap_tokens: int) -> int:
        return int(lib().kivi_seq_bytes(self.c(), cap_tokens))

    def decode_workspace_bytes(self, nseq: int, max_kv_len: int) -> int:
        return int(lib().kivi_decode_workspace_bytes(self.c(), nseq, max_kv_len))

    def decode_multi_workspace_bytes(self, nseq: int, n_query: int, max_kv_len: int) -> int:
        return int(lib().kivi_decode_multi_workspace_bytes(self.c(), nseq, n_query, max_kv_len))


# ---------------------------------------------------------------- codec
def quant_keys(cfg: Config, x: torch.Tensor):
    """Per-channel key quantization. x [S][T][D] (cfg dtype, T % G == 0) ->
    codes [S][T][D*k_bits/8] u8, scale/zero [S][T/G][D] (fp16 bit patterns as int16)."""
    _require_cuda(x, "x")
    S, T, D = x.shape
    codes = torch.empty((S, T, cfg.k_row_bytes), dtype=torch.uint8, device=x.device)
    scale = torch.empty((S, T // cfg.group, D), dtype=torch.int16, device=x.device)
    zero = torch.empty_like(scale)
    _check(lib().kivi_quant_keys(cfg.c(), S, T, _ptr(x), _ptr(codes), _ptr(scale), _ptr(zero),
                                 _stream(x.device)), "kivi_quant_keys")
    return codes, scale, zero


def quant_values(cfg: Config, x: torch.Tensor):
    """Per-token value quantization. x [S][T][D] -> codes [S][T][D*v_bits/8], scale/zero [S][T][D/G]."""
    _require_cuda(x, "x")
    S, T, D = x.shape
    codes = torch.empty((S, T, cfg.v_row_bytes), dtype=torch.uint8, device=x.device)
    scale = torch.empty((S, T, D // cfg.group), dtype=torch.int16, device=x.device)
    zero = torch.empty_like(scale)
    _check(lib().kivi_quant_values(cfg.c(), S, T, _ptr(x), _ptr(codes), _ptr(scale), _ptr(zero),
                                   _stream(x.device)), "kivi_quant_values")
    return codes, scale, zero


# ---------------------------------------------------------------- cache
class KVCache:
    """Packed KIVI caches of `nseq` sequences on one device, each with `cap_tokens`
    packed capacity, in the buffer layout of include/kivi.h. Buffers of all
    sequences live in one allocation per kind; the device array of kivi_seq
    records points into them."""

    def __init__(self, cfg: Config, nseq: int, cap_tokens: int, device="cuda", paged: bool = False,
                 page_seed: int = 0, spare_pages: int = 0):
        """paged: the packed buffers are one pool of G-token pages shared by all sequences,
        each sequence's groups mapped through a block table (kivi.h, paged layout); the pool
        has nseq * cap_tokens / G + spare_pages pages, handed out in a seeded random order."""
        if cap_tokens % cfg.group:
            raise ValueError("cap_tokens must be a multiple of G")
        if not torch.cuda.is_available():
            raise RuntimeError("KIVI kernels need a CUDA device; there is no CPU path")
        self.cfg, self.nseq, self.cap, self.paged = cfg, nseq, cap_tokens, paged
        self.device = torch.device(device)
        H, D, G = cfg.num_kv_heads, cfg.head_dim, cfg.group
        dev = self.device
        if paged:
            npg = nseq * (cap_tokens // G) + spare_pages
            self.k_codes = torch.zeros((npg, H, G, cfg.k_row_bytes), dtype=torch.uint8, device=dev)
            self.v_codes = torch.zeros((npg, H, G, cfg.v_row_bytes), dtype=torch.uint8, device=dev)
            self.k_scale = torch.zeros((npg, H, D), dtype=torch.int16, device=dev)
            self.v_scale = torch.zeros((npg, H, G, D // G), dtype=torch.int16, device=dev)
            perm = np.random.default_rng(page_seed).permutation(npg)[:nseq * (cap_tokens // G)]
            self.block_tables = torch.from_numpy(perm.reshape(nseq, cap_tokens // G).astype(np.int32)).to(dev)
        else:
            self.k_codes = torch.zeros((nseq, H, cap_tokens, cfg.k_row_bytes), dtype=torch.uint8, device=dev)
            self.v_codes = torch.zeros((nseq, H, cap_tokens, cfg.v_row_bytes), dtype=torch.uint8, device=dev)
            self.k_scale = torch.zeros((nseq, H, cap_tokens // G, D), dtype=torch.int16, device=dev)
            self.v_scale = torch.zeros((nseq, H, cap_tokens, D // G), dtype=torch.int16, device=dev)
            self.block_tables = None
        self.k_zero = torch.zeros_like(self.k_scale)
        self.v_zero = torch.zeros_like(self.v_scale)
        self.k_res = torch.zeros((nseq, H, cfg.ring, D), dtype=cfg.torch_dtype, device=dev)
        self.v_res = torch.zeros_like(self.k_res)
        self.kv_len = torch.zeros(nseq, dtype=torch.int32, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.max_len = 0            # host upper bound on every kv_len
        self._ws = None
        rec = np.zeros((nseq, SEQ_STRUCT_BYTES // 8), dtype=np.uint64)
        for b in range(nseq):
            for i, name in enumerate(SEQ_FIELDS):
                t = getattr(self, name)
                rec[b, i] = t.data_ptr() if (paged and name not in ("k_res", "v_res")) else t[b].data_ptr()
            # cap_tokens (low half), flags (high half); then the block table pointer
            rec[b, 8] = np.uint64(cap_tokens) | (np.uint64(SEQ_PAGED if paged else 0) << np.uint64(32))
            rec[b, 9] = np.uint64(self.block_tables[b].data_ptr()) if paged else np.uint64(0)
        self.seqs = torch.from_numpy(rec.view(np.uint8).reshape(-1)).to(dev)

    @property
    def max_tokens(self) -> int:
        return self.cap + self.cfg.ring - 1

    # -------------------------------------------------------------- append
    def append_ptrs(self, k_ptrs: torch.Tensor, v_ptrs: torch.Tensor, n_new: torch.Tensor, max_new: int) -> None:
        """Low-level append: device int64 arrays of per-sequence new-token pointers
        ([Hkv][n_b][D] each) and a device int32 array of counts (all <= max_new)."""
        _check(lib().kivi_append_flush(self.cfg.c(), self.nseq, _ptr(self.seqs), _ptr(self.kv_len),
                                       _ptr(k_ptrs), _ptr(v_ptrs), _ptr(n_new), int(max_new),
                                       _ptr(self.status), _stream(self.device)), "kivi_append_flush")
        self.max_len = min(self.max_len + int(max_new), self.max_tokens)

    def append(self, k_new, v_new) -> None:
        """Append new tokens. Either dense tensors [nseq][Hkv][n][D] (n tokens for
        every sequence) or lists of per-sequence tensors [Hkv][n_b][D]."""
        if isinstance(k_new, torch.Tensor):
            _require_cuda(k_new, "k_new")
            _require_cuda(v_new, "v_new")
            k_list, v_list = list(k_new.unbind(0)), list(v_new.unbind(0))
        else:
            k_list, v_list = list(k_new), list(v_new)
        assert len(k_list) == len(v_list) == self.nseq
        n = [int(k.shape[1]) for k in k_list]
        for k, v in zip(k_list, v_list):
            assert k.dtype == self.cfg.torch_dtype and v.shape == k.shape
            assert k.shape[1] == 0 or (k.is_contiguous() and v.is_contiguous())
        kp = torch.tensor([k.data_ptr() if k.numel() else 0 for k in k_list], dtype=torch.int64).to(self.device)
        vp = torch.tensor([v.data_ptr() if v.numel() else 0 for v in v_list], dtype=torch.int64).to(self.device)
        nn = torch.tensor(n, dtype=torch.int32).to(self.device)
        self.append_ptrs(kp, vp, nn, max(n) if n else 0)
        # keep the sources alive until the stream has consumed them
        self._keep = (k_list, v_list, kp, vp, nn)

    # -------------------------------------------------------------- attention
    def workspace(self, max_kv_len: int | None = None) -> torch.Tensor:
        need = self.cfg.decode_workspace_bytes(self.nseq, self.max_len if max_kv_len is None else max_kv_len)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=self.device)
        return self._ws

    def decode(self, q: torch.Tensor, out: torch.Tensor | None = None, softmax_scale: float | None = None,
               max_kv_len: int | None = None) -> torch.Tensor:
        """Decode attention. q [nseq][Hq][D] (cfg dtype) -> out [nseq][Hq][D] fp32."""
        _require_cuda(q, "q")
        cfg = self.cfg
        if out is None:
            out = torch.empty((self.nseq, cfg.num_q_heads, cfg.head_dim), dtype=torch.float32, device=q.device)
        scale = 1.0 / cfg.head_dim ** 0.5 if softmax_scale is None else softmax_scale
        mkl = self.max_len if max_kv_len is None else max_kv_len
        ws = self.workspace(mkl)
        _check(lib().kivi_decode_attn(cfg.c(), self.nseq, _ptr(self.seqs), _ptr(self.kv_len), _ptr(q), _ptr(out),
                                      float(scale), int(mkl), _ptr(ws), ws.numel(), _ptr(self.status),
                                      _stream(self.device)), "kivi_decode_attn")
        return out

    def decode_multi(self, q: torch.Tensor, out: torch.Tensor | None = None, softmax_scale: float | None = None,
                     max_kv_len: int | None = None) -> torch.Tensor:
        """Multi-query attention of each sequence's n_query newest tokens (already appended),
        query i attending causally to positions [0, kv_len - n_query + i].
        q [nseq][n_query][Hq][D] (cfg dtype) -> out [nseq][n_query][Hq][D] fp32."""
        _require_cuda(q, "q")
        cfg = self.cfg
        nq = int(q.shape[1])
        if out is None:
            out = torch.empty((self.nseq, nq, cfg.num_q_heads, cfg.head_dim), dtype=torch.float32, device=q.device)
        scale = 1.0 / cfg.head_dim ** 0.5 if softmax_scale is None else softmax_scale
        mkl = self.max_len if max_kv_len is None else max_kv_len
        need = cfg.decode_multi_workspace_bytes(self.nseq, nq, mkl)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=self.device)
        ws = self._ws
        _check(lib().kivi_decode_multi_attn(cfg.c(), self.nseq, _ptr(self.seqs), _ptr(self.kv_len), nq, _ptr(q),
                                            _ptr(out), float(scale), int(mkl), _ptr(ws), ws.numel(),
                                            _ptr(self.status), _stream(self.device)), "kivi_decode_multi_attn")
        return out

    # -------------------------------------------------------------- inspection
    def seq_numpy(self, b: int) -> dict:
        """Host copies of sequence b's buffers in the contiguous layout (a paged sequence's
        pages gathered through its block table; uint8 / uint16 views), and kv_len."""
        d = {}
        for name in SEQ_FIELDS:
            t = getattr(self, name)
            if self.paged and name not in ("k_res", "v_res"):
                t = t[self.block_tables[b].long()]          # [groups][H][...] in group order
                t = t.transpose(0, 1)                         # [H][groups][...]
                if name in ("k_codes", "v_codes", "v_scale", "v_zero"):
                    t = t.reshape(t.shape[0], -1, t.shape[-1])   # [H][cap][...]
            else:
                t = t[b]
            t = t.contiguous().cpu()
            if t.dtype in (torch.int16, torch.float16, torch.bfloat16):
                d[name] = t.view(torch.int16).numpy().view(np.uint16)
            else:
                d[name] = t.numpy()
        d["kv_len"] = int(self.kv_len[b].item())
        return d
