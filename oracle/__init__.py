"""KIVI oracle: a plain CPU statement of the KIVI codec and decode attention.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg import this package. The product library never
imports, links or executes it, and it never imports the product package.

The arithmetic lives in ``kivi_oracle.c`` (plain C, fp32 quantizer with one
IEEE operation per step, fp64 attention). This module only compiles it with
gcc and marshals numpy arrays through ctypes. See the C file's header for the
passages each function follows and the readings taken where the pages are
silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kivi_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libkivi_oracle.so")
# A test may point the wrapper at a deliberately broken build of the oracle (a
# "mutant") to check that the pins catch the mistake; nothing else sets this.
_LIB_OVERRIDE = os.environ.get("KIVI_ORACLE_LIB")
_CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-shared", "-fPIC", "-Wall", "-Wno-unused-function"]

F16, BF16 = 0, 1
OK, ERR_ARG, ERR_CAPACITY = 0, 1, 3

_lock = threading.Lock()
_lib = None


def compile_source(src: str, out: str) -> str:
    """Compile a C source with the oracle's flags into a shared library at `out`."""
    subprocess.run(["gcc", *_CFLAGS, src, "-o", out, "-lm"], check=True)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into oracle/_build/ (rebuilt when the source is newer)."""
    if _LIB_OVERRIDE:
        return _LIB_OVERRIDE
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Cfg(ctypes.Structure):
    _fields_ = [("k_bits", ctypes.c_int32), ("v_bits", ctypes.c_int32), ("group", ctypes.c_int32),
                ("residual", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("num_q_heads", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class _Seq(ctypes.Structure):
    _fields_ = [("k_codes", ctypes.c_void_p), ("k_scale", ctypes.c_void_p), ("k_zero", ctypes.c_void_p),
                ("v_codes", ctypes.c_void_p), ("v_scale", ctypes.c_void_p), ("v_zero", ctypes.c_void_p),
                ("k_res", ctypes.c_void_p), ("v_res", ctypes.c_void_p), ("cap", ctypes.c_int32)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            L.orc_f32_to_f16.restype = ctypes.c_uint16
            L.orc_f32_to_f16.argtypes = [ctypes.c_float]
            L.orc_f16_to_f32.restype = ctypes.c_float
            L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
            for name in ("orc_f32_to_f16_array", "orc_f16_to_f32_array"):
                getattr(L, name).argtypes = [P, P, ctypes.c_int64]
                getattr(L, name).restype = None
            for name in ("orc_quant_keys", "orc_quant_values"):
                getattr(L, name).argtypes = [ctypes.POINTER(_Cfg), ctypes.c_int, ctypes.c_int, P, P, P, P]
                getattr(L, name).restype = ctypes.c_int
            L.orc_append.argtypes = [ctypes.POINTER(_Cfg), ctypes.POINTER(_Seq), P, P, P, ctypes.c_int]
            L.orc_append.restype = ctypes.c_int
            L.orc_decode_seq.argtypes = [ctypes.POINTER(_Cfg), ctypes.POINTER(_Seq), ctypes.c_int64, P,
                                         ctypes.c_double, P, ctypes.c_int, ctypes.c_int]
            L.orc_decode_seq.restype = None
            L.orc_decode_multi_seq.argtypes = [ctypes.POINTER(_Cfg), ctypes.POINTER(_Seq), ctypes.c_int64,
                                               ctypes.c_int, P, ctypes.c_double, P]
            L.orc_decode_multi_seq.restype = ctypes.c_int
            L.orc_n_packed.argtypes = [ctypes.POINTER(_Cfg), ctypes.c_int64]
            L.orc_n_packed.restype = ctypes.c_int64
            L.orc_kv_bytes_plain.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                             ctypes.c_double, ctypes.c_double]
            L.orc_kv_bytes_plain.restype = ctypes.c_double
            L.orc_seq_bytes.argtypes = [ctypes.POINTER(_Cfg), ctypes.c_int64]
            L.orc_seq_bytes.restype = ctypes.c_int64
            L.orc_get_code.argtypes = [P, ctypes.c_int, ctypes.c_int]
            L.orc_get_code.restype = ctypes.c_int
            _lib = L
    return _lib


@dataclass(frozen=True)
class Cfg:
    """KIVI configuration: code widths, G, R, head_dim, query and kv heads, storage dtype.
    `bits` sets both code widths; k_bits / v_bits, when given, set one of them."""
    bits: int = 2
    group: int = 32
    residual: int = 128
    head_dim: int = 128
    num_q_heads: int = 1
    num_kv_heads: int = 1
    dtype: int = F16
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
    def k_row_bytes(self) -> int:
        return self.head_dim * self.k_bits // 8

    @property
    def v_row_bytes(self) -> int:
        return self.head_dim * self.v_bits // 8

    @property
    def ring(self) -> int:
        return self.residual + self.group


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a: np.ndarray) -> np.ndarray:
    if a.dtype in (np.float16,):
        return np.ascontiguousarray(a).view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return np.ascontiguousarray(a)


# ---------------------------------------------------------------- conversions
def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().orc_f32_to_f16_array(_p(x), _p(out), x.size)
    return out


def f16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float32)
    lib().orc_f16_to_f32_array(_p(h), _p(out), h.size)
    return out


# ---------------------------------------------------------------- codec
def quant_keys(cfg: Cfg, x_bits: np.ndarray):
    """x_bits [S][T][D] uint16 dtype patterns -> codes [S][T][D*b/8], scale/zero [S][T/G][D] (fp16 bits)."""
    x = _u16(x_bits)
    S, T, D = x.shape
    assert D == cfg.head_dim and T % cfg.group == 0
    codes = np.zeros((S, T, cfg.k_row_bytes), np.uint8)
    scale = np.zeros((S, T // cfg.group, D), np.uint16)
    zero = np.zeros_like(scale)
    rc = lib().orc_quant_keys(cfg.c(), S, T, _p(x), _p(codes), _p(scale), _p(zero))
    assert rc == OK
    return codes, scale, zero


def quant_values(cfg: Cfg, x_bits: np.ndarray):
    """x_bits [S][T][D] -> codes [S][T][D*b/8], scale/zero [S][T][D/G] (fp16 bits)."""
    x = _u16(x_bits)
    S, T, D = x.shape
    assert D == cfg.head_dim
    codes = np.zeros((S, T, cfg.v_row_bytes), np.uint8)
    scale = np.zeros((S, T, D // cfg.group), np.uint16)
    zero = np.zeros_like(scale)
    rc = lib().orc_quant_values(cfg.c(), S, T, _p(x), _p(codes), _p(scale), _p(zero))
    assert rc == OK
    return codes, scale, zero


def unpack_codes(cfg: Cfg, rows: np.ndarray) -> np.ndarray:
    """[..., D*b/8] packed rows -> [..., D] integer codes, using the oracle's packing rule
    (b, 2 or 4, from the row length)."""
    rows = np.ascontiguousarray(rows, dtype=np.uint8)
    bits = rows.shape[-1] * 8 // cfg.head_dim
    assert bits in (2, 4) and rows.shape[-1] == cfg.head_dim * bits // 8
    flat = rows.reshape(-1, rows.shape[-1])
    out = np.empty((flat.shape[0], cfg.head_dim), np.int32)
    L = lib()
    for i in range(flat.shape[0]):
        r = np.ascontiguousarray(flat[i])
        for d in range(cfg.head_dim):
            out[i, d] = L.orc_get_code(_p(r), d, bits)
    return out.reshape(*rows.shape[:-1], cfg.head_dim)


def n_packed(cfg: Cfg, L: int) -> int:
    return int(lib().orc_n_packed(cfg.c(), L))


# ---------------------------------------------------------------- sequence cache
class SeqCache:
    """One sequence's cache buffers in the library's layout, held in numpy."""

    def __init__(self, cfg: Cfg, cap: int):
        assert cap % cfg.group == 0
        H, D, G = cfg.num_kv_heads, cfg.head_dim, cfg.group
        self.cfg, self.cap = cfg, cap
        self.k_codes = np.zeros((H, cap, cfg.k_row_bytes), np.uint8)
        self.k_scale = np.zeros((H, cap // G, D), np.uint16)
        self.k_zero = np.zeros((H, cap // G, D), np.uint16)
        self.v_codes = np.zeros((H, cap, cfg.v_row_bytes), np.uint8)
        self.v_scale = np.zeros((H, cap, D // G), np.uint16)
        self.v_zero = np.zeros((H, cap, D // G), np.uint16)
        self.k_res = np.zeros((H, cfg.ring, D), np.uint16)
        self.v_res = np.zeros((H, cfg.ring, D), np.uint16)
        self.kv_len = np.zeros(1, np.int32)

    def _c(self) -> _Seq:
        return _Seq(self.k_codes.ctypes.data, self.k_scale.ctypes.data, self.k_zero.ctypes.data,
                    self.v_codes.ctypes.data, self.v_scale.ctypes.data, self.v_zero.ctypes.data,
                    self.k_res.ctypes.data, self.v_res.ctypes.data, self.cap)

    @property
    def L(self) -> int:
        return int(self.kv_len[0])

    def append(self, k_bits: np.ndarray, v_bits: np.ndarray) -> int:
        """k_bits, v_bits [Hkv][n_new][D] dtype patterns. Returns the oracle status."""
        k, v = _u16(k_bits), _u16(v_bits)
        assert k.shape == v.shape and k.shape[0] == self.cfg.num_kv_heads
        return int(lib().orc_append(self.cfg.c(), self._c(), _p(self.kv_len), _p(k), _p(v), k.shape[1]))

    def decode(self, q_bits: np.ndarray, scale: float, hq0: int = 0, nhq: int | None = None) -> np.ndarray:
        """q_bits [Hq][D] -> out [Hq][D] fp64 (rows outside the requested head range are NaN)."""
        q = _u16(q_bits)
        Hq = self.cfg.num_q_heads
        nhq = Hq - hq0 if nhq is None else nhq
        out = np.full((Hq, self.cfg.head_dim), np.nan, np.float64)
        lib().orc_decode_seq(self.cfg.c(), self._c(), self.L, _p(q), float(scale), _p(out), hq0, nhq)
        return out

    def decode_multi(self, q_bits: np.ndarray, scale: float) -> np.ndarray:
        """q_bits [n_query][Hq][D]: the n_query newest tokens' queries, query i attending causally
        to positions [0, L - n_query + i] -> out [n_query][Hq][D] fp64."""
        q = _u16(q_bits)
        nq = q.shape[0]
        assert q.shape[1:] == (self.cfg.num_q_heads, self.cfg.head_dim)
        out = np.full(q.shape, np.nan, np.float64)
        rc = lib().orc_decode_multi_seq(self.cfg.c(), self._c(), self.L, nq, _p(q), float(scale), _p(out))
        if rc != OK:
            raise ValueError(f"orc_decode_multi_seq: status {rc}")
        return out


def kv_bytes_plain(layers: int, kv_heads: int, head_dim: int, bits: float, seq: float, batch: float) -> float:
    return float(lib().orc_kv_bytes_plain(layers, kv_heads, head_dim, bits, seq, batch))


def seq_bytes(cfg: Cfg, cap: int) -> int:
    return int(lib().orc_seq_bytes(cfg.c(), cap))
