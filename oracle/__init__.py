"""CPU oracle for the KIVI quantized KV cache (test infrastructure).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may import
this package.  It loads ``libkivi_oracle.so`` (plain C++ compiled with
``-O2 -ffp-contract=off``), which shares no code with the CUDA library.

Sources of each computation are cited in ``kivi_oracle.cpp``; in short:
  * KV-cache quantization guide (pigeon), "How it works", steps 1-5;
  * tract #2458 "quantized KV-cache storage op (int8/int4)": f32 attention
    sinks, frozen per-channel key blocks;
  * tract #2329 "KIVI-style KV-cache quantization", "What's in the PR": GQA;
    the op takes the query with the new keys and values and returns an output
    shaped like the query.

fp16 arrays are passed as numpy ``float16`` (or their ``uint16`` bit view).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from .build import build as _build, LIB_PATH

_lib = None


class KoParams(ctypes.Structure):
    _fields_ = [
        ("bits", ctypes.c_int32), ("group", ctypes.c_int32), ("residual", ctypes.c_int32),
        ("sinks", ctypes.c_int32), ("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("max_tokens", ctypes.c_int64), ("window", ctypes.c_int64),
        ("outlier_permille", ctypes.c_int32), ("window_mode", ctypes.c_int32),
        ("rope_base", ctypes.c_double),
    ]


class KoLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "n_slots", "sink_k", "sink_v", "res_k", "res_v", "groups", "block_bytes",
        "blk_kq", "blk_ks", "blk_vq", "blk_vs", "blk_ko", "blk_vo", "n_outliers", "out_entries", "unit_bytes", "cache_bytes")]


def lib():
    """Load (building first if needed) the oracle shared library."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        _build()
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER
    u16p, u8p, f32p, f64p = P(ctypes.c_uint16), P(ctypes.c_uint8), P(ctypes.c_float), P(ctypes.c_double)
    vp = ctypes.c_void_p
    sig = {
        "ko_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
        "ko_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
        "ko_f32_to_f16_array": (None, [f32p, u16p, ctypes.c_int64]),
        "ko_f16_to_f32_array": (None, [u16p, f32p, ctypes.c_int64]),
        "ko_quantize": (None, [u16p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, u8p, u16p, u16p]),
        "ko_pack_row": (ctypes.c_int, [u8p, ctypes.c_int32, ctypes.c_int32, u8p]),
        "ko_unpack_row": (ctypes.c_int, [u8p, ctypes.c_int32, ctypes.c_int32, u8p]),
        "ko_validate": (ctypes.c_int, [P(KoParams)]),
        "ko_layout_of": (ctypes.c_int, [P(KoParams), P(KoLayout)]),
        "ko_state_of": (None, [P(KoParams), ctypes.c_int64, P(ctypes.c_int64), P(ctypes.c_int64), P(ctypes.c_int64)]),
        "ko_create": (ctypes.c_int, [P(KoParams), P(vp)]),
        "ko_destroy": (None, [vp]),
        "ko_append": (ctypes.c_int, [vp, u16p, u16p, ctypes.c_int64]),
        "ko_tokens": (ctypes.c_int64, [vp]),
        "ko_groups": (ctypes.c_int64, [vp]),
        "ko_residual_count": (ctypes.c_int64, [vp]),
        "ko_arena": (vp, [vp]),
        "ko_dequant_unit": (ctypes.c_int, [vp, ctypes.c_int32, ctypes.c_int32, f64p, f64p, u8p]),
        "ko_decode_attn": (ctypes.c_int, [vp, u16p, f64p, ctypes.c_int32]),
        "ko_prefill_attn": (ctypes.c_int, [vp, u16p, ctypes.c_int64, f64p, ctypes.c_int32]),
        "ko_decode_bytes": (ctypes.c_int64, [vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


# ---------------------------------------------------------------- primitives
def f32_to_f16(x: np.ndarray) -> np.ndarray:
    """fp32 -> fp16 bit patterns (round to nearest even)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    lib().ko_f32_to_f16_array(_ptr(x, ctypes.c_float), _ptr(out, ctypes.c_uint16), x.size)
    return out


def f16_to_f32(h: np.ndarray) -> np.ndarray:
    h = _u16(h)
    out = np.empty(h.shape, dtype=np.float32)
    lib().ko_f16_to_f32_array(_ptr(h, ctypes.c_uint16), _ptr(out, ctypes.c_float), h.size)
    return out


def quantize(x, bits: int):
    """One asymmetric quantization of a 1-D fp16 vector -> (codes u8, Δ16, min16)."""
    x = _u16(np.asarray(x))
    assert x.ndim == 1
    codes = np.empty(x.size, dtype=np.uint8)
    d16 = ctypes.c_uint16()
    m16 = ctypes.c_uint16()
    lib().ko_quantize(_ptr(x, ctypes.c_uint16), x.size, 1, bits, _ptr(codes, ctypes.c_uint8),
                      ctypes.byref(d16), ctypes.byref(m16))
    return codes, np.uint16(d16.value), np.uint16(m16.value)


def pack_row(codes, bits: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros(codes.size * bits // 8, dtype=np.uint8)
    rc = lib().ko_pack_row(_ptr(codes, ctypes.c_uint8), codes.size, bits, _ptr(out, ctypes.c_uint8))
    if rc != 0:
        raise ValueError("row length * bits must be a multiple of 32 (b in 2, 4, 8) or 8 (other b)")
    return out


def unpack_row(packed, L: int, bits: int) -> np.ndarray:
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros(L, dtype=np.uint8)
    rc = lib().ko_unpack_row(_ptr(packed, ctypes.c_uint8), L, bits, _ptr(out, ctypes.c_uint8))
    if rc != 0:
        raise ValueError("row length * bits must be a multiple of 32 (b in 2, 4, 8) or 8 (other b)")
    return out


# ---------------------------------------------------------------- cache
@dataclass
class Params:
    bits: int
    group: int
    residual: int
    sinks: int
    h_q: int
    h_kv: int
    head_dim: int
    batch: int
    max_tokens: int = 0
    window: int = 0
    outlier_permille: int = 0
    rope_base: float = 0.0
    # the other reading of a window composed with sinks: a pure window, in
    # which the sinks expire like any other token (0 = sinks stay visible)
    window_mode: int = 0

    def c(self) -> KoParams:
        return KoParams(self.bits, self.group, self.residual, self.sinks, self.h_q, self.h_kv,
                        self.head_dim, self.batch, self.max_tokens, self.window, self.outlier_permille,
                        self.window_mode, self.rope_base)


def validate(p: Params) -> int:
    cp = p.c()
    return lib().ko_validate(ctypes.byref(cp))


def layout(p: Params) -> dict:
    cp, lo = p.c(), KoLayout()
    if lib().ko_layout_of(ctypes.byref(cp), ctypes.byref(lo)) != 0:
        raise ValueError(f"invalid parameters {p}")
    return {n: getattr(lo, n) for n, _ in KoLayout._fields_}


def state_of(p: Params, T: int):
    cp = p.c()
    a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    lib().ko_state_of(ctypes.byref(cp), T, ctypes.byref(a), ctypes.byref(b), ctypes.byref(c))
    return a.value, b.value, c.value


class Cache:
    """The oracle cache: host arena bytes identical in layout to the device cache region."""

    def __init__(self, p: Params):
        self.p = p
        cp = p.c()
        h = ctypes.c_void_p()
        rc = lib().ko_create(ctypes.byref(cp), ctypes.byref(h))
        if rc != 0:
            raise ValueError(f"invalid parameters {p}")
        self._h = h
        self.layout = layout(p)

    def __del__(self):
        if getattr(self, "_h", None) is not None and _lib is not None:
            _lib.ko_destroy(self._h)
            self._h = None

    def append(self, k_new, v_new) -> int:
        """k_new, v_new: [B, H_kv, n, d] fp16.  Returns the status code."""
        k = _u16(k_new)
        v = _u16(v_new)
        B, H, n, d = k.shape
        assert (B, H, d) == (self.p.batch, self.p.h_kv, self.p.head_dim) and v.shape == k.shape
        return lib().ko_append(self._h, _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16), n)

    @property
    def T(self) -> int:
        return lib().ko_tokens(self._h)

    @property
    def n_groups(self) -> int:
        return lib().ko_groups(self._h)

    @property
    def n_res(self) -> int:
        return lib().ko_residual_count(self._h)

    def arena(self) -> np.ndarray:
        """A copy of the cache bytes."""
        n = self.layout["cache_bytes"]
        ptr = lib().ko_arena(self._h)
        if n == 0:
            return np.zeros(0, dtype=np.uint8)
        return np.ctypeslib.as_array(ctypes.cast(ptr, ctypes.POINTER(ctypes.c_uint8)), shape=(n,)).copy()

    def unit(self, b: int, h: int) -> np.ndarray:
        ub = self.layout["unit_bytes"]
        u = b * self.p.h_kv + h
        return self.arena()[u * ub:(u + 1) * ub]

    def dequant_unit(self, b: int, h: int):
        T, d = self.T, self.p.head_dim
        K = np.zeros((T, d), dtype=np.float64)
        V = np.zeros((T, d), dtype=np.float64)
        vis = np.zeros(T, dtype=np.uint8)
        rc = lib().ko_dequant_unit(self._h, b, h, _ptr(K, ctypes.c_double), _ptr(V, ctypes.c_double),
                                   _ptr(vis, ctypes.c_uint8))
        assert rc == 0
        return K, V, vis.astype(bool)

    def decode_attn(self, q, threads: int = 1) -> np.ndarray:
        """q: [B, H_q, d] fp16 -> out [B, H_q, d] fp64."""
        qq = _u16(q)
        assert qq.shape == (self.p.batch, self.p.h_q, self.p.head_dim)
        out = np.zeros(qq.shape, dtype=np.float64)
        rc = lib().ko_decode_attn(self._h, _ptr(qq, ctypes.c_uint16), _ptr(out, ctypes.c_double), threads)
        assert rc == 0
        return out

    def prefill_attn(self, q, threads: int = 1) -> np.ndarray:
        """q: [B, M, H_q, d] fp16, the M newest tokens as queries -> out [B, M, H_q, d] fp64."""
        qq = _u16(q)
        assert qq.ndim == 4 and qq.shape[0] == self.p.batch and qq.shape[2:] == (self.p.h_q, self.p.head_dim)
        out = np.zeros(qq.shape, dtype=np.float64)
        rc = lib().ko_prefill_attn(self._h, _ptr(qq, ctypes.c_uint16), qq.shape[1], _ptr(out, ctypes.c_double),
                                   threads)
        assert rc == 0, rc
        return out

    def decode_bytes(self) -> int:
        return lib().ko_decode_bytes(self._h)
