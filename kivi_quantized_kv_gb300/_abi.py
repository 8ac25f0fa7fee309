"""ctypes binding of libkivi.so (the C ABI declared in include/kivi.h).

Argument marshalling only: every step of the cache runs in the library's CUDA
kernels.  If the library is missing this module raises; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkivi.so")
LIB_PATH_DEBUG = os.path.join(HERE, "libkivi_debug.so")

KIVI_OK, KIVI_EINVAL, KIVI_EALIGN, KIVI_ECAPACITY, KIVI_ENOSPC, KIVI_ECUDA, KIVI_ENULL, KIVI_ESCRATCH = range(8)

# every entry point include/kivi.h declares
EXPORTS = (
    "kivi_cache_bytes", "kivi_cache_create", "kivi_cache_destroy", "kivi_append", "kivi_append_ragged",
    "kivi_cache_tokens", "kivi_prefill_attn_ragged", "kivi_cache_restore", "kivi_debug_inject_launch_failure",
    "kivi_debug_set_wait_limit",
    "kivi_decode_attn", "kivi_append_decode_attn", "kivi_append_decode_attn_host", "kivi_decode_attn_host",
    "kivi_decode_attn_noalloc", "kivi_prefill_attn", "kivi_prefill_scratch_bytes", "kivi_prefill_bytes",
    "kivi_read_error", "kivi_set_num_splits", "kivi_cache_layout", "kivi_layout_for",
    "kivi_decode_bytes", "kivi_status_string",
)


class KiviParams(ctypes.Structure):
    _fields_ = [
        ("bits", ctypes.c_int32), ("group", ctypes.c_int32), ("residual", ctypes.c_int32),
        ("sinks", ctypes.c_int32), ("h_q", ctypes.c_int32), ("h_kv", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("batch", ctypes.c_int32),
        ("max_tokens", ctypes.c_int64), ("window", ctypes.c_int64),
        ("outlier_permille", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("rope_base", ctypes.c_double),
    ]


class KiviLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "n_slots", "sink_k", "sink_v", "res_k", "res_v", "groups",
        "block_bytes", "blk_kq", "blk_ks", "blk_vq", "blk_vs",
        "unit_bytes", "cache_bytes", "workspace_offset", "workspace_bytes", "arena_bytes",
        "tokens", "n_sink", "n_groups", "n_res")] + [("max_splits", ctypes.c_int32), ("reserved", ctypes.c_int32)] + [
        (n, ctypes.c_int64) for n in ("blk_ko", "blk_vo", "n_outliers", "out_entries")]


class KiviError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None


def lib_path() -> str:
    """libkivi.so, or the checked build libkivi_debug.so when the environment
    sets KIVI_DEBUG_CHECKS=1."""
    if os.environ.get("KIVI_DEBUG_CHECKS", "0") == "1":
        return LIB_PATH_DEBUG
    return LIB_PATH


def lib():
    """Loads the library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        how = ("`python -m kivi_quantized_kv_gb300.build --debug-checks`" if path == LIB_PATH_DEBUG else
               "`python -c 'import __graft_entry__ as g; g.build()'`")
        raise ImportError(f"{path} is missing: build it with {how} (needs nvcc)")
    L = ctypes.CDLL(path)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
    P = ctypes.POINTER
    sig = {
        "kivi_cache_bytes": (ctypes.c_size_t, [P(KiviParams)]),
        "kivi_cache_create": (ctypes.c_int, [P(KiviParams), vp, ctypes.c_size_t, vp, P(vp)]),
        "kivi_cache_destroy": (None, [vp]),
        "kivi_append": (ctypes.c_int, [vp, vp, vp, i64, vp]),
        "kivi_append_ragged": (ctypes.c_int, [vp, vp, vp, P(i64), i64, vp]),
        "kivi_cache_tokens": (ctypes.c_int, [vp, P(i64)]),
        "kivi_cache_restore": (ctypes.c_int, [P(KiviParams), vp, ctypes.c_size_t, P(i64), vp, P(vp)]),
        "kivi_debug_inject_launch_failure": (ctypes.c_int, [i64]),
        "kivi_debug_set_wait_limit": (ctypes.c_int, [i64]),
        "kivi_prefill_attn_ragged": (ctypes.c_int, [vp, vp, vp, P(i64), i64, vp, ctypes.c_size_t, vp]),
        "kivi_decode_attn": (ctypes.c_int, [vp, vp, vp, vp]),
        "kivi_append_decode_attn": (ctypes.c_int, [vp, vp, vp, vp, vp, vp]),
        "kivi_append_decode_attn_host": (ctypes.c_int, [vp, vp, vp, vp, vp, vp]),
        "kivi_decode_attn_host": (ctypes.c_int, [vp, vp, vp, vp]),
        "kivi_decode_attn_noalloc": (ctypes.c_int, [vp, vp, vp, vp]),
        "kivi_prefill_attn": (ctypes.c_int, [vp, vp, vp, i64, vp, ctypes.c_size_t, vp]),
        "kivi_prefill_scratch_bytes": (ctypes.c_size_t, [vp, i64]),
        "kivi_prefill_bytes": (i64, [vp, i64]),
        "kivi_read_error": (ctypes.c_int, [vp, P(ctypes.c_uint32), vp]),
        "kivi_set_num_splits": (ctypes.c_int, [vp, i32]),
        "kivi_cache_layout": (ctypes.c_int, [vp, P(KiviLayout)]),
        "kivi_layout_for": (ctypes.c_int, [P(KiviParams), P(KiviLayout)]),
        "kivi_decode_bytes": (i64, [vp]),
        "kivi_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().kivi_status_string(status).decode()


def check(status: int, what: str) -> None:
    if status != KIVI_OK:
        raise KiviError(status, what)
