"""The C ABI on a machine without a GPU: the library loads, exports every entry
point include/kivi.h declares, sizes arenas, and rejects bad arguments on the
host before touching a device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def abi():
    from kivi_quantized_kv_gb300.build import build
    build()
    from kivi_quantized_kv_gb300 import _abi
    _abi.lib()
    return _abi


def header_functions():
    with open(os.path.join(ROOT, "include", "kivi.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(kivi_\w+)\(", text, flags=re.M)))


def test_exports_every_declared_symbol(abi):
    names = header_functions()
    assert len(names) >= 10, names
    lib = ctypes.CDLL(abi.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(abi.EXPORTS) == names


def test_checked_build_exports_the_same_symbols(abi):
    """KIVI_DEBUG_CHECKS=1 builds libkivi_debug.so with the same entry points;
    the binding picks it only when the environment asks for it."""
    from kivi_quantized_kv_gb300.build import build
    path = build(debug_checks=True)
    assert path.endswith("libkivi_debug.so") and path != abi.LIB_PATH
    lib = ctypes.CDLL(path)
    for n in header_functions():
        assert hasattr(lib, n), n
    assert abi.lib_path() == abi.LIB_PATH   # the product library unless KIVI_DEBUG_CHECKS=1


def params(**kw):
    from kivi_quantized_kv_gb300 import KiviConfig
    base = dict(bits=4, group=32, residual=32, sinks=4, h_q=4, h_kv=4, head_dim=64, batch=1, max_tokens=256)
    base.update(kw)
    return KiviConfig(**base)


def test_cache_bytes_covers_the_oracle_layout(abi, oracle_lib):
    from kivi_quantized_kv_gb300 import cache_bytes
    for kw in (dict(), dict(bits=2, head_dim=128, batch=8, h_q=32, h_kv=32, max_tokens=4096),
               dict(bits=8, group=64, residual=64, window=4096, max_tokens=0, h_q=32, h_kv=8, batch=32,
                    head_dim=128),
               dict(bits=3, head_dim=128, outlier_permille=10), dict(bits=3, outlier_permille=10),
               dict(bits=2, group=64, residual=64, outlier_permille=50)):
        cfg = params(**kw)
        lay = oracle_lib.layout(oracle_lib.Params(**cfg.__dict__))
        nb = cache_bytes(cfg)
        assert nb >= lay["cache_bytes"]
        # the workspace is small next to the cache: partials, counters, staging
        assert nb - lay["cache_bytes"] <= 8 * 1024 * 1024 + lay["cache_bytes"] // 100


@pytest.mark.parametrize("kw", [dict(bits=0), dict(bits=9), dict(bits=16), dict(bits=3, group=128, residual=128), dict(bits=5, group=16, residual=32), dict(head_dim=96), dict(group=8), dict(group=40),
                                dict(residual=16), dict(residual=48), dict(sinks=-1), dict(h_q=6),
                                dict(h_q=36, h_kv=4), dict(window=16, max_tokens=0), dict(window=-1),
                                dict(batch=0), dict(max_tokens=-1),
                                # outlier tables: 0..50 per mille, 2 to 4 bits, G a multiple of 32,
                                # 3 bits at head dim 128 only
                                dict(outlier_permille=-1), dict(outlier_permille=51),
                                dict(outlier_permille=10, bits=8), dict(outlier_permille=10, bits=1),
                                dict(outlier_permille=10, group=16, residual=32),
                                 # pre-RoPE keys: base 0 or in (1, 1e7], G 32 or 64, no outlier tables
                                dict(rope_base=1.0), dict(rope_base=-3.0), dict(rope_base=2e7),
                                dict(rope_base=10000.0, group=16, residual=32),
                                dict(rope_base=10000.0, group=128, residual=128),
                                dict(rope_base=10000.0, outlier_permille=10)])
def test_invalid_parameters_are_rejected(abi, kw):
    from kivi_quantized_kv_gb300 import cache_bytes
    cfg = params(**kw)
    assert cache_bytes(cfg) == 0
    p = cfg.c()
    h = ctypes.c_void_p()
    buf = ctypes.create_string_buffer(1 << 16)
    st = abi.lib().kivi_cache_create(ctypes.byref(p), ctypes.c_void_p(ctypes.addressof(buf)), 1 << 16, None,
                                     ctypes.byref(h))
    assert st == abi.KIVI_EINVAL


def test_host_side_errors_before_any_device_call(abi):
    L = abi.lib()
    p = params().c()
    need = L.kivi_cache_bytes(ctypes.byref(p))
    h = ctypes.c_void_p()
    assert L.kivi_cache_create(ctypes.byref(p), None, need, None, ctypes.byref(h)) == abi.KIVI_ENULL
    assert L.kivi_cache_create(None, ctypes.c_void_p(4096), need, None, ctypes.byref(h)) == abi.KIVI_ENULL
    assert L.kivi_cache_create(ctypes.byref(p), ctypes.c_void_p(4096 + 16), need, None,
                               ctypes.byref(h)) == abi.KIVI_EALIGN
    assert L.kivi_cache_create(ctypes.byref(p), ctypes.c_void_p(4096), need - 1, None,
                               ctypes.byref(h)) == abi.KIVI_ENOSPC
    assert L.kivi_append(None, None, None, 1, None) == abi.KIVI_ENULL
    assert L.kivi_decode_attn(None, None, None, None) == abi.KIVI_ENULL
    assert L.kivi_decode_attn_host(None, None, None, None) == abi.KIVI_ENULL
    assert L.kivi_set_num_splits(None, 2) == abi.KIVI_ENULL
    assert L.kivi_cache_layout(None, None) == abi.KIVI_ENULL
    assert L.kivi_decode_bytes(None) == -1
    for s in range(7):
        assert abi.status_string(s)
    assert abi.status_string(99) == "unknown status"


def test_python_binding_fails_loudly_without_library(monkeypatch):
    from kivi_quantized_kv_gb300 import _abi
    monkeypatch.setattr(_abi, "_lib", None)
    monkeypatch.setattr(_abi, "LIB_PATH", "/nonexistent/libkivi.so")
    with pytest.raises(ImportError):
        _abi.lib()


def test_fault_injection_arming_is_host_only(abi):
    L = abi.lib()
    assert L.kivi_debug_inject_launch_failure(-1) == abi.KIVI_EINVAL
    assert L.kivi_debug_inject_launch_failure(3) == abi.KIVI_OK
    assert L.kivi_debug_inject_launch_failure(0) == abi.KIVI_OK


def test_wait_limit_setting_is_host_only(abi):
    L = abi.lib()
    assert L.kivi_debug_set_wait_limit(-1) == abi.KIVI_EINVAL
    assert L.kivi_debug_set_wait_limit(5) == abi.KIVI_OK
    assert L.kivi_debug_set_wait_limit(0) == abi.KIVI_OK


def test_restore_rejects_bad_arguments_before_any_device_call(abi):
    import ctypes
    p = params().c()
    h = ctypes.c_void_p()
    toks = (ctypes.c_int64 * 1)(5)
    L = abi.lib()
    assert L.kivi_cache_restore(ctypes.byref(p), None, 1 << 20, toks, None, ctypes.byref(h)) == abi.KIVI_ENULL
    assert L.kivi_cache_restore(ctypes.byref(p), ctypes.c_void_p(256), 1 << 30, None, None,
                                ctypes.byref(h)) == abi.KIVI_ENULL
    bad = (ctypes.c_int64 * 1)(-1)
    assert L.kivi_cache_restore(ctypes.byref(p), ctypes.c_void_p(256), 1 << 30, bad, None,
                                ctypes.byref(h)) == abi.KIVI_EINVAL
    over = (ctypes.c_int64 * 1)(257)   # max_tokens 256
    assert L.kivi_cache_restore(ctypes.byref(p), ctypes.c_void_p(256), 1 << 30, over, None,
                                ctypes.byref(h)) == abi.KIVI_EINVAL
    assert L.kivi_cache_restore(ctypes.byref(p), ctypes.c_void_p(258), 1 << 30, toks, None,
                                ctypes.byref(h)) == abi.KIVI_EALIGN


LAYOUT_CASES = [
    dict(),
    dict(bits=2, head_dim=128, batch=8, h_q=32, h_kv=32, max_tokens=4096),
    dict(bits=8, group=64, residual=64, window=4096, max_tokens=0, h_q=32, h_kv=8, batch=32, head_dim=128),
    dict(bits=3, head_dim=128, outlier_permille=10),
    dict(bits=2, group=64, residual=64, outlier_permille=50),
    dict(bits=4, group=32, residual=96, sinks=0, outlier_permille=1, window=200, max_tokens=0),
    dict(bits=5, group=64, residual=64, rope_base=10000.0),
    dict(bits=1, group=32, residual=32, sinks=7, rope_base=500000.0, head_dim=128),
    dict(bits=7, group=32, residual=64, head_dim=128, sinks=3),
    dict(bits=6, group=64, residual=128, head_dim=64, sinks=0, window=300, max_tokens=0),
]


@pytest.mark.parametrize("kw", LAYOUT_CASES)
def test_host_layout_equals_the_oracle_layout(abi, oracle_lib, kw):
    """The library's byte layout (kivi_layout_for, host only) against the
    oracle's own computation of it, offset by offset: the cache region the
    GPU tests compare byte for byte starts from the same map."""
    cfg = params(**kw)
    p = cfg.c()
    lay = abi.KiviLayout()
    assert abi.lib().kivi_layout_for(ctypes.byref(p), ctypes.byref(lay)) == abi.KIVI_OK
    ref = oracle_lib.layout(oracle_lib.Params(**cfg.__dict__))
    for name in ("n_slots", "sink_k", "sink_v", "res_k", "res_v", "groups", "block_bytes", "blk_kq", "blk_ks",
                 "blk_vq", "blk_vs", "blk_ko", "blk_vo", "n_outliers", "unit_bytes", "cache_bytes"):
        assert getattr(lay, name) == ref[name], name
    assert lay.out_entries == ref["out_entries"]
    assert lay.tokens == 0 and lay.n_groups == 0 and lay.workspace_offset >= lay.cache_bytes
    assert lay.arena_bytes == cache_bytes_of(abi, p)


def cache_bytes_of(abi, p):
    return abi.lib().kivi_cache_bytes(ctypes.byref(p))


def test_host_layout_rejects_what_create_rejects(abi):
    lay = abi.KiviLayout()
    bad = params(bits=9).c()
    assert abi.lib().kivi_layout_for(ctypes.byref(bad), ctypes.byref(lay)) == abi.KIVI_EINVAL
    assert abi.lib().kivi_layout_for(None, ctypes.byref(lay)) == abi.KIVI_ENULL
    good = params().c()
    assert abi.lib().kivi_layout_for(ctypes.byref(good), None) == abi.KIVI_ENULL
