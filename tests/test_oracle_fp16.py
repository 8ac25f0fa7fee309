"""Pins the oracle's hand-written IEEE binary16 conversion against numpy's.

The oracle writes fp32 -> fp16 (round to nearest, ties to even) from the
format definition; every quantizer decision depends on it, so it is checked
exhaustively over all 2^32 fp32 bit patterns (NaNs only need to stay NaN)
and all 2^16 fp16 patterns in the other direction.
"""
import numpy as np
import pytest


def test_f16_to_f32_exhaustive(oracle_lib):
    h = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ours = oracle_lib.f16_to_f32(h)
    ref = h.view(np.float16).astype(np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _check_chunk(oracle_lib, start, n):
    bits = np.arange(start, start + n, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    ours = oracle_lib.f32_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    bad = (ours != ref) & ~nan
    if bad.any():
        i = int(np.flatnonzero(bad)[0])
        raise AssertionError(f"fp32 0x{int(bits[i]):08x}: oracle 0x{int(ours[i]):04x} numpy 0x{int(ref[i]):04x}")
    assert np.isnan(ours[nan].view(np.float16)).all()


def test_f32_to_f16_boundaries(oracle_lib):
    # every fp32 whose magnitude lies where binary16 rounding happens
    # (subnormal, normal and overflow boundaries), for one sign, at a stride,
    # plus exact ties and halfway cases around each binary16 value
    h = np.arange(0x7C01, dtype=np.uint32).astype(np.uint16)
    mid = h.view(np.float16).astype(np.float32)
    base = mid.view(np.uint32).astype(np.int64)
    # fp32 neighbours and the exact midpoints between consecutive binary16s
    cand = [base + k for k in (-2, -1, 0, 1, 2)]
    f = h.view(np.float16).astype(np.float64)
    mids = ((f[:-1] + f[1:]) / 2).astype(np.float32).view(np.uint32).astype(np.int64)
    cand += [mids + k for k in (-1, 0, 1)]
    allb = np.unique(np.clip(np.concatenate(cand), 0, 0xFFFFFFFF))
    allb = np.concatenate([allb, allb | 0x80000000]).astype(np.uint32)
    x = allb.view(np.float32)
    ours = oracle_lib.f32_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])


@pytest.mark.slow
def test_f32_to_f16_exhaustive(oracle_lib):
    chunk = 1 << 26
    for start in range(0, 1 << 32, chunk):
        _check_chunk(oracle_lib, start, chunk)


def test_f32_to_f16_strided_sample(oracle_lib):
    # a fast deterministic sample across the whole fp32 range (every 97th pattern
    # of 2^32 would take minutes; a random 2^24 sample plus a stride covers all
    # exponents)
    rng = np.random.default_rng(0)
    bits = rng.integers(0, 1 << 32, size=1 << 24, dtype=np.uint64).astype(np.uint32)
    bits = np.concatenate([bits, np.arange(0, 1 << 32, 4099, dtype=np.uint64).astype(np.uint32)])
    x = bits.view(np.float32)
    ours = oracle_lib.f32_to_f16(x)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
