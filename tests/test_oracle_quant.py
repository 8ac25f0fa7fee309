"""Pins the oracle's quantizer and packing (CPU only).

Sources: KV-cache quantization guide (pigeon), "How it works", step 3 (the
asymmetric formula); tract #2329 "KIVI-style KV-cache quantization", commit
"Training-free affine quantize<->dequantize": round-trip error <= scale/2 and
shrinking with bits.
"""
import numpy as np
import pytest

from conftest import read_table


def _f16(x):
    return np.asarray(x, dtype=np.float16)


@pytest.mark.parametrize("row", read_table("quantizer_cases.txt"), ids=lambda r: r[0])
def test_quantizer_golden(oracle_lib, row):
    name, bits, xs, d16, m16, codes = row
    x = _f16([float(v) for v in xs.split()])
    c, d, m = oracle_lib.quantize(x, int(bits))
    assert int(d) == int(d16, 16), name
    assert int(m) == int(m16, 16), name
    assert c.tolist() == [int(v) for v in codes.split()], name


@pytest.mark.parametrize("row", read_table("packing_cases.txt"), ids=lambda r: r[0])
def test_packing_golden(oracle_lib, row):
    name, bits, codes, packed = row
    codes = np.array([int(v) for v in codes.split()], dtype=np.uint8)
    expect = np.array([int(v, 16) for v in packed.split()], dtype=np.uint8)
    got = oracle_lib.pack_row(codes, int(bits))
    assert got.tolist() == expect.tolist(), name
    assert oracle_lib.unpack_row(got, codes.size, int(bits)).tolist() == codes.tolist()


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("L", [32, 64, 128])
def test_pack_unpack_roundtrip(oracle_lib, bits, L):
    rng = np.random.default_rng(bits * 1000 + L)
    codes = rng.integers(0, 1 << bits, size=L, dtype=np.uint8)
    packed = oracle_lib.pack_row(codes, bits)
    assert packed.size == L * bits // 8
    assert np.array_equal(oracle_lib.unpack_row(packed, L, bits), codes)
    # every code bit is used exactly once: distinct one-hot codes give distinct bits
    total = 0
    for j in range(L):
        one = np.zeros(L, dtype=np.uint8)
        one[j] = (1 << bits) - 1
        total += int(np.unpackbits(oracle_lib.pack_row(one, bits)).sum())
    assert total == L * bits


def _dequant(codes, d16, m16):
    dq = np.float64(np.uint16(d16).view(np.float16))
    mn = np.float64(np.uint16(m16).view(np.float16))
    return mn + codes.astype(np.float64) * dq, dq


@pytest.mark.parametrize("bits", [1, 2, 3, 4, 5, 6, 7, 8])
@pytest.mark.parametrize("dist", ["normal", "outlier", "tiny", "wide"])
def test_roundtrip_bound(oracle_lib, bits, dist):
    """|x - x̂| <= Δ16/2 + 2^-22 (max - min) for every element (tract #2329:
    "round-trip error <= scale/2"); the extra term covers the two fp32
    roundings that decide a code at a half-way point.  When Δ16 is an fp16
    subnormal (< 2^-14) it carries an absolute rounding error up to 2^-25, which
    the top code multiplies, so (2^b - 1) 2^-25 is added there.  A zero Δ16
    only happens when the range is below 255 * 2^-25, and then x̂ = min."""
    rng = np.random.default_rng(17 + bits)
    for trial in range(400):
        n = int(rng.integers(2, 200))
        x = rng.standard_normal(n)
        if dist == "outlier":
            x[rng.integers(0, n)] *= 40
        elif dist == "tiny":
            x *= 1e-6
        elif dist == "wide":
            x *= 3000
        x = _f16(x)
        c, d16, m16 = oracle_lib.quantize(x, bits)
        assert c.max() <= (1 << bits) - 1
        xf = x.astype(np.float64)
        xh, dq = _dequant(c, d16, m16)
        rng_ = xf.max() - xf.min()
        err = np.abs(xf - xh).max()
        if dq == 0:
            assert rng_ <= 255 * 2.0 ** -25
            assert np.all(xh == xf.min())
        else:
            sub = ((1 << bits) - 1) * 2.0 ** -25 if dq < 2.0 ** -14 else 0.0
            assert err <= dq / 2 + 2.0 ** -22 * rng_ + sub, (trial, err, dq)
            if dq >= 2.0 ** -14:
                # normal Δ16: the clamp costs at most (2^b-1) Δ 2^-11 <= Δ16/8
                assert err <= 0.5 * dq * (1 + 2.0 ** -9) + 2.0 ** -22 * rng_
        assert np.float64(np.uint16(m16).view(np.float16)) == xf.min()


def test_error_shrinks_with_bits(oracle_lib):
    rng = np.random.default_rng(5)
    errs = {}
    for bits in range(1, 9):
        e = []
        for _ in range(200):
            x = _f16(rng.standard_normal(128))
            c, d16, m16 = oracle_lib.quantize(x, bits)
            xh, _ = _dequant(c, d16, m16)
            e.append(np.abs(x.astype(np.float64) - xh).mean())
        errs[bits] = float(np.mean(e))
    assert all(errs[b + 1] < errs[b] for b in range(1, 8))
    # uniform-quantizer scaling: each extra bit roughly halves the step
    assert errs[2] / errs[4] > 3.0 and errs[4] / errs[8] > 8.0
    assert all(1.5 < errs[b] / errs[b + 1] < 3.0 for b in range(2, 8))


def test_codes_span_levels(oracle_lib):
    # the min maps to code 0 and the max to the top code (no dropped level)
    rng = np.random.default_rng(9)
    for bits in range(1, 9):
        for _ in range(100):
            x = _f16(rng.standard_normal(64) * 5)
            c, d16, m16 = oracle_lib.quantize(x, bits)
            xf = x.astype(np.float32)
            assert c[np.argmin(xf)] == 0
            assert c[np.argmax(xf)] == (1 << bits) - 1
