"""The flush kernel forms a code as rint((x - min) * RN(1 / step)) and falls
back to the IEEE quotient (x - min) / step only when that product lies within
2^-11 of a half-integer.  This checks the arithmetic fact the shortcut rests
on, in IEEE float32 on the CPU (numpy rounds every float32 operation to
nearest even, as the kernel's _rn intrinsics do): wherever the shortcut is
taken, it rounds to the same integer as the quotient, for steps anywhere in
the fp16 range (subnormals included), every code width 1..8, and numerators
chosen right next to the rounding boundaries.  The kernel's bytes are compared
with the oracle's on the GPU."""
import numpy as np


def _steps(rng, n):
    # positive finite fp16 values, from the smallest subnormal to 65504
    bits = rng.integers(1, 0x7C00, size=n, dtype=np.uint16)
    return bits.view(np.float16).astype(np.float32)


def _check(a, dq):
    a = a.astype(np.float32)
    dq = dq.astype(np.float32)
    q_div = a / dq
    rq = np.float32(1.0) / dq
    q_mul = a * rq
    fast = np.abs(q_mul - np.floor(q_mul) - np.float32(0.5)) >= np.float32(2.0 ** -11)
    assert np.array_equal(np.rint(q_mul[fast]), np.rint(q_div[fast]))
    return fast.mean()


def test_shortcut_rounds_like_the_quotient():
    rng = np.random.default_rng(1234)
    n = 400_000
    for b in range(1, 9):
        top = np.float32(2 ** b - 1)
        dq = _steps(rng, n)
        # the unrounded step the fp16 value came from lies within a rounding
        # of it: the quotient stays below 2 top < 512
        a = (rng.random(n, dtype=np.float32) * top * np.float32(1.999)) * dq
        frac_fast = _check(a, dq)
        assert frac_fast > 0.99
        assert float(np.max(a / dq)) < 512.0


def test_shortcut_next_to_half_integers():
    rng = np.random.default_rng(99)
    n = 200_000
    dq = _steps(rng, n)
    k = rng.integers(0, 510, size=n).astype(np.float32)
    base = (k + np.float32(0.5)) * dq
    for ulps in (-64, -8, -2, -1, 0, 1, 2, 8, 64):
        a = base.copy()
        step = np.float32(np.inf) if ulps > 0 else np.float32(-np.inf)
        for _ in range(abs(ulps)):
            a = np.nextafter(a, step).astype(np.float32)
        a = np.maximum(a, np.float32(0.0))
        _check(a, dq)
