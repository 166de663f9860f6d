"""Exact-arithmetic model of the block-floating-point rounding of a head's
half-D partial sums that the CTA pairs exchange (the forward's senders in
smqa_fwd.cu round partial scores this way, the backward's P/dS threads in
smqa_bwd.cu partial S and sm_scale dP, 32 slots at a time): the
exponent comes from the fp32 maximum times (1 + 2^-15), every mantissa then
stays within +-32767 without a clamp, and the absolute error stays within
2^-15 (1 + 2^-14) of the largest scaled partial.

Each fp32 step is emulated with numpy float32 (IEEE round-to-nearest-even);
the fused multiply-add x * f + 1.5 * 2^23 + 32768 is exact up to one rounding
to an integer (its result lies in [2^23, 2^24), where the fp32 spacing is 1),
so it is modelled as round-half-even of the exact product x * f."""
from fractions import Fraction

import numpy as np
import pytest

MARGIN = np.float32(1.0 + 2.0 ** -15)


def _exponent(v: np.float32) -> int:
    e = int((np.float32(v).view(np.uint32) >> 23) & 0xFF) - 127
    return min(max(e, -100), 100)


def _round_half_even(q: Fraction) -> int:
    fl = q.numerator // q.denominator
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        return fl + 1
    return fl


def _quantise(x: np.ndarray, s1: np.float32):
    """Mantissas n and exponent e of one head's block, as the sender forms them."""
    mx = np.max(np.abs(x)).astype(np.float32)
    v = np.float32(np.float32(mx * s1) * MARGIN)
    e = _exponent(v)
    f = np.float32(s1 * np.float32(2.0 ** (14 - e)))
    n = [_round_half_even(Fraction(float(xi)) * Fraction(float(f))) for xi in x]
    return n, e, Fraction(float(mx)) * Fraction(float(s1))


def _check(x: np.ndarray, s1: np.float32):
    n, e, vmax = _quantise(x.astype(np.float32), np.float32(s1))
    assert max(abs(k) for k in n) <= 32767
    if vmax == 0:
        return
    bound = Fraction(2) ** -15 * (1 + Fraction(2) ** -14) * vmax
    for k, xi in zip(n, x.astype(np.float32)):
        exact = Fraction(float(xi)) * Fraction(float(s1))
        assert abs(Fraction(k) * Fraction(2) ** (e - 14) - exact) <= bound


@pytest.mark.parametrize("seed", range(20))
def test_random_blocks(seed):
    rng = np.random.default_rng(seed)
    s1 = np.float32(rng.uniform(0.01, 0.2) * 1.4426950408889634)
    x = (rng.standard_normal(64) * 10.0 ** rng.uniform(-3, 3)).astype(np.float32)
    _check(x, s1)


@pytest.mark.parametrize("k", range(-30, 31, 3))
def test_maxima_at_power_of_two_boundaries(k):
    """The largest |x| * s1 just below, at and just above 2^k: the cases a
    plain floor(log2) exponent would round up to 32768."""
    rng = np.random.default_rng(1000 + k)
    for s1 in (np.float32(1.0), np.float32(0.0625 * 1.4426950408889634),
               np.float32(0.04419417 * 1.4426950408889634)):
        target = np.float32(np.float32(2.0 ** k) / s1)
        for step in range(-3, 4):
            mx = np.nextafter(target, np.float32(np.inf) if step > 0 else np.float32(0),
                              dtype=np.float32) if step else target
            for _ in range(abs(step) - 1):
                mx = np.nextafter(mx, np.float32(np.inf) if step > 0 else np.float32(0),
                                  dtype=np.float32)
            x = (rng.uniform(-1, 1, 64) * mx).astype(np.float32)
            x[rng.integers(64)] = -mx if rng.integers(2) else mx
            _check(x, s1)


def test_all_zero_block():
    n, e, _ = _quantise(np.zeros(64, dtype=np.float32), np.float32(0.09))
    assert e == -100 and all(k == 0 for k in n)


@pytest.mark.parametrize("seed", range(12))
def test_backward_blocks_at_gradient_scale(seed):
    """The backward's use: 32-value blocks of partial S (scale sm_scale log2 e)
    and partial dP (scale sm_scale) at magnitudes from gradient-sized (dO of
    2^-30 gives partial dP near 1e-9) to large; the bound is relative to the
    block's largest value, so it holds at every scale down to the exponent
    clamp at 2^-100."""
    rng = np.random.default_rng(50 + seed)
    for s1 in (np.float32(0.04419417 * 1.4426950408889634), np.float32(0.04419417)):
        for mag in (2.0 ** -60, 2.0 ** -30, 2.0 ** -20, 1.0, 2.0 ** 10):
            x = (rng.standard_normal(32) * mag).astype(np.float32)
            _check(x, s1)
