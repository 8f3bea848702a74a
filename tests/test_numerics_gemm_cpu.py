"""CPU checks of the exactness arguments behind the prefill GEMM's operands.

The GEMM prepass scales each F32 token row by 2^s, s = 15 - e for the row
maximum M = f * 2^e (f in [0.5, 1)), so the scaled maximum lies in
[2^14, 2^15); F16 rows are only scaled up (s >= 0). The split precision then
stores hi = fp16(x 2^s) and lo = fp16(x 2^s - hi), the difference taken in f32;
the single-fp16 precision stores hi alone. The weights enter as the fp16 values
(q - 1) d. These tests restate that arithmetic (fp16 rounding is numpy's
float16 cast, round to nearest even) and check with exact rationals:
  - the scaling is exact and puts the row maximum in [2^14, 2^15), so hi is finite;
  - the f32 difference x 2^s - hi is exact;
  - |x 2^s - hi - lo| <= 2^-22 |x 2^s| + 2^-25, i.e. |x - x_held| <= 2^-22 |x| +
    2^-39 M: 22 bits of each element's own value down to 2^-18 M, and an
    absolute floor of 2^-39 M below that; hi alone: 2^-11 |x| + 2^-39 M;
  - every product (q - 1) d * hi (and * lo) is exact in f32 for every fp16 d
    with |2 d| <= 65504, so the tensor core's products add no rounding.
Nothing here is shared with the CUDA sources.
"""
from fractions import Fraction

import numpy as np

F32 = np.float32
F16 = np.float16


def row_shift(x, f16_row: bool = False) -> int:
    m = float(np.max(np.abs(x.astype(np.float64))))
    if m == 0.0 or not np.isfinite(m):
        return 0
    e = int(np.frexp(m)[1])
    s = 15 - e
    return max(s, 0) if f16_row else s


def split_row(x, s):
    """(x 2^s in f32, hi, lo, whether the f32 difference was exact)."""
    xs = (x.astype(np.float64) * 2.0 ** s).astype(F32)
    hi = xs.astype(F16)
    diff = (xs - hi.astype(F32)).astype(F32)
    lo = diff.astype(F16)
    exact = all(Fraction(float(d)) == Fraction(float(a)) - Fraction(float(h))
                for d, a, h in zip(diff, xs, hi))
    return xs, hi, lo, exact


def _rows():
    g = np.random.default_rng(21)
    rows = []
    for t in range(200):
        x = g.standard_normal(256)
        x *= 10.0 ** g.uniform(-8, 8, 256) if t % 2 else 1.0
        x *= 10.0 ** g.uniform(-30, 30)
        if t % 5 == 0:
            x[g.integers(0, 256)] = 30.0 * 10.0 ** g.uniform(-3, 3)
        rows.append(x.astype(F32))
    rows.append(np.array([65504.0 * 4, -1e-30, 3.0, 2.0 ** -140], dtype=F32))
    rows.append(np.array([2.0 ** 15, 2.0 ** 14, -(2.0 ** 15) + 1], dtype=F32))
    rows.append(np.array([1e38, -3e38, 1.0, 1e-38], dtype=F32))
    return rows


def test_row_scaling_is_exact_and_bounds_the_maximum():
    for x in _rows():
        s = row_shift(x)
        xs, hi, _, _ = split_row(x, s)
        for a, b in zip(x, xs):
            if abs(float(a)) * 2.0 ** s >= 2.0 ** -126:  # f32 normal after scaling
                assert Fraction(float(b)) == Fraction(float(a)) * Fraction(2) ** s
        mx = float(np.max(np.abs(xs.astype(np.float64))))
        assert 2.0 ** 14 <= mx < 2.0 ** 15, (s, mx)
        assert np.all(np.isfinite(hi.astype(np.float64)))


def test_split_error_bound():
    for x in _rows():
        s = row_shift(x)
        m = Fraction(float(np.max(np.abs(x.astype(np.float64)))))
        xs, hi, lo, exact = split_row(x, s)
        assert exact
        for a, b, h, l in zip(x, xs, hi, lo):
            xv = Fraction(float(b))
            held = Fraction(float(h)) + Fraction(float(l))
            assert abs(xv - held) <= Fraction(2) ** -22 * abs(xv) + Fraction(2) ** -25
            # the same in the caller's units
            err = abs(Fraction(float(a)) - held * Fraction(2) ** -s)
            assert err <= Fraction(2) ** -22 * abs(Fraction(float(a))) + Fraction(2) ** -39 * m + \
                Fraction(2) ** -149 * Fraction(2) ** -s  # f32 underflow of x 2^s, if any
            # hi alone (single-fp16 precision)
            assert abs(xv - Fraction(float(h))) <= Fraction(2) ** -11 * abs(xv) + Fraction(2) ** -25


def test_f16_rows_are_only_scaled_up_and_stay_exact():
    g = np.random.default_rng(22)
    for t in range(100):
        x = (g.standard_normal(128) * 10.0 ** g.uniform(-6, 4)).astype(F16)
        s = row_shift(x.astype(F32), f16_row=True)
        assert s >= 0
        xs = x.astype(np.float64) * 2.0 ** s
        # scaled up by a power of two, an fp16 value stays an exact fp16 value
        # unless it overflows, which s = max(15 - e, 0) rules out
        assert np.array_equal(xs.astype(F16).astype(np.float64), xs)


def test_weight_times_activation_products_are_exact_in_f32():
    g = np.random.default_rng(23)
    bits = g.integers(0, 0x7C00, 4000).astype(np.uint16)  # finite non-negative halves
    d = bits.view(F16).astype(np.float64)
    d = d[np.abs(2 * d) <= 65504.0]
    d = np.concatenate([d, [2.0 ** -24, 65504.0 / 2, 0.0]])
    acts = np.concatenate([g.standard_normal(500) * 10.0 ** g.uniform(-8, 4, 500),
                           [2.0 ** 15 - 16, 2.0 ** -24, -(2.0 ** -14)]]).astype(F16).astype(np.float64)
    for q in (0, 1, 2, 3):
        w = (q - 1) * d
        assert np.array_equal(w.astype(F16).astype(np.float64), w)  # (q - 1) d exact in fp16
        prod = np.multiply.outer(w[:300], acts)
        assert np.array_equal(prod.astype(F32).astype(np.float64), prod)
