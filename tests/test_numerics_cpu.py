"""CPU checks of the exactness arguments behind the fp4 decode path (ncols = 1).

The fp4 mat-vec multiplies the codes, read as e2m1 values q/2, by 16 e2m1
pieces of each block's activations: for a block of 64 with M = max|x| =
f * 2^e (f in [0.5, 1)), v = x * 2^(2 - e) (max|v| in [2, 4)) and
p_i = e2m1(r_i * 4^i), r_0 = v, r_{i+1} = r_i - p_i * 4^-i. These tests
restate e2m1 round-to-nearest-even from the format's definition (sign, 2
exponent bits with bias 1, 1 mantissa bit; 0.5 is the one subnormal step) and
check, on random and boundary values and with exact rational arithmetic:
  - every subtraction r_i - p_i * 4^-i is exact in f32, every scaled residual
    after the first piece lies in [-2, 2] (no piece saturates), and after 16
    pieces |r_16| <= 2^-32;
  - the three groups H = sum_{i<6} 4^-i C_i, M = sum_{6<=i<12}, L = sum_{i>=12}
    of a block's per-piece sums C_i = sum_k (q_k/2) p_ik, formed in f32 in the
    epilogue's order, are exact, and so are the same groups for all-ones codes;
  - so (H_C - H_1) + (M_C - M_1) + (L_C - L_1) is within two roundings of the
    exact sum over the nonzero weights: a zero weight (code 1) under an element
    of any size contributes nothing.
Nothing here is shared with the CUDA sources.
"""
from fractions import Fraction

import numpy as np
import pytest

# e2m1 magnitudes with their mantissa bit (for ties to even)
_E2M1 = [(0.0, 0), (0.5, 1), (1.0, 0), (1.5, 1), (2.0, 0), (3.0, 1), (4.0, 0), (6.0, 1)]
F32 = np.float32


def e2m1_rne(v: float) -> float:
    a = abs(v)
    best = None
    for mag, mbit in _E2M1:
        d = abs(a - mag)
        if best is None or d < best[0] or (d == best[0] and mbit == 0 and best[2] == 1):
            best = (d, mag, mbit)
    return float(np.copysign(best[1], v))


def split_pieces(v, n: int = 16):
    """Pieces of an f32 v with every step in f32, as the prep kernel does;
    also returns the scaled residuals and whether each subtraction was exact."""
    r = F32(v)
    pieces, scaled, exact = [], [], True
    for i in range(n):
        s = F32(r * F32(4.0 ** i))
        scaled.append(float(s))
        p = e2m1_rne(float(s))
        pieces.append(p)
        step = F32(F32(p) * F32(4.0 ** -i))
        nr = F32(r - step)
        exact &= Fraction(float(nr)) == Fraction(float(r)) - Fraction(float(step))
        r = nr
    return pieces, scaled, float(r), exact


def block_scale(x):
    """e of the block maximum (M = f * 2^e, f in [0.5, 1)); 0 for an all-zero block."""
    m = float(np.max(np.abs(x)))
    return 0 if m == 0.0 else int(np.frexp(np.float32(m))[1])


def test_e2m1_grid_rounding():
    assert e2m1_rne(0.25) == 0.0          # tie between 0 and 0.5 -> even (0)
    assert e2m1_rne(0.75) == 1.0          # tie between 0.5 and 1 -> even (1)
    assert e2m1_rne(1.25) == 1.0          # tie between 1 and 1.5 -> even (1)
    assert e2m1_rne(2.5) == 2.0           # tie between 2 and 3 -> even (2)
    assert e2m1_rne(3.5) == 4.0           # tie between 3 and 4 -> even (4)
    assert e2m1_rne(-1.7) == -1.5
    assert e2m1_rne(5.0) == 4.0           # tie between 4 and 6 -> even (4)


def test_piece_split_residual_bound():
    g = np.random.default_rng(1)
    vals = list(g.uniform(-4.0, 4.0, 3000))
    vals += list(g.uniform(-1.0, 1.0, 1000) * 2.0 ** g.integers(-60, 0, 1000))
    # boundaries: the largest magnitudes, grid points, ties, tiny values
    vals += [3.999999761581421, -3.999999761581421, 2.0, -2.0, 1.0, 0.25, 0.75, 2.5, 3.5,
             1e-8, -1e-8, 0.0, 2.0 ** -40]
    for v in vals:
        v = float(F32(v))
        pieces, scaled, r, exact = split_pieces(v)
        assert exact, v
        assert all(abs(s) <= 2.0 for s in scaled[1:]), v
        assert abs(r) <= 2.0 ** -32, (v, r)
        assert Fraction(v) == sum(Fraction(p) * Fraction(4) ** -i for i, p in enumerate(pieces)) \
            + Fraction(r)


def test_block_scale_puts_the_maximum_in_2_to_4():
    g = np.random.default_rng(3)
    for _ in range(500):
        x = (g.standard_normal(64) * 10.0 ** g.uniform(-30, 30)).astype(F32)
        e = block_scale(x)
        v = np.abs(x.astype(np.float64)) * 2.0 ** (2 - e)
        assert 2.0 <= v.max() < 4.0


def _groups_f32(c):
    """H, M, L of sum_i 4^-i c_i in f32, in the epilogue's FMA order."""
    def fma(a, b, acc):
        return F32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(acc)))
    gh = F32(F32(c[5]) * F32(2.0 ** -10))
    gm = F32(F32(c[11]) * F32(2.0 ** -22))
    gl = F32(F32(c[15]) * F32(2.0 ** -30))
    for i in range(4, -1, -1):
        gh = fma(c[i], 4.0 ** -i, gh)
    for i in range(10, 5, -1):
        gm = fma(c[i], 4.0 ** -i, gm)
    for i in range(14, 11, -1):
        gl = fma(c[i], 4.0 ** -i, gl)
    return gh, gm, gl


def _exact_groups(c):
    return (sum(Fraction(c[i]) * Fraction(4) ** -i for i in range(0, 6)),
            sum(Fraction(c[i]) * Fraction(4) ** -i for i in range(6, 12)),
            sum(Fraction(c[i]) * Fraction(4) ** -i for i in range(12, 16)))


@pytest.mark.parametrize("n", [64, 128])
def test_block_groups_exact_and_zero_weights_cancel(n):
    """Blocks of 64 (the 18-byte layout) and of 128 (the group-128 layout, whose
    activations are scaled per 128 elements)."""
    g = np.random.default_rng(2 + n)
    for trial in range(60 if n == 64 else 30):
        x = g.standard_normal(n).astype(F32)
        q = g.integers(0, 4, n)
        if trial % 3 == 0:   # a large element under a zero weight
            k = int(g.integers(0, n))
            x[k] = F32(3000.0 * (1 if trial % 2 else -1))
            q[k] = 1
            x[np.arange(n) != k] *= F32(1e-2)
        e = block_scale(x)
        v = [float(F32(float(xx) * 2.0 ** (2 - e))) for xx in x]
        P = np.array([split_pieces(vv)[0] for vv in v])          # [n][16]
        c = [sum((qq / 2.0) * P[k, i] for k, qq in enumerate(q)) for i in range(16)]
        b = [sum(0.5 * P[k, i] for k in range(n)) for i in range(16)]
        # each per-piece sum is an exact f32 (multiples of 1/4 below 2^9 or 2^10)
        assert all(float(F32(ci)) == ci and abs(ci) < 8 * n for ci in c + b)
        gc, gb = _groups_f32(c), _groups_f32(b)
        ec, eb = _exact_groups(c), _exact_groups(b)
        assert all(Fraction(float(a)) == x_ for a, x_ in zip(gc, ec))
        assert all(Fraction(float(a)) == x_ for a, x_ in zip(gb, eb))
        t = F32(F32(F32(gc[0] - gb[0]) + F32(gc[1] - gb[1])) + F32(gc[2] - gb[2]))
        exact = sum(ec) - sum(eb)          # = sum_k (q_k - 1)/2 * (v_k - r_k)
        nonzero = sum(abs(Fraction(int(qq) - 1, 2)) * abs(Fraction(vv))
                      for qq, vv in zip(q, v))
        assert abs(Fraction(float(t)) - exact) <= Fraction(1, 2 ** 22) * nonzero + Fraction(1, 2 ** 40)


def _magic_round(s, first_piece):
    """The prep's rounding in f32: |s| + 2^23 (first piece, |s| > 2) or
    fma(|s|, 2, 2^23) rounds to an integer in its low mantissa bits; returns
    (piece value, e2m1 nibble)."""
    M = F32(8388608.0)
    a = F32(abs(s))
    if first_piece and a > 2.0:
        a1 = F32(a + M)
        m = int(np.array(a1, dtype=np.float32).view(np.uint32)) & 7
        mag, nib = float(a1 - M), m + 2
    else:
        a2 = F32(Fraction(float(a)) * 2 + Fraction(float(M)))   # one rounding, as fma
        k = int(np.array(a2, dtype=np.float32).view(np.uint32)) & 7
        mag, nib = float(a2 - M) / 2.0, k
    sign = 8 if np.signbit(F32(s)) else 0
    return float(np.copysign(mag, s)), nib | sign


_NIBBLE = {0.0: 0, 0.5: 1, 1.0: 2, 1.5: 3, 2.0: 4, 3.0: 5, 4.0: 6, 6.0: 7}


def test_prep_rounding_equals_e2m1_round_to_nearest_even():
    g = np.random.default_rng(4)
    first = list(g.uniform(-4.0, 4.0, 4000)) + [2.0, 2.5, 3.5, 3.999999761581421, -2.5, -3.5]
    later = list(g.uniform(-2.0, 2.0, 4000)) + [0.25, 0.75, 1.25, 1.75, -0.25, -1.75, 2.0, 0.0]
    for vals, is_first in ((first, True), (later, False)):
        for v in vals:
            v = float(F32(v))
            piece, nib = _magic_round(v, is_first)
            want = e2m1_rne(v)
            assert piece == want, (v, piece, want)
            assert nib & 7 == _NIBBLE[abs(want)], (v, nib)
            assert (nib & 8 != 0) == bool(np.signbit(F32(v))), v
