"""CPU checks of the exactness arguments behind the e4m3 decode path (ncols 3-8).

That path multiplies the codes, read as the signed e4m3 values q - 1, by 5 e4m3
pieces of each block's activations. For a block of 64 with M = max|x| =
f * 2^e (f in [0.5, 1)): v = x * 2^(8 - e), so max|v| lies in [128, 256);
p_i = e4m3(r_i * 16^i), r_0 = v, r_{i+1} = r_i - p_i * 16^-i, every step in f32.
These tests restate e4m3 round-to-nearest-even from the format's definition
(sign, 4 exponent bits with bias 7, 3 mantissa bits; subnormal step 2^-9;
largest finite 448), pin that restatement against PyTorch's float8_e4m3fn
cast, and check on random, wide-range and boundary values with exact rational
arithmetic:
  - every subtraction r_i - p_i * 16^-i is exact in f32, and no piece's input
    r_i * 16^i exceeds 448 (no piece saturates);
  - v = sum_i p_i 16^-i + r_5 exactly, with |r_5| <= 2^-20 |v| + 2^-26, i.e.
    each element keeps 20 bits of its own value down to 2^-33 of its block's
    maximum (the bound the header states for ncols 3..8).
Nothing here is shared with the CUDA sources.
"""
from fractions import Fraction

import numpy as np
import torch

F32 = np.float32
N_PIECES = 5


def _e4m3_grid():
    """All non-negative finite e4m3 values with their mantissa bit 0 (for ties)."""
    out = []
    for m in range(8):  # subnormals, exponent field 0: m/8 * 2^-6
        out.append((Fraction(m, 8) * Fraction(1, 64), m & 1))
    for E in range(1, 16):
        for m in range(8):
            if E == 15 and m == 7:  # the NaN encoding of e4m3fn
                continue
            out.append(((1 + Fraction(m, 8)) * Fraction(2) ** (E - 7), m & 1))
    return out


_GRID = _e4m3_grid()
E4M3_MAX = 448.0


def e4m3_rne_sat(v: float) -> float:
    """Round to the nearest e4m3 value, ties to an even mantissa; saturate to
    +-448 beyond the largest finite value."""
    a = Fraction(abs(v))
    if a >= Fraction(E4M3_MAX):
        return float(np.copysign(E4M3_MAX, v))
    best = None
    for mag, mbit in _GRID:
        d = abs(a - mag)
        if best is None or d < best[0] or (d == best[0] and mbit == 0 and best[2] == 1):
            best = (d, mag, mbit)
    return float(np.copysign(float(best[1]), v))


def e4m3_fast(v: float) -> float:
    """The same rounding by scaling to the value's quantum (2^(E - 3) in the
    binade 2^E, 2^-9 below 2^-6) and rounding half to even (np.rint): every
    step is exact in float64 for an f32 input."""
    a = abs(float(v))
    if a >= E4M3_MAX:
        return float(np.copysign(E4M3_MAX, v))
    quantum = 2.0 ** -9 if a < 2.0 ** -6 else 2.0 ** (int(np.frexp(a)[1]) - 1 - 3)
    r = float(np.rint(a / quantum)) * quantum
    return float(np.copysign(min(r, E4M3_MAX), v))


def split_pieces(v, n: int = N_PIECES):
    """Pieces of an f32 v with every step in f32; also the piece inputs and
    whether each subtraction was exact."""
    r = F32(v)
    pieces, inputs, exact = [], [], True
    for i in range(n):
        s = F32(r * F32(16.0 ** i))
        inputs.append(float(s))
        p = e4m3_fast(float(s))
        pieces.append(p)
        step = F32(F32(p) * F32(16.0 ** -i))
        nr = F32(r - step)
        exact &= Fraction(float(nr)) == Fraction(float(r)) - Fraction(float(step))
        r = nr
    return pieces, inputs, float(r), exact


def block_scale(x):
    m = float(np.max(np.abs(x)))
    return 0 if m == 0.0 else int(np.frexp(np.float32(m))[1])


def test_e4m3_grid_is_the_format():
    mags = sorted(float(m) for m, _ in _GRID)
    assert len(mags) == 127 and mags[0] == 0.0 and mags[-1] == 448.0
    assert mags[1] == 2.0 ** -9                     # smallest subnormal
    assert 2.0 ** -6 in mags and 1.75 * 2.0 ** 8 in mags


def test_e4m3_rounding_matches_torch_float8():
    """The restated rounding equals PyTorch's float8_e4m3fn cast on every
    in-range input tried: grid points, midpoints (ties), and random values."""
    g = np.random.default_rng(11)
    mags = sorted(float(m) for m, _ in _GRID)
    vals = list(mags) + [0.5 * (a + b) for a, b in zip(mags[:-1], mags[1:])]
    vals += list(g.uniform(-448.0, 448.0, 3000))
    vals += list(g.uniform(-1.0, 1.0, 2000) * 2.0 ** g.integers(-14, 9, 2000))
    vals = [float(F32(v)) for v in vals if abs(v) <= 448.0]
    vals += [-v for v in vals]
    got = [e4m3_rne_sat(v) for v in vals]
    ref = torch.tensor(vals, dtype=torch.float32).to(torch.float8_e4m3fn).to(torch.float32)
    assert np.array_equal(np.array(got, dtype=np.float32), ref.numpy())


def test_fast_rounding_equals_the_definition():
    g = np.random.default_rng(12)
    mags = sorted(float(m) for m, _ in _GRID)
    vals = list(mags) + [0.5 * (a + b) for a, b in zip(mags[:-1], mags[1:])]
    vals += list(g.uniform(-500.0, 500.0, 1500))
    vals += list(g.uniform(-1.0, 1.0, 1500) * 2.0 ** g.integers(-30, 9, 1500))
    vals += [464.0, 463.99, 480.0, 1e10, 2.0 ** -10, 2.0 ** -6 - 2.0 ** -12]
    for v in vals:
        v = float(F32(v))
        assert e4m3_fast(v) == e4m3_rne_sat(v), v
        assert e4m3_fast(-v) == e4m3_rne_sat(-v), v


def test_e4m3_ties_and_saturation():
    assert e4m3_rne_sat(1.0625) == 1.0        # tie between 1 and 1.125 -> even (1)
    assert e4m3_rne_sat(1.1875) == 1.25       # tie between 1.125 and 1.25 -> even (1.25)
    assert e4m3_rne_sat(2.0 ** -10) == 0.0    # tie between 0 and 2^-9 -> even (0)
    assert e4m3_rne_sat(3 * 2.0 ** -10) == 2.0 ** -8   # tie 2^-9 / 2^-8 -> even (2^-8)
    assert e4m3_rne_sat(1000.0) == 448.0 and e4m3_rne_sat(-1e30) == -448.0


def _check_split(v):
    v = float(F32(v))
    pieces, inputs, r, exact = split_pieces(v)
    assert exact, v
    assert all(abs(s) <= E4M3_MAX for s in inputs), (v, inputs)
    assert Fraction(v) == sum(Fraction(p) * Fraction(16) ** -i for i, p in enumerate(pieces)) \
        + Fraction(r)
    assert abs(Fraction(r)) <= Fraction(2) ** -20 * abs(Fraction(v)) + Fraction(2) ** -26, (v, r)


def test_piece_split_exact_and_bounded():
    g = np.random.default_rng(5)
    vals = list(g.uniform(-256.0, 256.0, 3000))
    vals += list(g.uniform(-1.0, 1.0, 2000) * 2.0 ** g.integers(-60, 8, 2000))
    # boundaries: the largest magnitudes, grid points and ties of the first
    # piece, values at the subnormal steps of the last pieces, zero
    vals += [255.99998474121094, -255.99998474121094, 128.0, 136.0, 132.0, 140.0, 248.0, 252.0,
             2.0 ** -9, 3 * 2.0 ** -10, 2.0 ** -25, 3 * 2.0 ** -27, 2.0 ** -26, 0.0, 1e-30]
    for v in vals:
        _check_split(v)


def test_block_scaling_bound_on_wide_range_blocks():
    """Whole blocks as the prep scales them: the maximum lands in [128, 256) and
    every element x is held to 2^-20 |x| + 2^-33 M_b."""
    g = np.random.default_rng(9)
    for t in range(300):
        x = (g.standard_normal(64) * 10.0 ** g.uniform(-6, 4, 64)).astype(F32)
        if t % 3 == 0:
            x[g.integers(0, 64)] = F32(3000.0)
        e = block_scale(x)
        mb = Fraction(float(np.max(np.abs(x))))
        sc = Fraction(2) ** (8 - e)
        v = [float(F32(Fraction(float(xi)) * sc)) for xi in x]  # exact power-of-two scaling
        assert 128 <= max(abs(Fraction(a)) for a in v) < 256
        for xi, vi in zip(x, v):
            pieces, _, r, exact = split_pieces(vi)
            assert exact
            held = sum(Fraction(p) * Fraction(16) ** -i for i, p in enumerate(pieces)) / sc
            err = abs(held - Fraction(float(xi)))
            assert err <= Fraction(2) ** -20 * abs(Fraction(float(xi))) + Fraction(2) ** -33 * mb
