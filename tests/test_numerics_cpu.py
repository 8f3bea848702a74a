"""CPU checks of the exactness arguments behind the fp4 decode path.

The fp4 mat-vec multiplies the codes, read as e2m1 values q/2, by 12 e2m1
pieces of v = 2u (u = x * 2^s, max|u| in [1, 2)): p_i = e2m1(r_i * 4^i),
r_0 = v, r_{i+1} = r_i - p_i * 4^-i. These tests restate e2m1 round-to-nearest-
even from the format's definition (sign, 2 exponent bits with bias 1, 1
mantissa bit; 0.5 is the one subnormal step) and check, on random and boundary
values:
  - every scaled residual after the first piece lies in [-2, 2], so no piece
    saturates;
  - after 12 pieces |v - sum p_i 4^-i| <= 2^-24;
  - a block's per-piece sum of (q/2) * p_i over 64 weights is exact in f32
    (the tensor core accumulates in f32), so the only rounding is the piece
    split itself.
Nothing here is shared with the CUDA sources.
"""
import numpy as np
import pytest

# e2m1 magnitudes with their mantissa bit (for ties to even)
_E2M1 = [(0.0, 0), (0.5, 1), (1.0, 0), (1.5, 1), (2.0, 0), (3.0, 1), (4.0, 0), (6.0, 1)]


def e2m1_rne(v: float) -> float:
    a = abs(v)
    best = None
    for mag, mbit in _E2M1:
        d = abs(a - mag)
        if best is None or d < best[0] or (d == best[0] and mbit == 0 and best[2] == 1):
            best = (d, mag, mbit)
    return float(np.copysign(best[1], v))


def split_pieces(v: float, n: int = 12):
    r, pieces, scaled = v, [], []
    for i in range(n):
        s = r * 4.0 ** i
        scaled.append(s)
        p = e2m1_rne(s)
        pieces.append(p)
        r = r - p * 4.0 ** -i
    return pieces, scaled, r


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
    vals = list(g.uniform(-4.0, 4.0, 20000))
    # boundaries: the largest magnitudes, grid points, ties, tiny values
    vals += [3.999999761581421, -3.999999761581421, 2.0, -2.0, 1.0, 0.25, 0.75, 2.5, 3.5,
             1e-8, -1e-8, 0.0]
    for v in vals:
        v = float(np.float32(v))
        pieces, scaled, r = split_pieces(v)
        assert all(abs(s) <= 2.0 for s in scaled[1:]), v
        assert abs(r) <= 2.0 ** -24, (v, r)


def test_block_sums_exact_in_f32():
    """sum over 64 weights of (q/2) * p_i is an exact f32 value for each piece i:
    the products are multiples of 2^-2 (pieces are multiples of 0.5, q/2 of
    0.5) bounded by 1.5 * 6, and 64 of them stay below 2^24 quarter units."""
    g = np.random.default_rng(2)
    for _ in range(200):
        q = g.integers(0, 4, 64)
        v = g.uniform(-4.0, 4.0, 64).astype(np.float32)
        for i in range(12):
            p = np.array([split_pieces(float(x))[0][i] for x in v])
            exact = sum((qq / 2.0) * pp for qq, pp in zip(q, p))
            f32 = np.float32(0.0)
            for qq, pp in zip(q, p):
                f32 = np.float32(f32 + np.float32(qq / 2.0) * np.float32(pp))
            assert float(f32) == exact
