"""Pins of the CPU oracle against what the Q2_0 pages and the mathematics fix.

Each test checks the oracle against something other than itself: a library
routine (numpy's float16 conversion, numpy's fp64 matmul), exact rational
arithmetic, hand-worked blocks (tests/golden/decode_blocks.txt), sizes printed
on the pages, closed forms and invariants.
"""
import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# fp16 codec (IEEE 754 binary16) vs numpy
# ---------------------------------------------------------------------------
def test_half_to_double_exhaustive(oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.halves_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros and infinities keep their sign
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _f32_from_bits(b):
    return np.asarray(b, dtype=np.uint32).view(np.float32)


def test_float_to_half_ties_and_boundaries(oracle_mod):
    h = np.arange(0, 0x7C00, dtype=np.uint16)          # all finite non-negative halves
    lo = h.view(np.float16).astype(np.float64)
    nxt = (h + 1).view(np.float16).astype(np.float64)  # 0x7c00 -> inf for the last one
    mid = (lo + nxt) / 2.0
    mid = mid[np.isfinite(mid)].astype(np.float32)      # exact in f32 (11 vs 24 bits)
    cands = [mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(0)),
             lo.astype(np.float32), np.float32([65504, 65519.996, 65520, 65536, 1e30, 2.0**-25,
                                                 2.0**-24, 3 * 2.0**-26, 2.0**-26, 1e-30])]
    v = np.concatenate(cands).astype(np.float32)
    v = np.concatenate([v, -v])
    got = oracle_mod.floats_to_half_rn(v)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


def test_float_to_half_random(oracle_mod):
    g = np.random.default_rng(7)
    bits = g.integers(0, 2**32, size=2_000_000, dtype=np.uint64).astype(np.uint32)
    v = _f32_from_bits(bits)
    v = v[np.isfinite(v)]
    w = g.standard_normal(1_000_000).astype(np.float32) * np.float32(2.0) ** g.integers(
        -30, 18, size=1_000_000).astype(np.float32)
    v = np.concatenate([v, w])
    got = oracle_mod.floats_to_half_rn(v)
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------------------
# Block decode vs hand-worked blocks
# ---------------------------------------------------------------------------
def _golden_blocks():
    out = []
    with open(os.path.join(GOLDEN, "decode_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            dhex, qhex, exp = [t.strip() for t in line.split("|")]
            d = int(dhex, 16)
            blk = bytes([d & 0xFF, d >> 8]) + bytes.fromhex(qhex)
            toks = exp.split()
            vals = [None] * 64
            if toks[0] == "fill":
                vals = [float(toks[1])] * 64
                for t in toks[2:]:
                    e, v = t.split(":")
                    vals[int(e)] = float(v)
            elif toks[0] == "cycle":
                cyc = [float(t) for t in toks[1:5]]
                vals = [cyc[e % 4] for e in range(64)]
            else:
                raise ValueError(line)
            out.append((blk, np.array(vals, dtype=np.float64)))
    return out


def test_decode_golden_blocks(oracle_mod):
    cases = _golden_blocks()
    assert len(cases) >= 15
    for blk, exp in cases:
        got = oracle_mod.decode_block(np.frombuffer(blk, dtype=np.uint8))
        assert np.array_equal(got, exp), (blk.hex(), got, exp)
        assert np.array_equal(np.signbit(got), np.signbit(exp)), blk.hex()


def test_code_table(oracle_mod):
    """Codes 0, 1, 2, 3 decode to -d, 0, +d, +2d for d = 0.75 (one byte pattern each)."""
    d = 0x3A00  # 0.75
    for q, level in [(0, -0.75), (1, 0.0), (2, 0.75), (3, 1.5)]:
        byte = q | (q << 2) | (q << 4) | (q << 6)
        blk = np.array([d & 0xFF, d >> 8] + [byte] * 16, dtype=np.uint8)
        assert np.all(oracle_mod.decode_block(blk) == level)
        assert np.all(oracle_mod.block_codes(blk) == q)


def test_dequantize_row_major_layout(oracle_mod):
    """Block (n, b) of an N x K matrix sits at byte offset (n*K/64 + b)*18."""
    g = np.random.default_rng(3)
    N, K = 5, 192
    w = synth.packed_matrix(g, N, K, 0.1, 1.0, 0.05)
    W = oracle_mod.dequantize(w, N, K)
    nb = K // 64
    for n in range(N):
        for b in range(nb):
            off = (n * nb + b) * 18
            assert np.array_equal(W[n, 64 * b:64 * b + 64], oracle_mod.decode_block(w[off:off + 18]))


# ---------------------------------------------------------------------------
# Sizes printed on the pages
# ---------------------------------------------------------------------------
def test_size_pins(oracle_mod):
    # "Osmnáct bajtů na čtyřiašedesát vah": 18 bytes per 64 weights = 2.25 bits/weight
    assert oracle_mod.lib().qo_bytes_per_block() == 18
    assert oracle_mod.lib().qo_weights_per_block() == 64
    assert oracle_mod.packed_bytes(1, 64) * 8 / 64 == 2.25
    # "Šest procent…": group 128 -> 34 bytes = 2.125 bits/weight; difference 5.9 %
    assert oracle_mod.packed_bytes(1, 128, 128) == 34
    assert oracle_mod.packed_bytes(1, 128, 128) * 8 / 128 == 2.125
    ratio = oracle_mod.packed_bytes(1, 128) / oracle_mod.packed_bytes(1, 128, 128)
    assert round((ratio - 1) * 100, 1) == 5.9
    # "Sedmkrát menší soubor" / "Šest procent…": the 8B model is 2.15 GiB at group 64,
    # 2.03 GiB at group 128 and 15.26 GiB in F16. Weights of the 8B-class shapes:
    # 36 layers x (q, k, v, o, gate, up, down) + 151936 x 4096 head + the same-sized
    # input embedding.
    mats = [(m.N, m.K) for _, m in synth.decode_step_8b(with_head=True)] + [(151936, 4096)]
    n_weights = sum(n * k for n, k in mats)
    gib = 2.0 ** 30
    g64 = sum(oracle_mod.packed_bytes(n, k) for n, k in mats) / gib
    g128 = sum(oracle_mod.packed_bytes(n, k, 128) for n, k in mats) / gib
    f16 = 2 * n_weights / gib
    assert round(g64, 2) == 2.15
    assert round(g128, 2) == 2.03
    assert round(f16, 2) == 15.26
    assert round(f16 / g64, 1) == 7.1


# ---------------------------------------------------------------------------
# Dequantize-then-dot
# ---------------------------------------------------------------------------
def _exact_dot(Wrow, xcol):
    return sum((Fraction(float(a)) * Fraction(float(b)) for a, b in zip(Wrow, xcol)), Fraction(0))


@pytest.mark.parametrize("N,K,ncols", [(1, 64, 1), (3, 128, 2), (4, 256, 3), (2, 192, 1)])
def test_matmul_exact_rational(oracle_mod, N, K, ncols):
    g = np.random.default_rng(N * 100 + K + ncols)
    w = synth.packed_matrix(g, N, K, 0.01, 3.0, 0.05)
    x = synth.activations(g, ncols, K, 0.05, 30.0)
    y, acc = oracle_mod.matmul(w, N, K, x)
    W = oracle_mod.dequantize(w, N, K)
    for c in range(ncols):
        for n in range(N):
            ex = _exact_dot(W[n], x[c])
            exa = sum((abs(Fraction(float(a)) * Fraction(float(b))) for a, b in zip(W[n], x[c])),
                      Fraction(0))
            bound = K * 2.0 ** -52 * float(exa)
            assert abs(Fraction(y[c, n]) - ex) <= Fraction(bound), (c, n)
            assert abs(Fraction(acc[c, n]) - exa) <= Fraction(bound), (c, n)


def test_matmul_vs_numpy(oracle_mod):
    g = np.random.default_rng(11)
    N, K, C = 37, 640, 5
    w = synth.packed_matrix(g, N, K, 0.005, 0.05, 0.01)
    x = synth.activations(g, C, K)
    y, acc = oracle_mod.matmul(w, N, K, x)
    W = oracle_mod.dequantize(w, N, K)
    ref = x.astype(np.float64) @ W.T
    refa = np.abs(x.astype(np.float64)) @ np.abs(W.T)
    assert np.allclose(y, ref, rtol=0, atol=1e-12 * refa.max())
    assert np.allclose(acc, refa, rtol=1e-13, atol=0)
    # a listed subset of rows gives the same numbers
    rows = np.array([36, 0, 17, 17])
    ys, accs = oracle_mod.matmul(w, N, K, x, rows=rows)
    assert np.array_equal(ys, y[:, rows]) and np.array_equal(accs, acc[:, rows])


def _const_code_matrix(N, K, q, dbits):
    byte = q | (q << 2) | (q << 4) | (q << 6)
    nb = N * (K // 64)
    blk = np.array([dbits & 0xFF, dbits >> 8] + [byte] * 16, dtype=np.uint8)
    return np.tile(blk, nb)


def test_matmul_closed_forms(oracle_mod):
    g = np.random.default_rng(5)
    N, K = 3, 512
    x = synth.activations(g, 2, K)
    sx = np.array([math.fsum(map(float, x[c])) for c in range(2)])
    sax = np.array([math.fsum(abs(float(v)) for v in x[c]) for c in range(2)])
    bound = K * 2.0 ** -52 * sax
    # all codes 1 -> every weight is 0 -> y = 0 exactly
    y, acc = oracle_mod.matmul(_const_code_matrix(N, K, 1, 0x3C00), N, K, x)
    assert np.all(y == 0) and np.all(acc == 0)
    # all codes 2 with d = 1 -> y = sum(x); all codes 0 -> y = -sum(x)
    y, acc = oracle_mod.matmul(_const_code_matrix(N, K, 2, 0x3C00), N, K, x)
    assert np.all(np.abs(y - sx[:, None]) <= bound[:, None])
    y, acc = oracle_mod.matmul(_const_code_matrix(N, K, 0, 0x3C00), N, K, x)
    assert np.all(np.abs(y + sx[:, None]) <= bound[:, None])
    # all codes 3 with d = 0.5 -> y = sum(x)
    y, acc = oracle_mod.matmul(_const_code_matrix(N, K, 3, 0x3800), N, K, x)
    assert np.all(np.abs(y - sx[:, None]) <= bound[:, None])
    # one weight non-zero -> y = (q-1) * d * x_e exactly
    w = _const_code_matrix(1, K, 1, 0x3C00)
    e = 200                       # block 3, element 8 -> word 0, bits 16-17 -> byte 2 of the codes
    w[3 * 18 + 2 + 2] = 0x56      # that byte's lowest field = 2 -> +1 * d
    w[3 * 18 + 0], w[3 * 18 + 1] = 0x00, 0xC2   # d = -3.0
    y, _ = oracle_mod.matmul(w, 1, K, x)
    assert np.array_equal(y[:, 0], -3.0 * x[:, e].astype(np.float64))


# ---------------------------------------------------------------------------
# get_rows
# ---------------------------------------------------------------------------
def test_get_rows_matches_decode(oracle_mod):
    g = np.random.default_rng(9)
    n_rows, K = 20, 256
    t = synth.packed_matrix(g, n_rows, K, 0.005, 0.05, 0.01)
    edges = synth.edge_blocks()
    t[:edges.size] = edges.reshape(-1)          # first rows hold the edge blocks
    ids = np.array([0, 1, 2, 19, 0, 7, 3], dtype=np.int32)
    out, bad = oracle_mod.get_rows(t, n_rows, K, ids)
    assert bad == 0 and out.dtype == np.float32
    W = oracle_mod.dequantize(t, n_rows, K)
    for r, i in enumerate(ids):
        ref = W[i].astype(np.float32)
        assert np.array_equal(out[r].view(np.uint32), ref.view(np.uint32))
        # row-sum invariant: sum of a row = sum_b d_b * sum_i (q - 1), exact in fp64
        s = 0.0
        for b in range(K // 64):
            blk = t[(i * (K // 64) + b) * 18:(i * (K // 64) + b) * 18 + 18]
            s += oracle_mod.half_to_double(int(blk[0]) | (int(blk[1]) << 8)) * float(
                np.sum(oracle_mod.block_codes(blk).astype(np.int64) - 1))
        assert math.isclose(float(np.sum(out[r].astype(np.float64))), s, rel_tol=0, abs_tol=0) or \
            np.isnan(s)
    # signed zeros survive: block 5 (all code 0, d=+0) -> all -0
    z = out[0, 64 * 5:64 * 6]
    assert np.all(z == 0) and np.all(np.signbit(z))


def test_get_rows_bad_ids(oracle_mod):
    g = np.random.default_rng(10)
    t = synth.packed_matrix(g, 4, 64, 0.1, 0.2)
    out, bad = oracle_mod.get_rows(t, 4, 64, np.array([0, 4, -1, 3], dtype=np.int32))
    assert bad == 2
    assert np.all(out[1] == 0) and np.all(out[2] == 0)


# ---------------------------------------------------------------------------
# Reference quantizer
# ---------------------------------------------------------------------------
def _nearest_level_codes(wblock):
    """Brute force from the pages' rule: scale = max |w|; each weight goes to the
    nearest of the levels (q-1)*scale, q = 0..3; exact rationals; ties away from 0."""
    amax = max(abs(Fraction(float(v))) for v in wblock)
    codes = []
    for v in wblock:
        fv = Fraction(float(v))
        if amax == 0:
            codes.append(1)
            continue
        dist = [(abs(fv - (q - 1) * amax), q) for q in range(4)]
        best = min(dd for dd, _ in dist)
        cands = [q for dd, q in dist if dd == best]
        # ties: pick the level farther from zero
        codes.append(max(cands, key=lambda q: abs(q - 1)))
    return codes


def test_quantizer_nearest_level_brute_force(oracle_mod):
    g = np.random.default_rng(21)
    blocks = [g.standard_normal(64).astype(np.float32) for _ in range(200)]
    # explicit ties and near-ties at +-amax/2
    b = g.uniform(-1, 1, 64).astype(np.float32)
    b[0] = 2.0
    b[1], b[2] = 1.0, -1.0
    b[3], b[4] = np.nextafter(np.float32(1.0), np.float32(0)), np.nextafter(np.float32(-1.0), np.float32(0))
    blocks.append(b)
    blocks.append(np.zeros(64, dtype=np.float32))
    blocks.append(np.full(64, -0.25, dtype=np.float32))
    for blk in blocks:
        q = oracle_mod.quantize(blk, 1, 64)
        amax = float(np.max(np.abs(blk)))
        assert oracle_mod.block_scale_bits(q) == int(np.float16(amax).view(np.uint16))
        assert list(oracle_mod.block_codes(q)) == _nearest_level_codes(blk)
    # spot values of the tie block
    q = oracle_mod.block_codes(oracle_mod.quantize(blocks[200], 1, 64))
    assert list(q[:5]) == [2, 2, 0, 1, 1]


def test_quantizer_round_trip(oracle_mod):
    """Q(DQ(B)) == B for blocks with codes in {0,1,2}, some code != 1, d > 0 normal."""
    g = np.random.default_rng(22)
    n = 14000
    w = synth.packed_matrix(g, n, 64, 0.001, 100.0)
    blocks = w.reshape(n, 18)
    keep = np.array([np.any(oracle_mod.block_codes(b) != 1) for b in blocks[:2000]])
    blocks = blocks[:2000][keep]
    W = oracle_mod.dequantize(blocks.reshape(-1), blocks.shape[0], 64).astype(np.float32)
    q = oracle_mod.quantize(W, blocks.shape[0], 64)
    assert np.array_equal(q, blocks.reshape(-1))


def test_quantizer_idempotent_and_edges(oracle_mod):
    g = np.random.default_rng(23)
    src = (g.standard_normal((64, 256)) * 3).astype(np.float32)
    q1 = oracle_mod.quantize(src, 64, 256)
    q2 = oracle_mod.quantize(oracle_mod.dequantize(q1, 64, 256).astype(np.float32), 64, 256)
    assert np.array_equal(q1, q2)
    # all-zero block: d = 0, every code 1
    z = oracle_mod.quantize(np.zeros(64, np.float32), 1, 64)
    assert oracle_mod.block_scale_bits(z) == 0 and np.all(oracle_mod.block_codes(z) == 1)
    # code 3 is never produced
    assert not np.any(np.stack([oracle_mod.block_codes(q1[i:i + 18])
                                for i in range(0, q1.size, 18)]) == 3)
    # scale rounding: amax = 1 + 2^-11 is a tie between 1 and 1 + 2^-10 -> even (1.0)
    blk = np.zeros(64, np.float32)
    blk[7] = np.float32(1 + 2.0 ** -11)
    assert oracle_mod.block_scale_bits(oracle_mod.quantize(blk, 1, 64)) == 0x3C00


# ---------------------------------------------------------------------------
# Group-128 blocks (34 bytes per 128 weights)
# ---------------------------------------------------------------------------
def _golden_blocks_g128():
    out = []
    with open(os.path.join(GOLDEN, "decode_blocks_g128.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            dhex, qhex, exp = [t.strip() for t in line.split("|")]
            d = int(dhex, 16)
            blk = bytes([d & 0xFF, d >> 8]) + bytes.fromhex(qhex)
            assert len(blk) == 34
            toks = exp.split()
            if toks[0] == "fill":
                vals = [float(toks[1])] * 128
                for t in toks[2:]:
                    e, v = t.split(":")
                    vals[int(e)] = float(v)
            elif toks[0] == "cycle":
                cyc = [float(t) for t in toks[1:5]]
                vals = [cyc[e % 4] for e in range(128)]
            else:
                raise ValueError(line)
            out.append((blk, np.array(vals, dtype=np.float64)))
    return out


def test_decode_golden_blocks_g128(oracle_mod):
    cases = _golden_blocks_g128()
    assert len(cases) >= 8
    for blk, exp in cases:
        got = oracle_mod.decode_block_g128(np.frombuffer(blk, dtype=np.uint8))
        assert np.array_equal(got, exp), (blk.hex(), got, exp)
        assert np.array_equal(np.signbit(got), np.signbit(exp)), blk.hex()


def _g128_matrix(g, N, K):
    """Random group-128 matrix bytes: fp16 scales in [0.01, 3), codes 0..3."""
    nb = K // 128
    d = g.uniform(0.01, 3.0, size=(N, nb)).astype(np.float16).view(np.uint16)
    blk = np.zeros((N, nb, 34), dtype=np.uint8)
    blk[:, :, 0] = d & 0xFF
    blk[:, :, 1] = d >> 8
    blk[:, :, 2:] = g.integers(0, 256, size=(N, nb, 32), dtype=np.uint8)
    return blk.reshape(-1)


def test_g128_halves_decode_as_group64_blocks(oracle_mod):
    """Each half of a group-128 block reads like a group-64 block with the same scale
    (the word rule runs over words 0-3 and 4-7): decode both ways."""
    g = np.random.default_rng(128)
    for _ in range(200):
        b = _g128_matrix(g, 1, 128)
        got = oracle_mod.decode_block_g128(b)
        lo = np.concatenate([b[:2], b[2:18]])
        hi = np.concatenate([b[:2], b[18:34]])
        ref = np.concatenate([oracle_mod.decode_block(lo), oracle_mod.decode_block(hi)])
        assert np.array_equal(got, ref)


@pytest.mark.parametrize("N,K,ncols", [(1, 128, 1), (3, 256, 2), (2, 384, 3)])
def test_matmul_g128_exact_rational(oracle_mod, N, K, ncols):
    g = np.random.default_rng(N * 1000 + K + ncols)
    w = _g128_matrix(g, N, K)
    x = synth.activations(g, ncols, K, 0.05, 30.0)
    y, acc = oracle_mod.matmul_g128(w, N, K, x)
    for c in range(ncols):
        for n in range(N):
            row = np.concatenate([oracle_mod.decode_block_g128(w[(n * (K // 128) + b) * 34:
                                                                 (n * (K // 128) + b + 1) * 34])
                                  for b in range(K // 128)])
            ex = _exact_dot(row, x[c])
            exa = sum((abs(Fraction(float(a)) * Fraction(float(v))) for a, v in zip(row, x[c])),
                      Fraction(0))
            bound = K * 2.0 ** -52 * float(exa)
            assert abs(Fraction(y[c, n]) - ex) <= Fraction(bound)
            assert abs(Fraction(acc[c, n]) - exa) <= Fraction(bound)


def test_g128_closed_forms_and_get_rows(oracle_mod):
    N, K = 3, 256
    d = np.float16(0.75).view(np.uint16)
    for q, level in [(0, -0.75), (1, 0.0), (2, 0.75), (3, 1.5)]:
        byte = q | (q << 2) | (q << 4) | (q << 6)
        blk = np.array([d & 0xFF, d >> 8] + [byte] * 32, dtype=np.uint8)
        w = np.tile(blk, N * (K // 128))
        x = np.random.default_rng(q).standard_normal((2, K)).astype(np.float32)
        y, _ = oracle_mod.matmul_g128(w, N, K, x)
        ref = level * x.astype(np.float64).sum(axis=1)
        assert np.allclose(y, ref[:, None], rtol=1e-14, atol=1e-14)
        out, bad = oracle_mod.get_rows_g128(w, N, K, np.array([2, 0, 5], dtype=np.int32))
        assert bad == 1
        assert np.all(out[:2] == np.float32(level)) and np.all(out[2] == 0)


# ---------------------------------------------------------------------------
# Expert mat-vec (mul_mat_id): each slot is the plain matmul of the selected
# expert ([WGPU] limitations paragraph names MUL_MAT_ID as the missing op)
# ---------------------------------------------------------------------------
def _experts(g, n_expert, N, K):
    return np.concatenate([synth.packed_matrix(g, N, K, 0.01, 3.0, 0.05) for _ in range(n_expert)])


def test_matmul_id_exact_rational(oracle_mod):
    g = np.random.default_rng(71)
    n_expert, N, K, n_tokens, n_used = 3, 2, 128, 2, 2
    w = _experts(g, n_expert, N, K)
    x = synth.activations(g, n_tokens * n_used, K, 0.05, 30.0).reshape(n_tokens, n_used, K)
    ids = np.array([[2, 0], [1, 2]], dtype=np.int32)
    y, acc, bad = oracle_mod.matmul_id(w, n_expert, N, K, x, ids)
    assert bad == 0
    eb = N * (K // 64) * 18
    for t in range(n_tokens):
        for i in range(n_used):
            W = oracle_mod.dequantize(w[ids[t, i] * eb:(ids[t, i] + 1) * eb], N, K)
            for n in range(N):
                ex = _exact_dot(W[n], x[t, i])
                exa = sum((abs(Fraction(float(a)) * Fraction(float(b))) for a, b in zip(W[n], x[t, i])),
                          Fraction(0))
                bound = K * 2.0 ** -52 * float(exa)
                assert abs(Fraction(y[t, i, n]) - ex) <= Fraction(bound), (t, i, n)
                assert abs(Fraction(acc[t, i, n]) - exa) <= Fraction(bound), (t, i, n)


def test_matmul_id_single_expert_is_matmul(oracle_mod):
    """One expert and every id 0: each slot equals the (pinned) plain matmul."""
    g = np.random.default_rng(72)
    N, K, n_tokens, n_used = 5, 256, 3, 2
    w = synth.packed_matrix(g, N, K, 0.005, 0.05, 0.01)
    x = synth.activations(g, n_tokens * n_used, K).reshape(n_tokens, n_used, K)
    y, acc, bad = oracle_mod.matmul_id(w, 1, N, K, x, np.zeros((n_tokens, n_used), np.int32))
    assert bad == 0
    ref, refa = oracle_mod.matmul(w, N, K, x.reshape(-1, K))
    assert np.array_equal(y.reshape(-1, N), ref) and np.array_equal(acc.reshape(-1, N), refa)


def test_matmul_id_expert_permutation_and_broadcast(oracle_mod):
    """Relabelling the experts (with the ids relabelled alike) changes nothing;
    one shared vector per token equals that vector repeated per slot; listed
    rows give the same numbers."""
    g = np.random.default_rng(73)
    n_expert, N, K, n_tokens, n_used = 6, 7, 192, 4, 3
    w = _experts(g, n_expert, N, K)
    eb = N * (K // 64) * 18
    x1 = synth.activations(g, n_tokens, K).reshape(n_tokens, 1, K)
    ids = g.integers(0, n_expert, size=(n_tokens, n_used)).astype(np.int32)
    y, acc, _ = oracle_mod.matmul_id(w, n_expert, N, K, x1, ids)
    perm = g.permutation(n_expert)            # new slot of expert e is perm[e]
    wp = np.empty_like(w)
    for e in range(n_expert):
        wp[perm[e] * eb:(perm[e] + 1) * eb] = w[e * eb:(e + 1) * eb]
    yp, accp, _ = oracle_mod.matmul_id(wp, n_expert, N, K, x1, perm[ids].astype(np.int32))
    assert np.array_equal(y, yp) and np.array_equal(acc, accp)
    xr = np.repeat(x1, n_used, axis=1)
    yr, accr, _ = oracle_mod.matmul_id(w, n_expert, N, K, xr, ids)
    assert np.array_equal(y, yr) and np.array_equal(acc, accr)
    rows = np.array([6, 0, 3])
    ys, _, _ = oracle_mod.matmul_id(w, n_expert, N, K, x1, ids, rows=rows)
    assert np.array_equal(ys, y[:, :, rows])


def test_matmul_id_bad_ids(oracle_mod):
    g = np.random.default_rng(74)
    n_expert, N, K = 2, 3, 64
    w = _experts(g, n_expert, N, K)
    x = synth.activations(g, 2, K).reshape(2, 1, K)
    ids = np.array([[0, 2], [-1, 1]], dtype=np.int32)
    y, acc, bad = oracle_mod.matmul_id(w, n_expert, N, K, x, ids)
    assert bad == 2
    assert np.isnan(y[0, 1]).all() and np.isnan(y[1, 0]).all()
    assert not np.isnan(y[0, 0]).any() and not np.isnan(y[1, 1]).any()


# ---------------------------------------------------------------------------
# Split layout (scales and codes in separate arrays; [KOPI] "Why the weight has
# to stay quantized" splits a block format's scales from its quants)
# ---------------------------------------------------------------------------
def test_soa_hand_built(oracle_mod):
    """Two blocks with every byte distinct, laid out by hand."""
    blk0 = np.arange(1, 19, dtype=np.uint8)            # d = 0x0201, codes 3..18
    blk1 = np.arange(101, 119, dtype=np.uint8)         # d = 0x6665, codes 103..118
    soa = oracle_mod.raw_to_soa(np.concatenate([blk0, blk1]), 1, 128)
    expect = np.zeros(512, dtype=np.uint8)
    expect[0:16] = np.arange(3, 19)
    expect[16:32] = np.arange(103, 119)
    expect[256:260] = [1, 2, 101, 102]
    assert oracle_mod.soa_bytes(1, 128) == 512
    assert np.array_equal(soa, expect)


def test_soa_round_trip_and_sizes(oracle_mod):
    g = np.random.default_rng(81)
    for N, K in [(1, 64), (7, 192), (33, 512), (300, 1024)]:
        w = synth.packed_matrix(g, N, K, 0.005, 0.05, 0.01)
        soa = oracle_mod.raw_to_soa(w, N, K)
        nblk = N * (K // 64)
        assert soa.size == -(-16 * nblk // 256) * 256 + -(-2 * nblk // 256) * 256
        assert np.array_equal(oracle_mod.soa_to_raw(soa, N, K), w)
        x = synth.activations(g, 2, K)
        assert np.array_equal(oracle_mod.matmul_soa(soa, N, K, x)[0], oracle_mod.matmul(w, N, K, x)[0])


def test_soa_element_decode(oracle_mod):
    """Element e of block (n, b) read from the split arrays (code byte e // 4,
    field e % 4; scale from d[]) equals the pinned block decode."""
    g = np.random.default_rng(82)
    N, K = 5, 256
    nb = K // 64
    w = synth.packed_matrix(g, N, K, 0.01, 3.0, 0.1)
    soa = oracle_mod.raw_to_soa(w, N, K)
    d_off = -(-16 * N * nb // 256) * 256
    for n in range(N):
        for b in range(nb):
            i = n * nb + b
            ref = oracle_mod.decode_block(w[18 * i:18 * i + 18])
            d = oracle_mod.half_to_double(int(soa[d_off + 2 * i]) | (int(soa[d_off + 2 * i + 1]) << 8))
            for e in range(64):
                q = (int(soa[16 * i + e // 4]) >> (2 * (e % 4))) & 3
                assert (q - 1) * d == ref[e]
