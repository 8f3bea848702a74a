"""Activation vectors with a wide dynamic range, and weight patterns that put
zero weights (code 1) under their largest elements: inputs for the parity
tests of the mat-vec and GEMM paths. The tolerance is relative to sum|w*x|, so
a small element must keep its own relative precision even when it shares a
vector (or a block of 64) with an element 10^5 times larger, and an element
whose weight is zero must contribute exactly nothing, however large it is.

The weight patterns are laid down through the format's word rule (element
16w+i of a block is bits 2i of the little-endian word at byte 2+4w); a CPU
test checks them against the oracle's decode.
"""
import numpy as np

import synth


def set_code(w, N, K, row, elem, code):
    """Sets the 2-bit code of weight (row, elem) in packed bytes w (in place)."""
    blk = (row * (K // 64) + elem // 64) * 18
    e = elem % 64
    byte = blk + 2 + 4 * (e // 16) + (e % 16) // 4
    sh = 2 * (e % 4)
    w[byte] = (int(w[byte]) & ~(3 << sh) & 0xFF) | (code << sh)


def all_code2(g, N, K):
    """N x K matrix whose codes are all 2 (+d), scales fp16 of U[0.005, 0.05]."""
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE)
    w.reshape(-1, 18)[:, 2:] = 0xAA
    return w


def wide_range_case(kind, g, N, K, ncols):
    """(w, x) for the wide-range kinds:
      const_outliers   x = 0.01 except one +-300 and one +-3000 per column; every
                       row all code 2 except code 1 at the outlier positions;
      normal_outliers  x ~ N(0, 0.01^2) with one +-3000 per column; random
                       codes, with code 1 at the outlier in the even rows;
      block_outliers   x = 0.01 except one +-100 in every block of 64 (at a
                       seeded element); rows all code 2, code 1 at those
                       elements;
      mixed_scales     blocks of x scaled by 10^k, k uniform in [-6, 4]; random
                       codes.
    """
    if kind == "const_outliers":
        x = np.full((ncols, K), 0.01, dtype=np.float32)
        w = all_code2(g, N, K)
        for c in range(ncols):
            p = g.choice(K, size=2, replace=False)
            s = np.where(g.integers(0, 2, size=2) == 0, -1.0, 1.0)
            x[c, p[0]] = np.float32(300.0 * s[0])
            x[c, p[1]] = np.float32(3000.0 * s[1])
            for r in range(N):
                set_code(w, N, K, r, int(p[0]), 1)
                set_code(w, N, K, r, int(p[1]), 1)
    elif kind == "normal_outliers":
        x = (g.standard_normal((ncols, K)) * 0.01).astype(np.float32)
        w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
        for c in range(ncols):
            p = int(g.integers(0, K))
            x[c, p] = np.float32(3000.0 if g.integers(0, 2) else -3000.0)
            for r in range(0, N, 2):
                set_code(w, N, K, r, p, 1)
    elif kind == "block_outliers":
        x = np.full((ncols, K), 0.01, dtype=np.float32)
        w = all_code2(g, N, K)
        pos = np.arange(0, K, 64) + g.integers(0, 64, size=K // 64)
        for c in range(ncols):
            x[c, pos] = np.float32(100.0)
        for r in range(N):
            for p in pos:
                set_code(w, N, K, r, int(p), 1)
    elif kind == "mixed_scales":
        x = g.standard_normal((ncols, K)).astype(np.float32)
        k = g.integers(-6, 5, size=(ncols, K // 64)).astype(np.float64)
        x = (x.reshape(ncols, K // 64, 64) * (10.0 ** k)[..., None]).astype(np.float32)
        x = x.reshape(ncols, K)
        w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    else:
        raise ValueError(kind)
    return w, x


WIDE_KINDS = ["const_outliers", "normal_outliers", "block_outliers", "mixed_scales"]


def to_g128(w, N, K):
    """The same codes in the group-128 packing: blocks 2i and 2i+1 of a row
    (18 bytes each) become one 34-byte block with block 2i's scale and the two
    blocks' code bytes in order. The weights of odd blocks change scale with it;
    the oracle reads the group-128 bytes, so both sides see the same matrix."""
    b = w.reshape(N, K // 128, 2, 18)
    out = np.empty((N, K // 128, 34), dtype=np.uint8)
    out[:, :, 0:2] = b[:, :, 0, 0:2]
    out[:, :, 2:18] = b[:, :, 0, 2:18]
    out[:, :, 18:34] = b[:, :, 1, 2:18]
    return out.reshape(-1)
