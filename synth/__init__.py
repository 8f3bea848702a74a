"""Seeded synthetic inputs shared by the tests, the benchmark and the smoke check.

This module holds no Q2_0 arithmetic: it never decodes a block, never maps an
element index to a bit position and never computes a product. It draws raw
block bytes by a layout-agnostic recipe — a 2-byte little-endian fp16 scale
followed by 16 code bytes whose four 2-bit fields are drawn independently — so
that neither the oracle nor the CUDA library depends on it for the format.

Workloads are the decoder shapes the Q2_0 pages discuss (Ternary Bonsai
1.7B/8B, built on Qwen3), stated with their sizes. No trained weights or
datasets are involved.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

BLOCK_WEIGHTS = 64
BLOCK_BYTES = 18

# All bytes whose four 2-bit fields each lie in {0, 1, 2}: 3^4 = 81 values.
_TERNARY_BYTES = np.array(
    [a | (b << 2) | (c << 4) | (d << 6)
     for a in range(3) for b in range(3) for c in range(3) for d in range(3)],
    dtype=np.uint8)


def rng(seed, *stream) -> np.random.Generator:
    """Independent PCG64 stream for (seed, *stream) — e.g. (config, layer, matrix)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([int(seed), *map(int, stream)])))


def fp16_bits(values) -> np.ndarray:
    """IEEE binary16 bit patterns of values (numpy's float16 conversion)."""
    return np.asarray(values, dtype=np.float32).astype(np.float16).view(np.uint16)


def packed_matrix(g: np.random.Generator, N: int, K: int, scale_lo: float, scale_hi: float,
                  frac_code3: float = 0.0) -> np.ndarray:
    """Raw bytes of an N x K Q2_0 matrix (N * K/64 blocks of 18 bytes).

    Scales: fp16 of U[scale_lo, scale_hi]. Codes: iid uniform over {0, 1, 2};
    then a fraction ``frac_code3`` of the 2-bit fields, at seeded positions, is
    set to 3 (the reserved level).
    """
    assert K % BLOCK_WEIGHTS == 0
    nb = N * (K // BLOCK_WEIGHTS)
    out = np.empty((nb, BLOCK_BYTES), dtype=np.uint8)
    d = fp16_bits(g.uniform(scale_lo, scale_hi, size=nb).astype(np.float32))
    out[:, 0] = (d & 0xFF).astype(np.uint8)
    out[:, 1] = (d >> 8).astype(np.uint8)
    out[:, 2:] = _TERNARY_BYTES[g.integers(0, 81, size=(nb, 16), dtype=np.uint8)]
    if frac_code3 > 0.0:
        nfields = nb * 16 * 4
        n3 = int(round(frac_code3 * nfields))
        pos = g.choice(nfields, size=n3, replace=False) if nfields < 1_000_000 else \
            np.unique(g.integers(0, nfields, size=n3, dtype=np.int64))
        byte_idx = pos // 4
        field = (pos % 4).astype(np.uint8)
        codes = out[:, 2:].reshape(-1)
        np.bitwise_or.at(codes, byte_idx, (np.uint8(3) << (2 * field)).astype(np.uint8))
        out[:, 2:] = codes.reshape(nb, 16)
    return out.reshape(-1)


def packed_matrix_device(torch, gen, N: int, K: int, scale_lo: float, scale_hi: float,
                         frac_code3: float, device):
    """The recipe of ``packed_matrix`` drawn on the GPU with a seeded
    ``torch.Generator`` (for timing large workloads whose host generation would
    take minutes; the bytes differ from the host stream, the distribution is the
    same). Returns a uint8 device tensor of N * K/64 * 18 bytes."""
    assert K % BLOCK_WEIGHTS == 0
    nb = N * (K // BLOCK_WEIGHTS)
    table = torch.from_numpy(_TERNARY_BYTES).to(device)
    d = (torch.rand(nb, generator=gen, device=device) * (scale_hi - scale_lo) + scale_lo).half()
    codes = table[torch.randint(0, 81, (nb, 16), generator=gen, device=device)]
    if frac_code3 > 0.0:
        field = torch.randint(0, 4, (nb, 16), generator=gen, device=device, dtype=torch.uint8)
        hit = torch.rand((nb, 16), generator=gen, device=device) < 4.0 * frac_code3
        # each code byte carries four fields: hitting a byte with probability 4f
        # and one field in it sets a fraction f of all fields to 3
        codes = torch.where(hit, codes | (torch.tensor(3, dtype=torch.uint8, device=device)
                                          << (2 * field)), codes)
    out = torch.empty((nb, BLOCK_BYTES), dtype=torch.uint8, device=device)
    out[:, 0:2] = d.view(torch.uint8).view(nb, 2)
    out[:, 2:] = codes
    return out.reshape(-1)


def packed_matrix_g128(g: np.random.Generator, N: int, K: int, scale_lo: float,
                       scale_hi: float) -> np.ndarray:
    """Raw bytes of an N x K matrix in the group-128 packing: N * K/128 blocks of
    34 bytes, a 2-byte fp16 scale (fp16 of U[scale_lo, scale_hi]) then 32 code
    bytes whose four 2-bit fields are iid uniform over {0, 1, 2}."""
    assert K % 128 == 0
    nb = N * (K // 128)
    out = np.empty((nb, 34), dtype=np.uint8)
    d = fp16_bits(g.uniform(scale_lo, scale_hi, size=nb).astype(np.float32))
    out[:, 0] = (d & 0xFF).astype(np.uint8)
    out[:, 1] = (d >> 8).astype(np.uint8)
    out[:, 2:] = _TERNARY_BYTES[g.integers(0, 81, size=(nb, 32), dtype=np.uint8)]
    return out.reshape(-1)


def activations(g: np.random.Generator, rows: int, K: int, frac_outlier: float = 0.0,
                outlier: float = 30.0) -> np.ndarray:
    """f32 [rows][K] ~ N(0,1); a fraction of entries at seeded positions = ±outlier."""
    x = g.standard_normal(size=(rows, K), dtype=np.float32)
    if frac_outlier > 0.0:
        n = int(round(frac_outlier * x.size))
        pos = g.choice(x.size, size=n, replace=False)
        sign = np.where(g.integers(0, 2, size=n) == 0, -1.0, 1.0).astype(np.float32)
        x.reshape(-1)[pos] = sign * np.float32(outlier)
    return x


def edge_blocks() -> np.ndarray:
    """Hand-chosen blocks: d = +0, subnormal d (0x0001, 0x03FF), negative d,
    all-code-3, all-code-1, all-code-0 with d = +0, and a large d."""
    rows = []

    def blk(dbits, qbyte):
        b = np.empty(BLOCK_BYTES, dtype=np.uint8)
        b[0] = dbits & 0xFF
        b[1] = dbits >> 8
        b[2:] = qbyte
        return b

    rows.append(blk(0x0000, 0x24))   # d = +0, mixed codes
    rows.append(blk(0x0001, 0x1B))   # smallest subnormal d
    rows.append(blk(0x03FF, 0x93))   # largest subnormal d
    rows.append(blk(0x3C00, 0xFF))   # all code 3, d = 1
    rows.append(blk(0x2E66, 0x55))   # all code 1 (zero weights)
    rows.append(blk(0x0000, 0x00))   # all code 0 with d = +0
    rows.append(blk(0xB800, 0x55))   # all code 1 with d = -0.5
    rows.append(blk(0x8000, 0xE4))   # d = -0
    rows.append(blk(0x7BFF, 0x86))   # d = 65504 (largest finite)
    return np.stack(rows)


def token_ids(g: np.random.Generator, n: int, vocab: int, frac_repeat: float = 0.05,
              head: np.ndarray | None = None) -> np.ndarray:
    """int32 ids uniform over [0, vocab); about ``frac_repeat`` of them repeat an
    earlier id; optional fixed ``head`` ids are placed first."""
    ids = g.integers(0, vocab, size=n, dtype=np.int64)
    nrep = int(round(frac_repeat * n))
    if nrep and n > 1:
        dst = g.choice(np.arange(1, n), size=min(nrep, n - 1), replace=False)
        for j in dst:
            ids[j] = ids[g.integers(0, j)]
    if head is not None:
        ids[:len(head)] = head
    return ids.astype(np.int32)


# ---------------------------------------------------------------------------
# Workloads (shapes of the 1.7B- and 8B-class decoders the pages discuss)
# ---------------------------------------------------------------------------
@dataclass(frozen=True)
class Mat:
    name: str
    N: int
    K: int


def decoder_1p7b_layer():
    h = 2048
    return [Mat("q", 2048, h), Mat("k", 1024, h), Mat("v", 1024, h), Mat("o", 2048, h),
            Mat("gate", 6144, h), Mat("up", 6144, h), Mat("down", h, 6144)]


def decoder_8b_layer():
    h = 4096
    return [Mat("q", 4096, h), Mat("k", 1024, h), Mat("v", 1024, h), Mat("o", 4096, h),
            Mat("gate", 12288, h), Mat("up", 12288, h), Mat("down", h, 12288)]


def decode_step_1p7b():
    """28 layers x 7 Q2_0 matrices = 196 matrices, hidden 2048."""
    return [(l, m) for l in range(28) for m in decoder_1p7b_layer()]


def decode_step_8b(with_head: bool = True):
    """36 layers x 7 matrices (+ a 151936 x 4096 output head) = 253 matrices."""
    mats = [(l, m) for l in range(36) for m in decoder_8b_layer()]
    if with_head:
        mats.append((36, Mat("head", 151936, 4096)))
    return mats


def packed_size(N: int, K: int) -> int:
    return N * (K // BLOCK_WEIGHTS) * BLOCK_BYTES


# Distributions of the decode-step workloads (codes, scales, activations).
DECODE_SCALE = (0.005, 0.05)
DECODE_FRAC_CODE3 = 0.01
MATVEC_SMALL_SCALE = (0.01, 0.05)
PREFILL_OUTLIER_FRAC = 0.001
PREFILL_OUTLIER = 30.0
