"""Q2_0 oracle — TEST INFRASTRUCTURE ONLY.

A plain fp64 CPU statement of the Q2_0 block decode, the dequantize-then-dot
product, get_rows and the reference quantizer, written in C
(``q2_0_oracle.c``) and loaded here through ctypes. Only the test suite,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may import it;
the product library (``bit_ternary_matmul_gb300``) never does, and the two
share no code.

``build()`` compiles the C file with gcc (OpenMP when available) into
``oracle/_lib/``. Pure-Python helpers below only marshal numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q2_0_oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "libq2_0_oracle.so")
_lock = threading.Lock()
_lib = None

WEIGHTS_PER_BLOCK = 64
BYTES_PER_BLOCK = 18


def build(force: bool = False) -> str:
    """Compile the oracle into a shared library; returns its path."""
    os.makedirs(_LIBDIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = ctypes.CDLL(path)
            u8p = ctypes.POINTER(ctypes.c_uint8)
            f32p = ctypes.POINTER(ctypes.c_float)
            f64p = ctypes.POINTER(ctypes.c_double)
            i64p = ctypes.POINTER(ctypes.c_int64)
            i32p = ctypes.POINTER(ctypes.c_int32)
            i64 = ctypes.c_int64
            L.qo_half_to_double.argtypes = [ctypes.c_uint16]
            L.qo_half_to_double.restype = ctypes.c_double
            L.qo_float_to_half_rn.argtypes = [ctypes.c_float]
            L.qo_float_to_half_rn.restype = ctypes.c_uint16
            L.qo_decode_block.argtypes = [u8p, f64p]
            L.qo_block_codes.argtypes = [u8p, u8p]
            L.qo_block_scale_bits.argtypes = [u8p]
            L.qo_block_scale_bits.restype = ctypes.c_uint16
            L.qo_dequantize_rows.argtypes = [u8p, i64, i64, i64, f64p]
            L.qo_matmul_rows.argtypes = [u8p, i64, i64, f32p, i64, i64p, i64, f64p, f64p]
            L.qo_get_rows.argtypes = [u8p, i64, i64, i32p, i64, f32p]
            L.qo_matmul_id.argtypes = [u8p, i64, i64, i64, f32p, i64, i32p, i64, i64, i64p, i64,
                                       f64p, f64p]
            L.qo_matmul_id.restype = i64
            L.qo_soa_bytes.argtypes = [i64, i64]
            L.qo_soa_bytes.restype = i64
            L.qo_raw_to_soa.argtypes = [u8p, i64, i64, u8p]
            L.qo_soa_to_raw.argtypes = [u8p, i64, i64, u8p]
            L.qo_get_rows.restype = i64
            L.qo_quantize_block.argtypes = [f32p, u8p]
            L.qo_quantize_rows.argtypes = [f32p, i64, i64, u8p]
            L.qo_packed_bytes.argtypes = [i64, i64, i64]
            L.qo_packed_bytes.restype = i64
            L.qo_half_to_double_array.argtypes = [ctypes.POINTER(ctypes.c_uint16), f64p, i64]
            L.qo_float_to_half_rn_array.argtypes = [f32p, ctypes.POINTER(ctypes.c_uint16), i64]
            L.qo_num_threads.restype = ctypes.c_int
            L.qo_set_num_threads.argtypes = [ctypes.c_int]
            L.qo_decode_block_g128.argtypes = [u8p, f64p]
            L.qo_matmul_rows_g128.argtypes = [u8p, i64, i64, f32p, i64, i64p, i64, f64p, f64p]
            L.qo_get_rows_g128.argtypes = [u8p, i64, i64, i32p, i64, f32p]
            L.qo_get_rows_g128.restype = i64
            L.qo_weights_per_block.restype = ctypes.c_int
            L.qo_bytes_per_block.restype = ctypes.c_int
            _lib = L
    return _lib


def _p(a: np.ndarray, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _u8(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.uint8)


def num_threads() -> int:
    return lib().qo_num_threads()


def set_num_threads(n: int) -> None:
    lib().qo_set_num_threads(int(n))


def half_to_double(bits: int) -> float:
    return lib().qo_half_to_double(int(bits) & 0xFFFF)


def halves_to_double(bits) -> np.ndarray:
    h = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float64)
    lib().qo_half_to_double_array(_p(h, ctypes.c_uint16), _p(out, ctypes.c_double), h.size)
    return out


def floats_to_half_rn(values) -> np.ndarray:
    f = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(f.shape, dtype=np.uint16)
    lib().qo_float_to_half_rn_array(_p(f, ctypes.c_float), _p(out, ctypes.c_uint16), f.size)
    return out


def float_to_half_rn(v: float) -> int:
    return int(lib().qo_float_to_half_rn(float(v)))


def block_scale_bits(block) -> int:
    b = _u8(block)
    assert b.size == BYTES_PER_BLOCK
    return int(lib().qo_block_scale_bits(_p(b, ctypes.c_uint8)))


def decode_block(block) -> np.ndarray:
    b = _u8(block)
    assert b.size == BYTES_PER_BLOCK
    out = np.empty(WEIGHTS_PER_BLOCK, dtype=np.float64)
    lib().qo_decode_block(_p(b, ctypes.c_uint8), _p(out, ctypes.c_double))
    return out


def block_codes(block) -> np.ndarray:
    b = _u8(block)
    out = np.empty(WEIGHTS_PER_BLOCK, dtype=np.uint8)
    lib().qo_block_codes(_p(b, ctypes.c_uint8), _p(out, ctypes.c_uint8))
    return out


def dequantize(w, N: int, K: int, r0: int = 0, nr: int | None = None) -> np.ndarray:
    """fp64 [nr][K] of rows r0..r0+nr of the packed N x K matrix."""
    wb = _u8(w)
    nr = N - r0 if nr is None else nr
    assert wb.size >= N * (K // 64) * 18
    out = np.empty((nr, K), dtype=np.float64)
    lib().qo_dequantize_rows(_p(wb, ctypes.c_uint8), K, r0, nr, _p(out, ctypes.c_double))
    return out


def matmul(w, N: int, K: int, x, rows=None):
    """fp64 (y, acc): y[c][j] = sum_k W[rows[j]][k] x[c][k], acc = sum |W x|.

    x is f32 [ncols][K] (a 1-D x is one column). rows=None means all N rows.
    """
    wb = _u8(w)
    xx = np.ascontiguousarray(x, dtype=np.float32)
    if xx.ndim == 1:
        xx = xx[None, :]
    assert xx.shape[1] == K and K % 64 == 0
    assert wb.size >= N * (K // 64) * 18
    ncols = xx.shape[0]
    if rows is None:
        nr = N
        rp = None
    else:
        rr = np.ascontiguousarray(rows, dtype=np.int64)
        assert rr.size == 0 or (rr.min() >= 0 and rr.max() < N)
        nr = rr.size
        rp = _p(rr, ctypes.c_int64)
    y = np.empty((ncols, nr), dtype=np.float64)
    acc = np.empty((ncols, nr), dtype=np.float64)
    lib().qo_matmul_rows(_p(wb, ctypes.c_uint8), N, K, _p(xx, ctypes.c_float), ncols,
                         rp, nr, _p(y, ctypes.c_double), _p(acc, ctypes.c_double))
    return y, acc


def matmul_id(w, n_expert: int, N: int, K: int, x, ids, rows=None):
    """Expert mat-vec: (y, acc, n_bad), y and acc fp64 [n_tokens][n_used][nr].

    w: n_expert matrices of N x K, one after another. ids: int [n_tokens][n_used].
    x: f32 [n_tokens][n_x][K] with n_x = 1 (shared by the token's experts) or
    n_used. Slots with an id outside [0, n_expert) are counted in n_bad and
    their rows of y and acc are NaN.
    """
    wb = _u8(w)
    ii = np.ascontiguousarray(ids, dtype=np.int32)
    assert ii.ndim == 2
    n_tokens, n_used = ii.shape
    xx = np.ascontiguousarray(x, dtype=np.float32)
    assert xx.ndim == 3 and xx.shape[0] == n_tokens and xx.shape[2] == K and K % 64 == 0
    n_x = xx.shape[1]
    assert n_x in (1, n_used)
    assert wb.size >= n_expert * N * (K // 64) * 18
    if rows is None:
        nr, rp = N, None
    else:
        rr = np.ascontiguousarray(rows, dtype=np.int64)
        assert rr.size == 0 or (rr.min() >= 0 and rr.max() < N)
        nr, rp = rr.size, _p(rr, ctypes.c_int64)
    y = np.full((n_tokens, n_used, nr), np.nan, dtype=np.float64)
    acc = np.full((n_tokens, n_used, nr), np.nan, dtype=np.float64)
    bad = lib().qo_matmul_id(_p(wb, ctypes.c_uint8), n_expert, N, K, _p(xx, ctypes.c_float), n_x,
                             _p(ii, ctypes.c_int32), n_used, n_tokens, rp, nr,
                             _p(y, ctypes.c_double), _p(acc, ctypes.c_double))
    return y, acc, int(bad)


def soa_bytes(N: int, K: int) -> int:
    """Bytes of the split layout: 16 code bytes per block, then (256-byte
    aligned) a 2-byte scale per block."""
    return int(lib().qo_soa_bytes(N, K))


def raw_to_soa(w, N: int, K: int) -> np.ndarray:
    wb = _u8(w)
    assert wb.size >= N * (K // 64) * 18
    out = np.zeros(soa_bytes(N, K), dtype=np.uint8)
    lib().qo_raw_to_soa(_p(wb, ctypes.c_uint8), N, K, _p(out, ctypes.c_uint8))
    return out


def soa_to_raw(soa, N: int, K: int) -> np.ndarray:
    sb = _u8(soa)
    assert sb.size >= soa_bytes(N, K)
    out = np.empty(N * (K // 64) * 18, dtype=np.uint8)
    lib().qo_soa_to_raw(_p(sb, ctypes.c_uint8), N, K, _p(out, ctypes.c_uint8))
    return out


def matmul_soa(soa, N: int, K: int, x, rows=None):
    """matmul of a matrix stored in the split layout (back to blocks, then dot)."""
    return matmul(soa_to_raw(soa, N, K), N, K, x, rows)


def get_rows(table, n_rows: int, K: int, ids):
    """(out f32 [n_ids][K], n_bad); rows of out for bad ids are zero."""
    tb = _u8(table)
    ii = np.ascontiguousarray(ids, dtype=np.int32)
    out = np.zeros((ii.size, K), dtype=np.float32)
    bad = lib().qo_get_rows(_p(tb, ctypes.c_uint8), n_rows, K, _p(ii, ctypes.c_int32),
                            ii.size, _p(out, ctypes.c_float))
    return out, int(bad)


# ---- group-128 blocks (34 bytes per 128 weights) ------------------------------
def decode_block_g128(block) -> np.ndarray:
    b = _u8(block)
    assert b.size == 34
    out = np.empty(128, dtype=np.float64)
    lib().qo_decode_block_g128(_p(b, ctypes.c_uint8), _p(out, ctypes.c_double))
    return out


def matmul_g128(w, N: int, K: int, x, rows=None):
    """As matmul for an N x K group-128 matrix (K % 128 == 0)."""
    wb = _u8(w)
    xx = np.ascontiguousarray(x, dtype=np.float32)
    if xx.ndim == 1:
        xx = xx[None, :]
    assert xx.shape[1] == K and K % 128 == 0
    assert wb.size >= N * (K // 128) * 34
    ncols = xx.shape[0]
    if rows is None:
        nr, rp = N, None
    else:
        rr = np.ascontiguousarray(rows, dtype=np.int64)
        assert rr.size == 0 or (rr.min() >= 0 and rr.max() < N)
        nr, rp = rr.size, _p(rr, ctypes.c_int64)
    y = np.empty((ncols, nr), dtype=np.float64)
    acc = np.empty((ncols, nr), dtype=np.float64)
    lib().qo_matmul_rows_g128(_p(wb, ctypes.c_uint8), N, K, _p(xx, ctypes.c_float), ncols, rp,
                              nr, _p(y, ctypes.c_double), _p(acc, ctypes.c_double))
    return y, acc


def get_rows_g128(table, n_rows: int, K: int, ids):
    """As get_rows for a group-128 table."""
    tb = _u8(table)
    ii = np.ascontiguousarray(ids, dtype=np.int32)
    out = np.zeros((ii.size, K), dtype=np.float32)
    bad = lib().qo_get_rows_g128(_p(tb, ctypes.c_uint8), n_rows, K, _p(ii, ctypes.c_int32),
                                 ii.size, _p(out, ctypes.c_float))
    return out, int(bad)


def quantize(src, nrows: int, K: int) -> np.ndarray:
    """Reference quantizer: f32 [nrows][K] -> packed bytes (uint8)."""
    s = np.ascontiguousarray(src, dtype=np.float32)
    assert s.size == nrows * K and K % 64 == 0
    dst = np.zeros(nrows * (K // 64) * 18, dtype=np.uint8)
    lib().qo_quantize_rows(_p(s, ctypes.c_float), nrows, K, _p(dst, ctypes.c_uint8))
    return dst


def packed_bytes(N: int, K: int, group: int = 64) -> int:
    return int(lib().qo_packed_bytes(N, K, group))


def within_tolerance(gpu, y, acc, rel: float, abs_: float = 0.0):
    """Mask of |gpu - y| <= rel * acc + abs_ (NaN/inf in gpu fails)."""
    g = np.asarray(gpu, dtype=np.float64)
    ok = np.isfinite(g) & (np.abs(g - y) <= rel * acc + abs_)
    return ok
