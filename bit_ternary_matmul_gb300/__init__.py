"""GB300-native Q2_0 dequantize-fused matmul — Python binding of libq2_0.

Thin ctypes marshalling over the C ABI declared in ``include/q2_0.h``: the
functions here carry the same names as the C entry points, check tensor
dtype/device/contiguity, pass ``data_ptr()`` values and the current CUDA stream,
and raise on a non-OK status. Every result is computed by the library's CUDA
kernels; there is no CPU path. PyTorch provides device memory and streams only.

Q2_0 (sources: "WebGPU: add Q2_0 support", bisque.today write-up of llama.cpp
PR 30914, format paragraph; "Llama.cpp umí dvoubitový Q2_0 i na kartách
NVIDIA", aisvetem.cz, section "Osmnáct bajtů na čtyřiašedesát vah"): 64 weights
per 18-byte block — fp16 scale d, then four little-endian u32 words of 2-bit
codes q; a weight is (q - 1) * d.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from ._build import LIB as _LIB_PATH
from ._build import build as _build

BLOCK_WEIGHTS = 64
BLOCK_BYTES = 18

Q2_0_OK = 0
Q2_0_EINVAL = 1
Q2_0_ECUDA = 2
Q2_0_EUNSUPPORTED = 3
Q2_0_EDEVICE = 4
Q2_0_ENOSPACE = 5
Q2_0_NOALLOC_SCRATCH_BYTES = 1 << 20

Q2_0_PREC_F16_SPLIT = 0
Q2_0_PREC_F16 = 1

Q2_0_DEVERR_NONE = 0
Q2_0_DEVERR_BAD_ID = 1
Q2_0_DEVERR_TIMEOUT = 2

_STATUS = {0: "Q2_0_OK", 1: "Q2_0_EINVAL", 2: "Q2_0_ECUDA", 3: "Q2_0_EUNSUPPORTED",
           4: "Q2_0_EDEVICE", 5: "Q2_0_ENOSPACE"}

# Every symbol include/q2_0.h declares.
EXPORTS = (
    "q2_0_version", "q2_0_device_check", "q2_0_mul_mat_vec", "q2_0_mul_mat_vec_workspace_size",
    "q2_0_mul_mat_vec_ws", "q2_0_mul_mat_vec_noalloc", "q2_0_test_inject_stall",
    "q2_0_mv_plan_create", "q2_0_mv_plan_execute",
    "q2_0_mv_plan_launches", "q2_0_mv_plan_destroy", "q2_0_mul_mat_workspace_size",
    "q2_0_mul_mat", "q2_0_get_rows", "q2_0_quantize_ref", "q2_0_get_error",
    "q2_0_mul_mat_vec_f16", "q2_0_mul_mat_f16",
    "q2_0_g128_to_g64", "q2_0_g128_get_rows", "q2_0_g128_mul_mat_vec",
    "q2_0_mul_mat_id_workspace_size", "q2_0_mul_mat_id",
    "q2_0_split_bytes", "q2_0_split_layout", "q2_0_join_layout", "q2_0_mul_mat_vec_split",
    "q2_0_mm_plan_create", "q2_0_mm_plan_execute", "q2_0_mm_plan_launches",
    "q2_0_mm_plan_destroy",
)


class Q2Error(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {_STATUS.get(status, status)}")
        self.status = status


class _MvDesc(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class _MmDesc(ctypes.Structure):
    _fields_ = [("w", ctypes.c_void_p), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p),
                ("N", ctypes.c_int64), ("K", ctypes.c_int64), ("M", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile libq2_0.so in-tree for sm_103a (no-op when up to date)."""
    return _build(force=force)


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded libq2_0 (raises if it has not been built: there is no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise RuntimeError(
                    "libq2_0.so is not built; run bit_ternary_matmul_gb300.build() "
                    "(the CUDA library is required, there is no CPU fallback)")
            L = ctypes.CDLL(_LIB_PATH)
            vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
            L.q2_0_version.restype = ctypes.c_char_p
            L.q2_0_device_check.restype = i32
            L.q2_0_mul_mat_vec.argtypes = [vp, vp, vp, i64, i64, i32, vp]
            L.q2_0_mul_mat_vec.restype = i32
            L.q2_0_mul_mat_vec_workspace_size.argtypes = [i64, i32]
            L.q2_0_mul_mat_vec_workspace_size.restype = sz
            L.q2_0_mul_mat_vec_ws.argtypes = [vp, vp, vp, i64, i64, i32, vp, sz, vp]
            L.q2_0_mul_mat_vec_ws.restype = i32
            L.q2_0_mul_mat_vec_noalloc.argtypes = [vp, vp, vp, i64, i64, i32, vp]
            L.q2_0_mul_mat_vec_noalloc.restype = i32
            L.q2_0_test_inject_stall.argtypes = [i32, ctypes.c_uint64]
            L.q2_0_test_inject_stall.restype = i32
            L.q2_0_mv_plan_create.argtypes = [ctypes.POINTER(_MvDesc), i32, i32,
                                              ctypes.POINTER(vp)]
            L.q2_0_mv_plan_create.restype = i32
            L.q2_0_mv_plan_execute.argtypes = [vp, vp]
            L.q2_0_mv_plan_execute.restype = i32
            L.q2_0_mv_plan_launches.argtypes = [vp]
            L.q2_0_mv_plan_launches.restype = i32
            L.q2_0_mv_plan_destroy.argtypes = [vp]
            L.q2_0_mv_plan_destroy.restype = None
            L.q2_0_mul_mat_workspace_size.argtypes = [i64, i64, i64, i32]
            L.q2_0_mul_mat_workspace_size.restype = sz
            L.q2_0_mul_mat.argtypes = [vp, vp, vp, i64, i64, i64, i32, vp, sz, vp]
            L.q2_0_mul_mat.restype = i32
            L.q2_0_mm_plan_create.argtypes = [ctypes.POINTER(_MmDesc), i32, i32,
                                              ctypes.POINTER(vp)]
            L.q2_0_mm_plan_create.restype = i32
            L.q2_0_mm_plan_execute.argtypes = [vp, vp]
            L.q2_0_mm_plan_execute.restype = i32
            L.q2_0_mm_plan_launches.argtypes = [vp]
            L.q2_0_mm_plan_launches.restype = i32
            L.q2_0_mm_plan_destroy.argtypes = [vp]
            L.q2_0_mm_plan_destroy.restype = None
            L.q2_0_mul_mat_vec_f16.argtypes = [vp, vp, vp, i64, i64, i32, vp]
            L.q2_0_mul_mat_vec_f16.restype = i32
            L.q2_0_mul_mat_f16.argtypes = [vp, vp, vp, i64, i64, i64, vp, sz, vp]
            L.q2_0_mul_mat_f16.restype = i32
            L.q2_0_g128_to_g64.argtypes = [vp, vp, i64, i64, vp]
            L.q2_0_g128_to_g64.restype = i32
            L.q2_0_g128_get_rows.argtypes = [vp, i64, i64, vp, i64, vp, vp]
            L.q2_0_g128_get_rows.restype = i32
            L.q2_0_g128_mul_mat_vec.argtypes = [vp, vp, vp, i64, i64, i32, vp]
            L.q2_0_g128_mul_mat_vec.restype = i32
            L.q2_0_get_rows.argtypes = [vp, i64, i64, vp, i64, vp, vp]
            L.q2_0_get_rows.restype = i32
            L.q2_0_mul_mat_id_workspace_size.argtypes = [i64, i64, i64]
            L.q2_0_mul_mat_id_workspace_size.restype = sz
            L.q2_0_mul_mat_id.argtypes = [vp, i64, i64, i64, vp, i64, vp, i64, i64, vp, vp, sz, vp]
            L.q2_0_mul_mat_id.restype = i32
            L.q2_0_split_bytes.argtypes = [i64, i64]
            L.q2_0_split_bytes.restype = sz
            L.q2_0_split_layout.argtypes = [vp, vp, i64, i64, vp]
            L.q2_0_split_layout.restype = i32
            L.q2_0_join_layout.argtypes = [vp, vp, i64, i64, vp]
            L.q2_0_join_layout.restype = i32
            L.q2_0_mul_mat_vec_split.argtypes = [vp, vp, vp, i64, i64, i32, vp]
            L.q2_0_mul_mat_vec_split.restype = i32
            L.q2_0_quantize_ref.argtypes = [vp, vp, i64, i64, vp]
            L.q2_0_quantize_ref.restype = i32
            L.q2_0_get_error.argtypes = [vp, ctypes.POINTER(i64)]
            L.q2_0_get_error.restype = i32
            _lib = L
    return _lib


def _check(fn: str, status: int):
    if status != Q2_0_OK:
        raise Q2Error(fn, status)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str, dtype, numel: int | None = None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return t.data_ptr()


def packed_bytes(N: int, K: int) -> int:
    return N * (K // BLOCK_WEIGHTS) * BLOCK_BYTES


def q2_0_version() -> str:
    return lib().q2_0_version().decode()


def q2_0_device_check() -> int:
    return lib().q2_0_device_check()


def q2_0_mul_mat_vec(w: torch.Tensor, x: torch.Tensor, N: int, K: int, ncols: int | None = None,
                     y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[c][n] = sum_k W[n][k] x[c][k]; w uint8 packed, x f32 [ncols][K]."""
    ncols = x.shape[0] if (ncols is None and x.dim() == 2) else (ncols or 1)
    if y is None:
        y = torch.empty((ncols, N), dtype=torch.float32, device=x.device)
    st = lib().q2_0_mul_mat_vec(_dev(w, "w", torch.uint8, packed_bytes(N, K)),
                                _dev(x, "x", torch.float32, ncols * K),
                                _dev(y, "y", torch.float32, ncols * N), N, K, ncols, _stream(stream))
    _check("q2_0_mul_mat_vec", st)
    return y


def q2_0_mul_mat_vec_f16(w: torch.Tensor, x: torch.Tensor, N: int, K: int,
                         ncols: int | None = None, y: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    """As q2_0_mul_mat_vec with x F16 [ncols][K]."""
    ncols = x.shape[0] if (ncols is None and x.dim() == 2) else (ncols or 1)
    if y is None:
        y = torch.empty((ncols, N), dtype=torch.float32, device=x.device)
    st = lib().q2_0_mul_mat_vec_f16(_dev(w, "w", torch.uint8, packed_bytes(N, K)),
                                    _dev(x, "x", torch.float16, ncols * K),
                                    _dev(y, "y", torch.float32, ncols * N), N, K, ncols,
                                    _stream(stream))
    _check("q2_0_mul_mat_vec_f16", st)
    return y


def q2_0_mul_mat_vec_workspace_size(K: int, ncols: int) -> int:
    return int(lib().q2_0_mul_mat_vec_workspace_size(K, ncols))


def q2_0_mul_mat_vec_ws(w, x, N, K, ncols, workspace: torch.Tensor, y=None, stream=None):
    if y is None:
        y = torch.empty((ncols, N), dtype=torch.float32, device=x.device)
    need = q2_0_mul_mat_vec_workspace_size(K, ncols)
    st = lib().q2_0_mul_mat_vec_ws(_dev(w, "w", torch.uint8, packed_bytes(N, K)),
                                   _dev(x, "x", torch.float32, ncols * K),
                                   _dev(y, "y", torch.float32, ncols * N), N, K, ncols,
                                   _dev(workspace, "workspace", torch.uint8, need),
                                   workspace.numel(), _stream(stream))
    _check("q2_0_mul_mat_vec_ws", st)
    return y


def q2_0_mul_mat_vec_noalloc(w: torch.Tensor, x: torch.Tensor, N: int, K: int,
                             ncols: int | None = None, y: torch.Tensor | None = None,
                             stream=None) -> torch.Tensor:
    """q2_0_mul_mat_vec whose scratch is the library's static device array.

    For callers that cannot allocate device memory at call time. The output
    tensor is allocated here only when ``y`` is None; pass ``y`` to keep the call
    allocation-free. Calls that overlap on the GPU share the array and race.
    """
    ncols = x.shape[0] if (ncols is None and x.dim() == 2) else (ncols or 1)
    if y is None:
        y = torch.empty((ncols, N), dtype=torch.float32, device=x.device)
    st = lib().q2_0_mul_mat_vec_noalloc(_dev(w, "w", torch.uint8, packed_bytes(N, K)),
                                        _dev(x, "x", torch.float32, ncols * K),
                                        _dev(y, "y", torch.float32, ncols * N), N, K, ncols,
                                        _stream(stream))
    _check("q2_0_mul_mat_vec_noalloc", st)
    return y


class MvPlan:
    """A batched mat-vec plan (q2_0_mv_plan_*): keeps references to its tensors."""

    def __init__(self, entries, ncols: int):
        """entries: iterable of (w uint8, x f32 [ncols][K], y f32 [ncols][N], N, K)."""
        self._keep = []
        descs = []
        for (w, x, y, N, K) in entries:
            descs.append(_MvDesc(_dev(w, "w", torch.uint8, packed_bytes(N, K)),
                                 _dev(x, "x", torch.float32, ncols * K),
                                 _dev(y, "y", torch.float32, ncols * N), N, K))
            self._keep.append((w, x, y))
        arr = (_MvDesc * len(descs))(*descs)
        h = ctypes.c_void_p()
        _check("q2_0_mv_plan_create",
               lib().q2_0_mv_plan_create(arr, len(descs), ncols, ctypes.byref(h)))
        self._h = h
        self.ncols = ncols
        self.n = len(descs)

    @property
    def launches(self) -> int:
        return int(lib().q2_0_mv_plan_launches(self._h))

    def execute(self, stream=None):
        _check("q2_0_mv_plan_execute", lib().q2_0_mv_plan_execute(self._h, _stream(stream)))

    def close(self):
        if getattr(self, "_h", None):
            lib().q2_0_mv_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def q2_0_mul_mat_workspace_size(M: int, N: int, K: int, prec: int = Q2_0_PREC_F16_SPLIT) -> int:
    return int(lib().q2_0_mul_mat_workspace_size(M, N, K, prec))


def q2_0_mul_mat(w: torch.Tensor, x: torch.Tensor, N: int, K: int, M: int | None = None,
                 prec: int = Q2_0_PREC_F16_SPLIT, y: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y[m][n] = sum_k W[n][k] X[m][k]; x f32 [M][K] -> y f32 [M][N]."""
    M = x.shape[0] if M is None else M
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_bytes = workspace.numel()
        ws_ptr = _dev(workspace, "workspace", torch.uint8,
                      q2_0_mul_mat_workspace_size(M, N, K, prec))
    st = lib().q2_0_mul_mat(_dev(w, "w", torch.uint8, packed_bytes(N, K)),
                            _dev(x, "x", torch.float32, M * K),
                            _dev(y, "y", torch.float32, M * N), N, K, M, prec, ws_ptr, ws_bytes,
                            _stream(stream))
    _check("q2_0_mul_mat", st)
    return y


class MmPlan:
    """A grouped GEMM plan (q2_0_mm_plan_*): keeps references to its tensors."""

    def __init__(self, entries, prec: int = Q2_0_PREC_F16_SPLIT):
        """entries: iterable of (w uint8, x f32 [M][K], y f32 [M][N], N, K, M)."""
        self._keep = []
        descs = []
        for (w, x, y, N, K, M) in entries:
            descs.append(_MmDesc(_dev(w, "w", torch.uint8, packed_bytes(N, K)),
                                 _dev(x, "x", torch.float32, M * K),
                                 _dev(y, "y", torch.float32, M * N), N, K, M))
            self._keep.append((w, x, y))
        arr = (_MmDesc * len(descs))(*descs)
        h = ctypes.c_void_p()
        _check("q2_0_mm_plan_create",
               lib().q2_0_mm_plan_create(arr, len(descs), prec, ctypes.byref(h)))
        self._h = h
        self.prec = prec
        self.n = len(descs)

    @property
    def launches(self) -> int:
        return int(lib().q2_0_mm_plan_launches(self._h))

    def execute(self, stream=None):
        _check("q2_0_mm_plan_execute", lib().q2_0_mm_plan_execute(self._h, _stream(stream)))

    def close(self):
        if getattr(self, "_h", None):
            lib().q2_0_mm_plan_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def q2_0_mul_mat_f16(w: torch.Tensor, x: torch.Tensor, N: int, K: int, M: int | None = None,
                     y: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """As q2_0_mul_mat with x F16 [M][K] (exact fp16 operands; workspace size of
    Q2_0_PREC_F16)."""
    M = x.shape[0] if M is None else M
    if y is None:
        y = torch.empty((M, N), dtype=torch.float32, device=x.device)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        ws_bytes = workspace.numel()
        ws_ptr = _dev(workspace, "workspace", torch.uint8,
                      q2_0_mul_mat_workspace_size(M, N, K, Q2_0_PREC_F16))
    st = lib().q2_0_mul_mat_f16(_dev(w, "w", torch.uint8, packed_bytes(N, K)),
                                _dev(x, "x", torch.float16, M * K),
                                _dev(y, "y", torch.float32, M * N), N, K, M, ws_ptr, ws_bytes,
                                _stream(stream))
    _check("q2_0_mul_mat_f16", st)
    return y


def q2_0_get_rows(table: torch.Tensor, n_rows: int, K: int, ids: torch.Tensor,
                  out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """out[r] = row ids[r] of the Q2_0 table as F32 (bit-exact)."""
    n_ids = ids.numel()
    if out is None:
        out = torch.empty((n_ids, K), dtype=torch.float32, device=ids.device)
    if n_ids == 0:
        return out
    st = lib().q2_0_get_rows(_dev(table, "table", torch.uint8, packed_bytes(n_rows, K)), n_rows, K,
                             _dev(ids, "ids", torch.int32, n_ids), n_ids,
                             _dev(out, "out", torch.float32, n_ids * K), _stream(stream))
    _check("q2_0_get_rows", st)
    return out


def q2_0_mul_mat_id_workspace_size(K: int, n_tokens: int, n_x: int) -> int:
    return int(lib().q2_0_mul_mat_id_workspace_size(K, n_tokens, n_x))


def q2_0_mul_mat_id(w: torch.Tensor, n_expert: int, N: int, K: int, x: torch.Tensor,
                    ids: torch.Tensor, y: torch.Tensor | None = None,
                    workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Expert mat-vec: y[t][i] = W_{ids[t][i]} x[t][i or 0].

    w: n_expert packed N x K matrices, one after another; x: f32 [n_tokens][n_x][K]
    (n_x = 1 or n_used; a 2-D x is n_x = 1); ids: int32 [n_tokens][n_used];
    y: f32 [n_tokens][n_used][N].
    """
    n_tokens, n_used = ids.shape
    n_x = 1 if x.dim() == 2 else x.shape[1]
    if y is None:
        y = torch.empty((n_tokens, n_used, N), dtype=torch.float32, device=ids.device)
    if n_tokens == 0:
        return y
    need = q2_0_mul_mat_id_workspace_size(K, n_tokens, n_x)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=ids.device)
    wsp = _dev(workspace, "workspace", torch.uint8, need) if need > 0 else None
    st = lib().q2_0_mul_mat_id(_dev(w, "w", torch.uint8, n_expert * packed_bytes(N, K)), n_expert,
                               N, K, _dev(x, "x", torch.float32, n_tokens * n_x * K), n_x,
                               _dev(ids, "ids", torch.int32, n_tokens * n_used), n_used, n_tokens,
                               _dev(y, "y", torch.float32, n_tokens * n_used * N), wsp,
                               need if need > 0 else 0, _stream(stream))
    _check("q2_0_mul_mat_id", st)
    return y


def q2_0_split_bytes(N: int, K: int) -> int:
    return int(lib().q2_0_split_bytes(N, K))


def q2_0_split_layout(w: torch.Tensor, N: int, K: int, dst: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """18-byte blocks -> split layout (codes, then 256-byte aligned fp16 scales)."""
    nbytes = q2_0_split_bytes(N, K)
    if dst is None:
        dst = torch.empty(nbytes, dtype=torch.uint8, device=w.device)
    st = lib().q2_0_split_layout(_dev(w, "w", torch.uint8, packed_bytes(N, K)),
                                 _dev(dst, "dst", torch.uint8, nbytes), N, K, _stream(stream))
    _check("q2_0_split_layout", st)
    return dst


def q2_0_join_layout(src: torch.Tensor, N: int, K: int, w: torch.Tensor | None = None,
                     stream=None) -> torch.Tensor:
    """Split layout -> 18-byte blocks."""
    if w is None:
        w = torch.empty(packed_bytes(N, K), dtype=torch.uint8, device=src.device)
    st = lib().q2_0_join_layout(_dev(src, "src", torch.uint8, q2_0_split_bytes(N, K)),
                                _dev(w, "w", torch.uint8, packed_bytes(N, K)), N, K, _stream(stream))
    _check("q2_0_join_layout", st)
    return w


def q2_0_mul_mat_vec_split(w: torch.Tensor, x: torch.Tensor, N: int, K: int, ncols: int = 1,
                           y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[c][n] = sum_k W[n][k] x[c][k] with W in the split layout."""
    if y is None:
        y = torch.empty((ncols, N), dtype=torch.float32, device=x.device)
    st = lib().q2_0_mul_mat_vec_split(_dev(w, "w", torch.uint8, q2_0_split_bytes(N, K)),
                                      _dev(x, "x", torch.float32, ncols * K),
                                      _dev(y, "y", torch.float32, ncols * N), N, K, ncols,
                                      _stream(stream))
    _check("q2_0_mul_mat_vec_split", st)
    return y


def q2_0_quantize_ref(src: torch.Tensor, nrows: int, K: int, dst: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
    """Reference quantizer: f32 [nrows][K] -> packed uint8 blocks."""
    if dst is None:
        dst = torch.empty(packed_bytes(nrows, K), dtype=torch.uint8, device=src.device)
    st = lib().q2_0_quantize_ref(_dev(src, "src", torch.float32, nrows * K),
                                 _dev(dst, "dst", torch.uint8, packed_bytes(nrows, K)), nrows, K,
                                 _stream(stream))
    _check("q2_0_quantize_ref", st)
    return dst


def q2_0_test_inject_stall(stage: int, wait_limit_ns: int) -> None:
    """Test only: the next fp4 mat-vec launch on the current device stalls before
    pipeline stage `stage` and its waits give up after wait_limit_ns."""
    _check("q2_0_test_inject_stall", lib().q2_0_test_inject_stall(int(stage), int(wait_limit_ns)))


def q2_0_get_error(stream=None):
    """(code, info): synchronises the stream, reads and clears the device error word."""
    info = ctypes.c_int64(0)
    code = lib().q2_0_get_error(_stream(stream), ctypes.byref(info))
    if code < 0:
        raise Q2Error("q2_0_get_error", Q2_0_ECUDA)
    return code, info.value


# ---- group-128 packing (34-byte blocks of 128 weights) ---------------------------
def packed_bytes_g128(N: int, K: int) -> int:
    return N * (K // 128) * 34


def q2_0_g128_to_g64(src: torch.Tensor, nrows: int, K: int, dst: torch.Tensor | None = None,
                    stream=None) -> torch.Tensor:
    """Exact repack of a group-128 matrix into the 64-weight layout (uint8)."""
    if dst is None:
        dst = torch.empty(packed_bytes(nrows, K), dtype=torch.uint8, device=src.device)
    st = lib().q2_0_g128_to_g64(_dev(src, "src", torch.uint8, packed_bytes_g128(nrows, K)),
                               _dev(dst, "dst", torch.uint8, packed_bytes(nrows, K)), nrows, K,
                               _stream(stream))
    _check("q2_0_g128_to_g64", st)
    return dst


def q2_0_g128_get_rows(table: torch.Tensor, n_rows: int, K: int, ids: torch.Tensor,
                      out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    n_ids = ids.numel()
    if out is None:
        out = torch.empty((n_ids, K), dtype=torch.float32, device=ids.device)
    if n_ids == 0:
        return out
    st = lib().q2_0_g128_get_rows(_dev(table, "table", torch.uint8, packed_bytes_g128(n_rows, K)),
                                 n_rows, K, _dev(ids, "ids", torch.int32, n_ids), n_ids,
                                 _dev(out, "out", torch.float32, n_ids * K), _stream(stream))
    _check("q2_0_g128_get_rows", st)
    return out


def q2_0_g128_mul_mat_vec(w: torch.Tensor, x: torch.Tensor, N: int, K: int,
                         ncols: int | None = None, y: torch.Tensor | None = None,
                         stream=None) -> torch.Tensor:
    ncols = x.shape[0] if (ncols is None and x.dim() == 2) else (ncols or 1)
    if y is None:
        y = torch.empty((ncols, N), dtype=torch.float32, device=x.device)
    st = lib().q2_0_g128_mul_mat_vec(_dev(w, "w", torch.uint8, packed_bytes_g128(N, K)),
                                    _dev(x, "x", torch.float32, ncols * K),
                                    _dev(y, "y", torch.float32, ncols * N), N, K, ncols,
                                    _stream(stream))
    _check("q2_0_g128_mul_mat_vec", st)
    return y
