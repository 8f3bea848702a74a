"""q2_0_mul_mat_vec_noalloc: the decode mat-vec for callers that cannot allocate
device memory when they call it (an allocator that owns all of HBM, a decode
loop that must not call an allocator). Its scratch is a static device array
inside the library; these checks call it through the C ABI and compare it with
q2_0_mul_mat_vec and with the oracle on the same inputs, twice in a row with
different shapes so that the second call runs on scratch the first one left
behind, and check that it takes nothing from the device's memory pool.

This file is collected last, so that a run stopping at the first failure has
run every other test before it."""
import ctypes
import glob
import os

import numpy as np
import pytest
import torch

import bit_ternary_matmul_gb300 as q
import oracle
import synth

pytestmark = pytest.mark.gpu

REL, ABS = 1e-5, 1e-7   # the mat-vec tolerance used by the parity tests


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    q.build()
    oracle.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    assert q.q2_0_device_check() == q.Q2_0_OK
    return d


def _case(seed, N, K, ncols, dev):
    g = synth.rng(seed, N, K, ncols)
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    x = synth.activations(g, ncols, K, 0.001, 30.0)
    return w, x, torch.from_numpy(w).to(dev), torch.from_numpy(x).to(dev)


def _noalloc(wd, xd, y, N, K, ncols):
    return q.lib().q2_0_mul_mat_vec_noalloc(
        ctypes.c_void_p(wd.data_ptr()), ctypes.c_void_p(xd.data_ptr()),
        ctypes.c_void_p(y.data_ptr()), N, K, ncols,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _within(got, ref, acc):
    return np.all(np.isfinite(got)) and np.all(np.abs(got.astype(np.float64) - ref) <= REL * acc + ABS)


def test_noalloc_matches_mul_mat_vec_and_oracle_twice(dev):
    # first call: large scratch; the later calls: smaller ones over the leftovers
    for seed, (N, K, ncols) in [(1, (300, 6144, 4)), (2, (129, 1024, 1)), (3, (200, 2048, 8))]:
        w, x, wd, xd = _case(9100 + seed, N, K, ncols, dev)
        y_ref = q.q2_0_mul_mat_vec(wd, xd, N, K, ncols)
        y = torch.full((ncols, N), float("nan"), device=dev)
        assert _noalloc(wd, xd, y, N, K, ncols) == q.Q2_0_OK
        got, ref = y.cpu().numpy(), y_ref.cpu().numpy()
        yo, acc = oracle.matmul(w, N, K, x)
        assert _within(got, yo, acc), ("vs oracle", N, K, ncols)
        assert _within(got, ref.astype(np.float64), acc), ("vs q2_0_mul_mat_vec", N, K, ncols)
    code, info = q.q2_0_get_error()
    assert code == 0, (code, info)


def test_noalloc_python_wrapper_and_limits(dev):
    w, x, wd, xd = _case(9200, 64, 512, 2, dev)
    y = q.q2_0_mul_mat_vec_noalloc(wd, xd, 64, 512, 2)
    yo, acc = oracle.matmul(w, 64, 512, x)
    assert _within(y.cpu().numpy(), yo, acc)
    # a tensor-core call that needs more scratch than the static array is
    # refused, nothing launched
    big_k = 64 * 1024
    assert q.q2_0_mul_mat_vec_workspace_size(big_k, 8) > q.Q2_0_NOALLOC_SCRATCH_BYTES
    p = ctypes.c_void_p(wd.data_ptr())
    assert q.lib().q2_0_mul_mat_vec_noalloc(p, p, p, 1, big_k, 8, None) == q.Q2_0_ENOSPACE
    assert q.lib().q2_0_mul_mat_vec_noalloc(p, p, p, 1, 100, 1, None) == q.Q2_0_EINVAL


def _cudart():
    """The CUDA runtime already loaded by torch (or the toolkit's), or None."""
    cands = ["libcudart.so", "libcudart.so.13"]
    tl = os.path.join(os.path.dirname(torch.__file__), "lib")
    cands += sorted(glob.glob(os.path.join(tl, "libcudart*.so*")))
    cands += sorted(glob.glob("/usr/local/cuda/lib64/libcudart.so*"))
    for c in cands:
        try:
            return ctypes.CDLL(c)
        except OSError:
            continue
    return None


def test_noalloc_takes_nothing_from_the_memory_pool(dev):
    """The high-water mark of the device's default memory pool (where
    q2_0_mul_mat_vec takes its scratch) does not move during a noalloc call;
    the same probe around q2_0_mul_mat_vec shows that it would see one."""
    rt = _cudart()
    if rt is None:
        pytest.skip("no CUDA runtime library to read the memory pool")
    used_high = 8   # cudaMemPoolAttrUsedMemHigh
    pool = ctypes.c_void_p()
    assert rt.cudaDeviceGetDefaultMemPool(ctypes.byref(pool), 0) == 0

    def high_after(fn):
        torch.cuda.synchronize()
        zero = ctypes.c_uint64(0)
        assert rt.cudaMemPoolSetAttribute(pool, used_high, ctypes.byref(zero)) == 0
        fn()
        torch.cuda.synchronize()
        v = ctypes.c_uint64(0)
        assert rt.cudaMemPoolGetAttribute(pool, used_high, ctypes.byref(v)) == 0
        return v.value

    N, K, ncols = 256, 4096, 2
    _, _, wd, xd = _case(9300, N, K, ncols, dev)
    y = torch.empty((ncols, N), device=dev)
    base = high_after(lambda: None)
    st = []
    with_noalloc = high_after(lambda: st.append(_noalloc(wd, xd, y, N, K, ncols)))
    assert st == [q.Q2_0_OK]
    with_pool = high_after(lambda: q.q2_0_mul_mat_vec(wd, xd, N, K, ncols, y=y))
    assert with_noalloc == base
    assert with_pool >= base + q.q2_0_mul_mat_vec_workspace_size(K, ncols)
