"""q2_0_mul_mat_vec_noalloc: the decode mat-vec for callers that cannot allocate
device memory when they call it (an allocator that owns all of HBM, a decode
loop that must not call an allocator). Its scratch is a static device array
inside the library; these checks call it through the C ABI and compare it with
q2_0_mul_mat_vec on the same inputs, twice in a row with different shapes so
that the second call runs on scratch the first one left behind."""
import ctypes

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


def test_noalloc_matches_mul_mat_vec_twice(dev):
    # first call: large scratch; second call: smaller one over the first's leftovers
    for seed, (N, K, ncols) in [(1, (300, 6144, 4)), (2, (129, 1024, 1)), (3, (200, 2048, 8))]:
        w, x, wd, xd = _case(9100 + seed, N, K, ncols, dev)
        y_ref = q.q2_0_mul_mat_vec(wd, xd, N, K, ncols)
        y = torch.full((ncols, N), float("nan"), device=dev)
        st = q.lib().q2_0_mul_mat_vec_noalloc(ctypes.c_void_p(wd.data_ptr()),
                                             ctypes.c_void_p(xd.data_ptr()),
                                             ctypes.c_void_p(y.data_ptr()), N, K, ncols,
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == q.Q2_0_OK
        got, ref = y.cpu().numpy(), y_ref.cpu().numpy()
        _, acc = oracle.matmul(w, N, K, x)
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got.astype(np.float64) - ref) <= REL * acc + ABS), (N, K, ncols)
    code, info = q.q2_0_get_error()
    assert code == 0, (code, info)


def test_noalloc_python_wrapper_and_limits(dev):
    w, x, wd, xd = _case(9200, 64, 512, 2, dev)
    y = q.q2_0_mul_mat_vec_noalloc(wd, xd, 64, 512, 2)
    yo, acc = oracle.matmul(w, 64, 512, x)
    assert np.all(np.abs(y.cpu().numpy().astype(np.float64) - yo) <= REL * acc + ABS)
    # a call that needs more scratch than the static array is refused, nothing launched
    big_k = 64 * 1024
    assert q.q2_0_mul_mat_vec_workspace_size(big_k, 8) > q.Q2_0_NOALLOC_SCRATCH_BYTES
    p = ctypes.c_void_p(wd.data_ptr())
    assert q.lib().q2_0_mul_mat_vec_noalloc(p, p, p, 1, big_k, 8, None) == q.Q2_0_ENOSPACE
    assert q.lib().q2_0_mul_mat_vec_noalloc(p, p, p, 1, 100, 1, None) == q.Q2_0_EINVAL
