"""Failure detection on the GPU without a fault: every pipeline wait of the
tensor-core kernels is bounded. The test hook q2_0_test_inject_stall makes the
next fp4 mat-vec launch stop feeding its pipeline at a chosen stage with a
2 ms wait limit; the waits on that stage run out, the kernel records
Q2_0_DEVERR_TIMEOUT (info 111, the wait for a stage's copies), drains its own
copies, frees its tensor memory and returns. Nothing traps, faults or waits
without a limit, and the next normal call on the same context is correct."""
import time

import numpy as np
import pytest
import torch

import bit_ternary_matmul_gb300 as q
import oracle
import synth

pytestmark = pytest.mark.gpu

TAG_STAGE_COPIES = 111


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    q.build()
    oracle.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    assert q.q2_0_device_check() == q.Q2_0_OK
    code, _ = q.q2_0_get_error()
    assert code == 0
    return d


def _case(dev, seed, N, K, ncols=1):
    g = synth.rng(seed, N, K)
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    x = synth.activations(g, ncols, K)
    return w, x, torch.from_numpy(w).to(dev), torch.from_numpy(x).to(dev)


@pytest.mark.parametrize("stage,ncols", [(0, 1), (3, 1), (0, 2), (5, 2)])
def test_stalled_pipeline_times_out_and_recovers(dev, stage, ncols):
    """ncols 1 and 2 (the two-column fp4 kernel, whose epilogue warps also hand
    their tile sums over through bounded waits)."""
    N, K = 1000, 4096
    w, x, wd, xd = _case(dev, 6101, N, K, ncols)
    yo, acc = oracle.matmul(w, N, K, x)
    q.q2_0_test_inject_stall(stage, 2_000_000)          # 2 ms
    t0 = time.perf_counter()
    q.q2_0_mul_mat_vec(wd, xd, N, K, ncols)
    code, info = q.q2_0_get_error()                     # synchronises
    elapsed = time.perf_counter() - t0
    assert code == q.Q2_0_DEVERR_TIMEOUT and info == TAG_STAGE_COPIES, (code, info)
    assert elapsed < 5.0
    # the next calls run normally on the same context
    for _ in range(2):
        y = q.q2_0_mul_mat_vec(wd, xd, N, K, ncols).cpu().numpy()
        assert oracle.within_tolerance(y, yo, acc, 1e-5, 1e-7).all()
        code, info = q.q2_0_get_error()
        assert code == 0, (code, info)


def test_stall_in_a_plan(dev):
    """A plan's launch stalls the same way; the plan then runs normally."""
    ents, host = [], []
    for i, (N, K) in enumerate([(300, 2048), (1000, 6144)]):
        w, x, wd, xd = _case(dev, 6102 + i, N, K)
        ents.append((wd, xd, torch.empty((1, N), device=dev), N, K))
        host.append((w, x))
    plan = q.MvPlan(ents, 1)
    q.q2_0_test_inject_stall(1, 2_000_000)
    plan.execute()
    code, info = q.q2_0_get_error()
    assert code == q.Q2_0_DEVERR_TIMEOUT and info == TAG_STAGE_COPIES, (code, info)
    plan.execute()
    torch.cuda.synchronize()
    for (w, x), (_, _, yd, N, K) in zip(host, ents):
        yo, acc = oracle.matmul(w, N, K, x)
        assert oracle.within_tolerance(yd.cpu().numpy(), yo, acc, 1e-5, 1e-7).all()
    plan.close()
    code, _ = q.q2_0_get_error()
    assert code == 0


def test_inject_stall_argument_checks(dev):
    L = q.lib()
    assert L.q2_0_test_inject_stall(-1, 1000) == q.Q2_0_EINVAL
    assert L.q2_0_test_inject_stall(0, 0) == q.Q2_0_EINVAL
    assert L.q2_0_test_inject_stall(0, 20_000_000_000) == q.Q2_0_EINVAL
