"""Host-side checks of the C-ABI library: it builds for sm_103a, loads, exports
every symbol include/q2_0.h declares, and rejects bad arguments before touching
a GPU. No compute call is made here."""
import ctypes
import os
import re

import pytest

import bit_ternary_matmul_gb300 as q

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "q2_0.h")


@pytest.fixture(scope="module")
def L():
    q.build()
    return q.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(q2_0_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(L):
    names = _declared()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n
    assert sorted(q.EXPORTS) == names


def test_version_and_no_device(L):
    assert "sm_103a" in q.q2_0_version()
    import torch
    if not torch.cuda.is_available():
        assert q.q2_0_device_check() in (q.Q2_0_ECUDA, q.Q2_0_EUNSUPPORTED)


def test_argument_validation_without_gpu(L):
    p = ctypes.c_void_p(0x1000)  # never dereferenced: validation fails first
    null = ctypes.c_void_p(0)
    EINVAL = q.Q2_0_EINVAL
    # mat-vec: null pointers, K not a multiple of 64, ncols out of range, N < 1
    assert L.q2_0_mul_mat_vec(null, p, p, 4, 64, 1, null) == EINVAL
    assert L.q2_0_mul_mat_vec(p, p, p, 4, 100, 1, null) == EINVAL
    assert L.q2_0_mul_mat_vec(p, p, p, 4, 64, 0, null) == EINVAL
    assert L.q2_0_mul_mat_vec(p, p, p, 4, 64, 9, null) == EINVAL
    assert L.q2_0_mul_mat_vec(p, p, p, 0, 64, 1, null) == EINVAL
    assert L.q2_0_mul_mat_vec_f16(null, p, p, 4, 64, 1, null) == EINVAL
    assert L.q2_0_mul_mat_vec_f16(p, p, p, 4, 100, 1, null) == EINVAL
    assert L.q2_0_mul_mat_vec_f16(p, p, p, 4, 64, 9, null) == EINVAL
    assert L.q2_0_mul_mat_f16(p, p, p, 4, 65, 4, null, 0, null) == EINVAL
    assert L.q2_0_mul_mat_f16(p, null, p, 4, 64, 4, null, 0, null) == EINVAL
    # group-128: K must be a multiple of 128
    assert L.q2_0_g128_to_g64(p, p, 4, 64, null) == EINVAL
    assert L.q2_0_g128_to_g64(null, p, 4, 128, null) == EINVAL
    assert L.q2_0_g128_get_rows(p, 4, 192, p, 3, p, null) == EINVAL
    assert L.q2_0_g128_get_rows(p, 4, 128, p, 0, p, null) == q.Q2_0_OK
    assert L.q2_0_g128_mul_mat_vec(p, p, p, 4, 128, 9, null) == EINVAL
    assert L.q2_0_g128_mul_mat_vec(p, p, p, 0, 128, 1, null) == EINVAL
    # expert mat-vec: shapes, n_x, limits, workspace; n_tokens == 0 is a no-op
    ids = ctypes.c_void_p(0x2000)
    assert L.q2_0_mul_mat_id(p, 4, 8, 512, p, 1, ids, 2, 0, p, null, 0, null) == q.Q2_0_OK
    assert L.q2_0_mul_mat_id(p, 4, 8, 500, p, 1, ids, 2, 1, p, null, 0, null) == EINVAL  # K % 64
    assert L.q2_0_mul_mat_id(p, 0, 8, 512, p, 1, ids, 2, 1, p, null, 0, null) == EINVAL  # no expert
    assert L.q2_0_mul_mat_id(p, 4, 8, 512, p, 3, ids, 2, 1, p, null, 0, null) == EINVAL  # n_x
    assert L.q2_0_mul_mat_id(p, 4, 8, 512, p, 1, null, 2, 1, p, null, 0, null) == EINVAL  # ids
    assert L.q2_0_mul_mat_id(p, 1 << 20, 1 << 12, 512, p, 1, ids, 2, 1, p, null, 0,
                             null) == EINVAL  # n_expert * N >= 2^31
    assert L.q2_0_mul_mat_id(p, 4, 8, 512, p, 1, ids, 2, 40000, p, null, 0, null) == EINVAL
    need = L.q2_0_mul_mat_id_workspace_size(512, 3, 2)
    assert need == 2 * 3 * L.q2_0_mul_mat_vec_workspace_size(512, 1)
    assert L.q2_0_mul_mat_id_workspace_size(576, 3, 2) == 0  # off the fast path: no scratch
    assert L.q2_0_mul_mat_id(p, 4, 8, 512, p, 2, ids, 2, 3, p, ctypes.c_void_p(0x100000), need - 1,
                             null) == EINVAL
    assert L.q2_0_mul_mat_id(p, 4, 8, 512, p, 2, ids, 2, 3, p, ctypes.c_void_p(0x100010), need,
                             null) == EINVAL  # workspace not 256-byte aligned
    # split layout: sizes and argument checks
    assert L.q2_0_split_bytes(1, 128) == 512
    assert L.q2_0_split_bytes(300, 1024) == 76800 + 9728
    assert L.q2_0_split_bytes(0, 128) == 0 and L.q2_0_split_bytes(4, 100) == 0
    assert L.q2_0_split_layout(null, p, 4, 64, null) == EINVAL
    assert L.q2_0_join_layout(p, p, 4, 96, null) == EINVAL
    assert L.q2_0_mul_mat_vec_split(p, p, p, 4, 64, 9, null) == EINVAL
    assert L.q2_0_mul_mat_vec_split(p, p, p, 0, 64, 1, null) == EINVAL
    # mat-vec with workspace: too small, misaligned
    need = L.q2_0_mul_mat_vec_workspace_size(512, 1)
    assert need > 0 and need % 256 == 0
    assert L.q2_0_mul_mat_vec_ws(p, p, p, 4, 512, 1, p, need - 1, null) == EINVAL
    assert L.q2_0_mul_mat_vec_ws(p, p, p, 4, 512, 1, ctypes.c_void_p(0x1010), need, null) == EINVAL
    assert L.q2_0_mul_mat_vec_workspace_size(100, 1) == 0
    assert L.q2_0_mul_mat_vec_workspace_size(512, 9) == 0
    # the allocation-free entry's documented K limits (largest K that fits, then the next
    # multiple of 512) against its scratch size
    cap = q.Q2_0_NOALLOC_SCRATCH_BYTES
    for ncols, k_max in [(1, 126976), (2, 63488), (3, 63488), (4, 31744), (6, 31744), (7, 21504), (8, 21504)]:
        assert L.q2_0_mul_mat_vec_workspace_size(k_max, ncols) <= cap, ncols
        assert L.q2_0_mul_mat_vec_workspace_size(k_max + 512, ncols) > cap, ncols
    # GEMM: bad precision, bad K, small workspace
    assert L.q2_0_mul_mat(p, p, p, 4, 64, 4, 7, null, 0, null) == EINVAL
    assert L.q2_0_mul_mat(p, p, p, 4, 65, 4, 0, null, 0, null) == EINVAL
    ws = L.q2_0_mul_mat_workspace_size(4, 4, 512, 0)
    assert ws >= 2 * 4 * 512 * 2
    # F16 needs no lo half of X; both hold the same stream-K counters and partial tiles
    ws16 = L.q2_0_mul_mat_workspace_size(4, 4, 512, 1)
    assert ws16 % 256 == 0 and ws16 + 4 * 512 * 2 <= ws
    assert L.q2_0_mul_mat(p, p, p, 4, 512, 4, 0, ctypes.c_void_p(0x100000), ws - 1, null) == EINVAL
    # get_rows: n_ids == 0 is a no-op, negative is invalid
    assert L.q2_0_get_rows(p, 4, 64, p, 0, p, null) == q.Q2_0_OK
    assert L.q2_0_get_rows(p, 4, 64, p, -1, p, null) == EINVAL
    assert L.q2_0_get_rows(null, 4, 64, p, 3, p, null) == EINVAL
    # quantize
    assert L.q2_0_quantize_ref(p, p, 0, 64, null) == EINVAL
    assert L.q2_0_quantize_ref(p, p, 2, 96, null) == EINVAL
    # plans
    h = ctypes.c_void_p()
    assert L.q2_0_mv_plan_create(None, 1, 1, ctypes.byref(h)) == EINVAL
    assert L.q2_0_mv_plan_execute(null, null) == EINVAL
    assert L.q2_0_mv_plan_launches(null) == 0
    L.q2_0_mv_plan_destroy(null)
    # grouped GEMM plans: null arguments, no descriptors, bad precision, and a
    # descriptor with a bad K / M / null pointer are refused before any device call
    assert L.q2_0_mm_plan_create(None, 1, 0, ctypes.byref(h)) == EINVAL
    d = q._MmDesc(0x100000, 0x100000, 0x100000, 4, 512, 4)
    arr = (q._MmDesc * 1)(d)
    assert L.q2_0_mm_plan_create(arr, 1, 0, None) == EINVAL
    assert L.q2_0_mm_plan_create(arr, 0, 0, ctypes.byref(h)) == EINVAL
    assert L.q2_0_mm_plan_create(arr, 1, 2, ctypes.byref(h)) == EINVAL
    for bad in (q._MmDesc(0x100000, 0x100000, 0x100000, 4, 100, 4),
                q._MmDesc(0x100000, 0x100000, 0x100000, 4, 512, 0),
                q._MmDesc(0x100000, 0x100000, 0x100000, 0, 512, 4),
                q._MmDesc(0x100000, None, 0x100000, 4, 512, 4)):
        two = (q._MmDesc * 2)(d, bad)
        assert L.q2_0_mm_plan_create(two, 2, 0, ctypes.byref(h)) == EINVAL
        assert not h.value
    assert L.q2_0_mm_plan_execute(null, null) == EINVAL
    assert L.q2_0_mm_plan_launches(null) == 0
    L.q2_0_mm_plan_destroy(null)
