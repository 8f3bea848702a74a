"""GPU parity: every C-ABI entry point against the CPU oracle on the same seeded
inputs. Bit-exact for get_rows and the quantizer; for the matmuls
|gpu - oracle| <= 1e-5 * sum|w*x| + 1e-7 (split / mat-vec paths) or
<= 4e-3 * sum|w*x| (single-fp16 GEMM path), with the oracle's fp64 values."""
import numpy as np
import pytest
import torch

import bit_ternary_matmul_gb300 as q
import oracle
import synth
import wide_range as wr

pytestmark = pytest.mark.gpu

TOL_SPLIT = (1e-5, 1e-7)
TOL_F16 = (4e-3, 0.0)


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


def _to(dev, a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dev)


def _assert_close(gpu, y, acc, tol, what):
    ok = oracle.within_tolerance(gpu, y, acc, tol[0], tol[1])
    if not ok.all():
        bad = np.argwhere(~ok)[:5]
        msgs = [f"{tuple(i)}: gpu={gpu[tuple(i)]!r} ref={y[tuple(i)]!r} acc={acc[tuple(i)]!r}"
                for i in bad]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance\n" +
                             "\n".join(msgs))


def _assert_same_blocks(got, ref, what):
    if np.array_equal(got, ref):
        return
    g = got.reshape(-1, 18)
    r = ref.reshape(-1, 18)
    bad = np.nonzero(np.any(g != r, axis=1))[0]
    b = bad[0]
    raise AssertionError(f"{what}: {bad.size} of {r.shape[0]} blocks differ; first block {b}: "
                         f"gpu={g[b].tobytes().hex()} ref={r[b].tobytes().hex()}; "
                         f"d differs in {int(np.sum(np.any(g[bad, :2] != r[bad, :2], axis=1)))}")


def _no_device_error():
    code, info = q.q2_0_get_error()
    assert code == 0, (code, info)


# ---------------------------------------------------------------------------
# get_rows
# ---------------------------------------------------------------------------
def _edge_table(g, n_rows, K, edge_rows):
    t = synth.packed_matrix(g, n_rows, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    edges = synth.edge_blocks()
    nb = K // 64
    tv = t.reshape(n_rows, nb, 18)
    for i, r in enumerate(edge_rows):
        # whole row of one edge pattern, then every pattern in turn
        tv[r, :, :] = edges[i % len(edges)]
        for j in range(min(nb, len(edges))):
            tv[r, j] = edges[(i + j) % len(edges)]
    return t


def test_get_rows_embedding_table(dev):
    """151936 x 4096 table, 512 seeded ids with repeats; ids[0..8] hit edge rows."""
    g = synth.rng(1005, 1)
    n_rows, K = 151936, 4096
    head = np.array([7, 151935, 0, 77777, 4242, 123, 99999, 31, 5], dtype=np.int32)
    t = _edge_table(g, n_rows, K, head)
    ids = synth.token_ids(g, 512, n_rows, 0.05, head)
    out = q.q2_0_get_rows(_to(dev, t), n_rows, K, _to(dev, ids)).cpu().numpy()
    ref, bad = oracle.get_rows(t, n_rows, K, ids)
    assert bad == 0
    assert np.array_equal(out.view(np.uint32), ref.view(np.uint32))
    _no_device_error()


@pytest.mark.parametrize("K,offset", [(64, 0), (576, 0), (1024, 1), (2048, 4)])
def test_get_rows_shapes_and_alignment(dev, K, offset):
    g = synth.rng(77, K, offset)
    n_rows = 37
    t = _edge_table(g, n_rows, K, [0, 5, 36])
    ids = np.array([0, 36, 5, 5, 1, 0, 20], dtype=np.int32)
    # packed table at a byte offset (any alignment), output at a float offset
    tb = torch.zeros(t.size + 16, dtype=torch.uint8, device=dev)
    tb[offset:offset + t.size] = _to(dev, t)
    ob = torch.full((ids.size * K + 1,), float("nan"), device=dev)
    out = ob[1:] if offset else ob[:-1]
    q.q2_0_get_rows(tb[offset:offset + t.size], n_rows, K, _to(dev, ids), out=out)
    ref, _ = oracle.get_rows(t, n_rows, K, ids)
    got = out.cpu().numpy().reshape(ids.size, K)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    # the guard element next to the output is untouched
    guard = ob[0] if offset else ob[-1]
    assert torch.isnan(guard)
    _no_device_error()


def test_get_rows_bad_ids_recorded(dev):
    g = synth.rng(78)
    n_rows, K = 10, 128
    t = synth.packed_matrix(g, n_rows, K, 0.1, 0.2)
    ids = np.array([3, 10, 9, -1], dtype=np.int32)
    out = torch.full((4, K), 7.0, device=dev)
    q.q2_0_get_rows(_to(dev, t), n_rows, K, _to(dev, ids), out=out)
    code, info = q.q2_0_get_error()
    assert code == q.Q2_0_DEVERR_BAD_ID and info in (1, 3)
    o = out.cpu().numpy()
    ref, bad = oracle.get_rows(t, n_rows, K, ids)
    assert bad == 2
    assert np.array_equal(o[0].view(np.uint32), ref[0].view(np.uint32))
    assert np.array_equal(o[2].view(np.uint32), ref[2].view(np.uint32))
    assert np.all(o[1] == 7.0) and np.all(o[3] == 7.0)   # rows of bad ids untouched
    _no_device_error()


# ---------------------------------------------------------------------------
# reference quantizer
# ---------------------------------------------------------------------------
def test_quantize_random_blocks_bitexact(dev):
    """>= 14,000 random blocks (normal, uniform, heavy-tailed, ties, zeros), bit-exact."""
    g = synth.rng(31337)
    rows = []
    rows.append(g.standard_normal((4000, 64)))
    rows.append(g.uniform(-1, 1, (4000, 64)))
    rows.append(g.standard_cauchy((4000, 64)) * 1e-3)
    tie = g.uniform(-1, 1, (2000, 64))
    amax = np.max(np.abs(tie), axis=1, keepdims=True)
    sel = g.integers(0, 64, (2000, 8))
    for r in range(2000):
        tie[r, sel[r, :4]] = amax[r] / 2
        tie[r, sel[r, 4:]] = -amax[r] / 2
    rows.append(tie)
    rows.append(np.zeros((50, 64)))
    rows.append(g.standard_normal((100, 64)) * 1e-7)    # scale rounds to subnormal fp16
    rows.append(g.standard_normal((100, 64)) * 1e4)     # scale near the fp16 top
    src = np.concatenate(rows).astype(np.float32)
    n = src.shape[0]
    assert n >= 14000
    got = q.q2_0_quantize_ref(_to(dev, src), n, 64).cpu().numpy()
    ref = oracle.quantize(src, n, 64)
    _assert_same_blocks(got, ref, "quantize random blocks")
    _no_device_error()


def test_quantize_rows_misaligned_dst(dev):
    g = synth.rng(31338)
    src = g.standard_normal((9, 576)).astype(np.float32)
    nbytes = 9 * 9 * 18
    buf = torch.zeros(nbytes + 3, dtype=torch.uint8, device=dev)
    q.q2_0_quantize_ref(_to(dev, src), 9, 576, dst=buf[1:1 + nbytes])
    _assert_same_blocks(buf[1:1 + nbytes].cpu().numpy(), oracle.quantize(src, 9, 576),
                        "quantize misaligned")
    assert int(buf[0]) == 0 and int(buf[-1]) == 0
    _no_device_error()


# ---------------------------------------------------------------------------
# decode mat-vec
# ---------------------------------------------------------------------------
MV_CASES = [
    (2048, 2048, 1),   # the 2048 x 2048 single-matrix workload
    (1, 512, 1), (3, 1024, 2), (127, 512, 3), (300, 2048, 4), (257, 1536, 5),
    (64, 512, 8), (1000, 6144, 7), (513, 4096, 6),
    (300, 2048, 2), (1000, 6144, 2), (129, 512, 2), (257, 4608, 2),   # fp4 path, two columns
    (33, 576, 1), (5, 64, 3), (130, 1088, 8),   # K % 512 != 0: CUDA-core path
]


@pytest.mark.parametrize("N,K,ncols", MV_CASES)
def test_matvec_parity(dev, N, K, ncols):
    g = synth.rng(2001, N, K, ncols)
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    x = synth.activations(g, ncols, K, 0.001, 30.0)
    y = q.q2_0_mul_mat_vec(_to(dev, w), _to(dev, x), N, K, ncols).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, f"mat-vec {N}x{K} ncols={ncols}")
    _no_device_error()


@pytest.mark.parametrize("offset", [1, 2, 8])
def test_matvec_unaligned_weights(dev, offset):
    g = synth.rng(2002, offset)
    N, K, ncols = 70, 1024, 2
    w = synth.packed_matrix(g, N, K, 0.01, 0.05, 0.01)
    x = synth.activations(g, ncols, K)
    buf = torch.zeros(w.size + 16, dtype=torch.uint8, device=dev)
    buf[offset:offset + w.size] = _to(dev, w)
    y = q.q2_0_mul_mat_vec(buf[offset:offset + w.size], _to(dev, x), N, K, ncols).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, f"mat-vec offset {offset}")


@pytest.mark.parametrize("kind", ["tiny", "huge", "zero_col", "outliers", "edge_blocks", "code3"])
def test_matvec_value_ranges(dev, kind):
    g = synth.rng(2003, hash(kind) % 1000)
    N, K, ncols = 260, 2048, 4
    w = synth.packed_matrix(g, N, K, 0.005, 0.05, 0.01)
    x = synth.activations(g, ncols, K)
    if kind == "tiny":
        x *= np.float32(1e-6)
    elif kind == "huge":
        x *= np.float32(1e3)
    elif kind == "zero_col":
        x[1] = 0
        x[3, ::7] = 0
    elif kind == "outliers":
        x = synth.activations(g, ncols, K, 0.01, 30.0)
    elif kind == "edge_blocks":
        edges = synth.edge_blocks()
        wv = w.reshape(N, K // 64, 18)
        # finite edge blocks only (the 65504 scale keeps |2d| finite in f32)
        for r in range(0, N, 3):
            wv[r, r % (K // 64)] = edges[r % len(edges)]
    elif kind == "code3":
        w = synth.packed_matrix(g, N, K, 0.005, 0.05, 0.3)
    y = q.q2_0_mul_mat_vec(_to(dev, w), _to(dev, x), N, K, ncols).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, f"mat-vec {kind}")


def test_matvec_ws_entry_point(dev):
    g = synth.rng(2004)
    N, K, ncols = 400, 3072, 3
    w = synth.packed_matrix(g, N, K, 0.01, 0.05)
    x = synth.activations(g, ncols, K)
    need = q.q2_0_mul_mat_vec_workspace_size(K, ncols)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    y = q.q2_0_mul_mat_vec_ws(_to(dev, w), _to(dev, x), N, K, ncols, ws).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, "mat-vec ws")


@pytest.mark.parametrize("ncols", [1, 2, 4, 8])
def test_plan_mixed_shapes(dev, ncols):
    g = synth.rng(2005, ncols)
    shapes = [(256, 512), (1000, 2048), (1, 1024), (777, 1536), (96, 576), (2048, 6144), (33, 64)]
    ents, host = [], []
    for (N, K) in shapes:
        w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
        x = synth.activations(g, ncols, K)
        yd = torch.full((ncols, N), float("nan"), device=dev)
        ents.append((_to(dev, w), _to(dev, x), yd, N, K))
        host.append((w, x))
    plan = q.MvPlan(ents, ncols)
    assert plan.launches == 2 + 2   # prep + tensor-core kernel, two CUDA-core matrices
    for rep in range(2):
        plan.execute()
        torch.cuda.synchronize()
        for (w, x), (_, _, yd, N, K) in zip(host, ents):
            yo, acc = oracle.matmul(w, N, K, x)
            _assert_close(yd.cpu().numpy(), yo, acc, TOL_SPLIT, f"plan {N}x{K} rep {rep}")
    plan.close()
    _no_device_error()


@pytest.mark.parametrize("seed,ncols", [(1, 1), (2, 1), (3, 3), (4, 8), (5, 2)])
def test_plan_random_shapes(dev, seed, ncols):
    """Seeded random plans: 24-40 matrices of 1-1500 rows (ragged last tiles,
    single-row matrices), K a multiple of 512 up to 6144 or off the tensor-core
    rules; every row checked, executed twice (the scratch and schedule reused)."""
    g = synth.rng(2010, seed)
    n_mat = int(g.integers(24, 41))
    ents, host = [], []
    for i in range(n_mat):
        N = int(g.integers(1, 1501)) if i % 5 else int(g.integers(1, 4))
        K = int(512 * g.integers(1, 13)) if i % 7 else int(64 * g.integers(1, 40))
        w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
        x = synth.activations(g, ncols, K, 0.001, 30.0)
        ents.append((_to(dev, w), _to(dev, x), torch.full((ncols, N), float("nan"), device=dev), N, K))
        host.append((w, x))
    plan = q.MvPlan(ents, ncols)
    for rep in range(2):
        plan.execute()
        torch.cuda.synchronize()
        for (w, x), (_, _, yd, N, K) in zip(host, ents):
            yo, acc = oracle.matmul(w, N, K, x)
            _assert_close(yd.cpu().numpy(), yo, acc, TOL_SPLIT, f"random plan {N}x{K} rep {rep}")
    plan.close()
    _no_device_error()


def _decode_step(dev, mats, seed, ncols):
    ents, host = [], []
    for idx, (layer, m) in enumerate(mats):
        g = synth.rng(seed, idx)
        w = synth.packed_matrix(g, m.N, m.K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
        x = synth.activations(g, ncols, m.K)
        ents.append((_to(dev, w), _to(dev, x), torch.empty((ncols, m.N), device=dev), m.N, m.K))
        host.append((w, x))
    return ents, host


@pytest.mark.parametrize("ncols", [1, 2, 3, 4, 8])
def test_plan_1p7b_decode_step_sampled(dev, ncols):
    """All 196 matrices of the 1.7B-class step; 24 sampled rows of each checked."""
    mats = synth.decode_step_1p7b()
    ents, host = _decode_step(dev, mats, 1002, ncols)
    plan = q.MvPlan(ents, ncols)
    plan.execute()
    torch.cuda.synchronize()
    g = synth.rng(1002, 999)
    for (w, x), (_, _, yd, N, K) in zip(host, ents):
        rows = np.unique(np.concatenate([[0, N - 1], g.integers(0, N, 22)]))
        yo, acc = oracle.matmul(w, N, K, x, rows=rows)
        _assert_close(yd[:, rows].cpu().numpy(), yo, acc, TOL_SPLIT, f"1.7B step {N}x{K}")
    plan.close()
    _no_device_error()


def test_plan_8b_decode_step_sampled(dev):
    """All 253 matrices of the 8B-class step with the 151936 x 4096 head, ncols = 1."""
    mats = synth.decode_step_8b(with_head=True)
    ents, host = _decode_step(dev, mats, 1003, 1)
    plan = q.MvPlan(ents, 1)
    plan.execute()
    torch.cuda.synchronize()
    g = synth.rng(1003, 999)
    for (w, x), (_, _, yd, N, K) in zip(host, ents):
        rows = np.unique(np.concatenate([[0, N - 1], g.integers(0, N, 14)]))
        yo, acc = oracle.matmul(w, N, K, x, rows=rows)
        _assert_close(yd[:, rows].cpu().numpy(), yo, acc, TOL_SPLIT, f"8B step {N}x{K}")
    plan.close()
    _no_device_error()


# ---------------------------------------------------------------------------
# prefill GEMM
# ---------------------------------------------------------------------------
GEMM_SMALL = [(128, 512, 128), (300, 1024, 70), (1, 512, 1), (200, 1536, 17), (130, 2048, 257),
              (256, 512, 300), (40, 576, 9), (17, 64, 5),
              # few output units over a long K: each unit split over many stream-K CTAs
              (300, 8192, 64), (513, 4096, 129)]


@pytest.mark.parametrize("prec", [q.Q2_0_PREC_F16_SPLIT, q.Q2_0_PREC_F16])
@pytest.mark.parametrize("N,K,M", GEMM_SMALL)
def test_gemm_parity_small(dev, N, K, M, prec):
    g = synth.rng(3001, N, K, M)
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    x = synth.activations(g, M, K, synth.PREFILL_OUTLIER_FRAC, synth.PREFILL_OUTLIER)
    y = q.q2_0_mul_mat(_to(dev, w), _to(dev, x), N, K, M, prec).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x)
    tol = TOL_SPLIT if prec == q.Q2_0_PREC_F16_SPLIT else TOL_F16
    _assert_close(y, yo, acc, tol, f"GEMM {N}x{K} M={M} prec={prec}")
    _no_device_error()


def test_gemm_caller_workspace_and_unaligned(dev):
    g = synth.rng(3002)
    N, K, M = 200, 1024, 33
    w = synth.packed_matrix(g, N, K, 0.01, 0.05)
    x = synth.activations(g, M, K)
    ws = torch.empty(q.q2_0_mul_mat_workspace_size(M, N, K), dtype=torch.uint8, device=dev)
    y = q.q2_0_mul_mat(_to(dev, w), _to(dev, x), N, K, M, workspace=ws).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, "GEMM caller workspace")
    buf = torch.zeros(w.size + 8, dtype=torch.uint8, device=dev)
    buf[3:3 + w.size] = _to(dev, w)
    y = q.q2_0_mul_mat(buf[3:3 + w.size], _to(dev, x), N, K, M).cpu().numpy()
    _assert_close(y, yo, acc, TOL_SPLIT, "GEMM unaligned weights")


@pytest.mark.parametrize("prec", [q.Q2_0_PREC_F16_SPLIT, q.Q2_0_PREC_F16])
@pytest.mark.parametrize("N,K,M", [(6144, 2048, 512), (2048, 6144, 512), (4096, 4096, 2048),
                                   (12288, 4096, 2048), (4096, 12288, 2048)])
def test_gemm_prefill_shapes_sampled(dev, N, K, M, prec):
    """The 1.7B (M=512) and 8B (M=2048) prefill shapes; 96 sampled weight rows x all M."""
    g = synth.rng(3003, N, K, M)
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    x = synth.activations(g, M, K, synth.PREFILL_OUTLIER_FRAC, synth.PREFILL_OUTLIER)
    y = q.q2_0_mul_mat(_to(dev, w), _to(dev, x), N, K, M, prec)
    rows = np.unique(np.concatenate([[0, 127, 128, N - 1], g.integers(0, N, 92)]))
    yo, acc = oracle.matmul(w, N, K, x, rows=rows)
    got = y[:, torch.from_numpy(rows).to(dev)].cpu().numpy()
    tol = TOL_SPLIT if prec == q.Q2_0_PREC_F16_SPLIT else TOL_F16
    _assert_close(got, yo, acc, tol, f"GEMM {N}x{K} M={M} prec={prec}")
    _no_device_error()


# ---------------------------------------------------------------------------
# grouped GEMM plans: several products in one prepass, one tensor-core launch
# over the pooled tiles and one stream-K reduction
# ---------------------------------------------------------------------------
def _mm_case(g, N, K, M, x=None):
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    if x is None:
        x = synth.activations(g, M, K, synth.PREFILL_OUTLIER_FRAC, synth.PREFILL_OUTLIER)
    return w, x


@pytest.mark.parametrize("prec", [q.Q2_0_PREC_F16_SPLIT, q.Q2_0_PREC_F16])
def test_mm_plan_parity_small(dev, prec):
    """Five products: two share one X (one prepass for both), one has K % 512 != 0
    (the CUDA-core kernel inside execute), ragged N and M everywhere; the pooled
    slab order is cut into few-slab stream-K ranges that cross unit and product
    boundaries."""
    g = synth.rng(3401, prec)
    shapes = [(300, 1024, 70), (513, 1024, 70), (130, 2048, 257), (40, 576, 9), (256, 512, 128)]
    cases = []
    for i, (N, K, M) in enumerate(shapes):
        x_shared = cases[0][1] if i == 1 else None
        cases.append(_mm_case(g, N, K, M, x_shared))
    xs = {}
    entries, ys = [], []
    for (w, x), (N, K, M) in zip(cases, shapes):
        xd = xs.setdefault(id(x), _to(dev, x))
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        entries.append((_to(dev, w), xd, y, N, K, M))
        ys.append(y)
    plan = q.MmPlan(entries, prec)
    # one prepass launch (4 distinct X on the tensor-core path), the GEMM and its
    # reduction, one CUDA-core launch
    assert plan.launches == 4
    plan.execute()
    tol = TOL_SPLIT if prec == q.Q2_0_PREC_F16_SPLIT else TOL_F16
    first = [y.clone() for y in ys]
    for (w, x), (N, K, M), y in zip(cases, shapes, ys):
        yo, acc = oracle.matmul(w, N, K, x)
        _assert_close(y.cpu().numpy(), yo, acc, tol, f"GEMM plan {N}x{K} M={M} prec={prec}")
    # deterministic: a second execute, and a CUDA-graph replay, give the same bits
    for y in ys:
        y.fill_(float("nan"))
    plan.execute()
    for a, b in zip(first, ys):
        assert torch.equal(a, b)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr, stream=s):
        plan.execute(s)
    for y in ys:
        y.fill_(float("nan"))
    gr.replay()
    torch.cuda.synchronize()
    for a, b in zip(first, ys):
        assert torch.equal(a, b)
    plan.close()
    _no_device_error()


def test_mm_plan_many_activations(dev):
    """Ten products with ten distinct X: two prepass launches of up to 8 each."""
    g = synth.rng(3402)
    shapes = [(64 + 37 * i, 512 * (1 + i % 3), 3 + 11 * i) for i in range(10)]
    cases = [_mm_case(g, N, K, M) for (N, K, M) in shapes]
    entries, ys = [], []
    for (w, x), (N, K, M) in zip(cases, shapes):
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        entries.append((_to(dev, w), _to(dev, x), y, N, K, M))
        ys.append(y)
    plan = q.MmPlan(entries)
    assert plan.launches == 4
    plan.execute()
    for (w, x), (N, K, M), y in zip(cases, shapes, ys):
        yo, acc = oracle.matmul(w, N, K, x)
        _assert_close(y.cpu().numpy(), yo, acc, TOL_SPLIT, f"GEMM plan {N}x{K} M={M}")
    plan.close()
    _no_device_error()


@pytest.mark.parametrize("prec", [q.Q2_0_PREC_F16_SPLIT, q.Q2_0_PREC_F16])
def test_mm_plan_prefill_sampled(dev, prec):
    """The 1.7B-class prefill products as one plan: gate and up (6144 x 2048)
    on one X of 512 tokens, down (2048 x 6144) on its own X; 96 sampled weight
    rows of each x all tokens."""
    g = synth.rng(3403, prec)
    M = 512
    shapes = [(6144, 2048), (6144, 2048), (2048, 6144)]
    x1 = synth.activations(g, M, 2048, synth.PREFILL_OUTLIER_FRAC, synth.PREFILL_OUTLIER)
    x2 = synth.activations(g, M, 6144, synth.PREFILL_OUTLIER_FRAC, synth.PREFILL_OUTLIER)
    xd1, xd2 = _to(dev, x1), _to(dev, x2)
    ws, entries, ys = [], [], []
    for i, (N, K) in enumerate(shapes):
        w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        entries.append((_to(dev, w), xd2 if i == 2 else xd1, y, N, K, M))
        ws.append(w)
        ys.append(y)
    plan = q.MmPlan(entries, prec)
    assert plan.launches == 3
    plan.execute()
    tol = TOL_SPLIT if prec == q.Q2_0_PREC_F16_SPLIT else TOL_F16
    for i, ((N, K), w, y) in enumerate(zip(shapes, ws, ys)):
        x = x2 if i == 2 else x1
        rows = np.unique(np.concatenate([[0, 255, 256, N - 1], g.integers(0, N, 92)]))
        yo, acc = oracle.matmul(w, N, K, x, rows=rows)
        got = y[:, torch.from_numpy(rows).to(dev)].cpu().numpy()
        _assert_close(got, yo, acc, tol, f"GEMM plan {N}x{K} M={M} prec={prec}")
    plan.close()
    _no_device_error()


def test_mm_plan_wide_range(dev):
    """The wide-range activation kinds, one product each, in one plan."""
    N, K, M = 260, 2048, 24
    cases = [wr.wide_range_case(kind, synth.rng(3404, i), N, K, M)
             for i, kind in enumerate(wr.WIDE_KINDS)]
    entries, ys = [], []
    for w, x in cases:
        y = torch.empty((M, N), dtype=torch.float32, device=dev)
        entries.append((_to(dev, w), _to(dev, x), y, N, K, M))
        ys.append(y)
    plan = q.MmPlan(entries)
    plan.execute()
    for kind, (w, x), y in zip(wr.WIDE_KINDS, cases, ys):
        yo, acc = oracle.matmul(w, N, K, x)
        _assert_close(y.cpu().numpy(), yo, acc, TOL_SPLIT, f"GEMM plan {kind}")
    plan.close()
    _no_device_error()


# ---------------------------------------------------------------------------
# F16 activations (the missing path of the WebGPU port's limitations paragraph)
# ---------------------------------------------------------------------------
F16_MV_CASES = [(2048, 2048, 1), (300, 2048, 2), (257, 1536, 3), (1000, 6144, 4),
                (513, 4096, 8), (33, 576, 1), (130, 1088, 8)]


@pytest.mark.parametrize("N,K,ncols", F16_MV_CASES)
def test_matvec_f16_parity(dev, N, K, ncols):
    g = synth.rng(2101, N, K, ncols)
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    x16 = synth.activations(g, ncols, K, 0.001, 30.0).astype(np.float16)
    y = q.q2_0_mul_mat_vec_f16(_to(dev, w), _to(dev, x16), N, K, ncols).cpu().numpy()
    # the oracle gets the exact values of the fp16 activations
    yo, acc = oracle.matmul(w, N, K, x16.astype(np.float32))
    _assert_close(y, yo, acc, TOL_SPLIT, f"mat-vec f16 {N}x{K} ncols={ncols}")
    _no_device_error()


@pytest.mark.parametrize("N,K,M", [(128, 512, 128), (300, 1024, 70), (17, 64, 5),
                                   (130, 2048, 257), (40, 576, 9)])
def test_gemm_f16_parity_small(dev, N, K, M):
    g = synth.rng(3101, N, K, M)
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    x16 = synth.activations(g, M, K, synth.PREFILL_OUTLIER_FRAC,
                            synth.PREFILL_OUTLIER).astype(np.float16)
    y = q.q2_0_mul_mat_f16(_to(dev, w), _to(dev, x16), N, K, M).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x16.astype(np.float32))
    _assert_close(y, yo, acc, TOL_SPLIT, f"GEMM f16 {N}x{K} M={M}")
    _no_device_error()


@pytest.mark.parametrize("N,K,M", [(6144, 2048, 512), (2048, 6144, 512)])
def test_gemm_f16_prefill_sampled(dev, N, K, M):
    g = synth.rng(3103, N, K, M)
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    x16 = synth.activations(g, M, K, synth.PREFILL_OUTLIER_FRAC,
                            synth.PREFILL_OUTLIER).astype(np.float16)
    ws = torch.empty(q.q2_0_mul_mat_workspace_size(M, N, K, q.Q2_0_PREC_F16), dtype=torch.uint8,
                     device=dev)
    y = q.q2_0_mul_mat_f16(_to(dev, w), _to(dev, x16), N, K, M, workspace=ws)
    rows = np.unique(np.concatenate([[0, 127, 128, N - 1], g.integers(0, N, 60)]))
    yo, acc = oracle.matmul(w, N, K, x16.astype(np.float32), rows=rows)
    got = y[:, torch.from_numpy(rows).to(dev)].cpu().numpy()
    _assert_close(got, yo, acc, TOL_SPLIT, f"GEMM f16 {N}x{K} M={M}")
    _no_device_error()


# ---------------------------------------------------------------------------
# Group-128 packing (34-byte blocks)
# ---------------------------------------------------------------------------
def _g128_matrix(g, N, K, lo=0.005, hi=0.05, frac_code3=0.01):
    """Seeded group-128 bytes: the same draw as the 64-weight generator, laid out
    as 34-byte blocks (scale, then 32 code bytes)."""
    nb = K // 128
    d = g.uniform(lo, hi, size=(N, nb)).astype(np.float16).view(np.uint16)
    codes = g.integers(0, 3, size=(N, nb, 128), dtype=np.uint8)
    codes[g.random((N, nb, 128)) < frac_code3] = 3
    q = codes.reshape(N, nb, 32, 4)
    byte = (q[..., 0] | (q[..., 1] << 2) | (q[..., 2] << 4) | (q[..., 3] << 6)).astype(np.uint8)
    blk = np.zeros((N, nb, 34), dtype=np.uint8)
    blk[:, :, 0] = d & 0xFF
    blk[:, :, 1] = d >> 8
    blk[:, :, 2:] = byte
    return blk.reshape(-1)


def test_g128_get_rows_bit_exact(dev):
    g = synth.rng(4101)
    n_rows, K = 3000, 4096
    table = _g128_matrix(g, n_rows, K)
    tb = table.reshape(n_rows, K // 128, 34)
    tb[0, 0, :2] = [0x00, 0x80]        # d = -0: signed zeros
    tb[1, 1, :2] = [0x01, 0x00]        # subnormal d
    tb[2, 2, 2:] = 0xFF                # all code 3
    ids = np.concatenate([[0, 1, 2, 2999], g.integers(0, n_rows, 508)]).astype(np.int32)
    got = q.q2_0_g128_get_rows(_to(dev, table), n_rows, K, _to(dev, ids)).cpu().numpy()
    ref, bad = oracle.get_rows_g128(table, n_rows, K, ids)
    assert bad == 0
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
    _no_device_error()


def test_g128_repack_then_fast_paths(dev):
    """The repacked matrix decodes to the same weights, and the fast mat-vec and
    GEMM on it match the group-128 oracle."""
    g = synth.rng(4102)
    N, K = 777, 2048
    w128 = _g128_matrix(g, N, K)
    w64 = q.q2_0_g128_to_g64(_to(dev, w128), N, K).cpu().numpy()
    rows = np.arange(N, dtype=np.int32)
    dec128, _ = oracle.get_rows_g128(w128, N, K, rows)
    assert np.array_equal(oracle.dequantize(w64, N, K).astype(np.float32).view(np.uint32),
                          dec128.view(np.uint32))
    for ncols in (1, 2, 5):
        x = synth.activations(g, ncols, K, 0.001, 30.0)
        y = q.q2_0_mul_mat_vec(_to(dev, w64), _to(dev, x), N, K, ncols).cpu().numpy()
        yo, acc = oracle.matmul_g128(w128, N, K, x)
        _assert_close(y, yo, acc, TOL_SPLIT, f"repacked mat-vec ncols={ncols}")
    x = synth.activations(g, 64, K, synth.PREFILL_OUTLIER_FRAC, synth.PREFILL_OUTLIER)
    y = q.q2_0_mul_mat(_to(dev, w64), _to(dev, x), N, K, 64).cpu().numpy()
    yo, acc = oracle.matmul_g128(w128, N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, "repacked GEMM")
    _no_device_error()


@pytest.mark.parametrize("N,K,ncols", [(300, 1024, 1), (129, 2048, 3), (64, 128, 8), (5, 896, 2),
                                       (1000, 4096, 1), (257, 2048, 1), (2000, 6144, 1),
                                       (77, 3072, 1)])
def test_g128_matvec_direct(dev, N, K, ncols):
    """ncols 1 with K % 1024 == 0 runs the fp4 tensor-core kernel on 272-byte
    stage boxes (several tiles, ragged last tile); the rest the CUDA-core kernel."""
    g = synth.rng(4103, N, K, ncols)
    w = _g128_matrix(g, N, K)
    x = synth.activations(g, ncols, K, 0.001, 30.0)
    y = q.q2_0_g128_mul_mat_vec(_to(dev, w), _to(dev, x), N, K, ncols).cpu().numpy()
    yo, acc = oracle.matmul_g128(w, N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, f"g128 mat-vec {N}x{K} ncols={ncols}")
    _no_device_error()


# ---------------------------------------------------------------------------
# Expert mat-vec (mul_mat_id; the limitations paragraph of the WebGPU port
# names MUL_MAT_ID as missing)
# ---------------------------------------------------------------------------
def _experts(g, n_expert, N, K):
    return np.concatenate([synth.packed_matrix(g, N, K, *synth.DECODE_SCALE,
                                               synth.DECODE_FRAC_CODE3) for _ in range(n_expert)])


@pytest.mark.parametrize("n_expert,N,K,n_tokens,n_used,n_x", [
    (4, 300, 1024, 3, 2, 1),     # ragged N: the last tile runs into the next expert's rows
    (4, 300, 1024, 3, 2, 2),     # one vector per slot
    (6, 128, 512, 5, 3, 1),      # one tile per expert
    (3, 97, 768, 2, 2, 2),       # K % 512 != 0: the CUDA-core kernel
    (1, 640, 2048, 4, 1, 1),     # a single expert
])
def test_mul_mat_id_parity(dev, n_expert, N, K, n_tokens, n_used, n_x):
    g = synth.rng(4101, n_expert, N, K, n_tokens, n_used, n_x)
    w = _experts(g, n_expert, N, K)
    x = synth.activations(g, n_tokens * n_x, K).reshape(n_tokens, n_x, K)
    ids = g.integers(0, n_expert, size=(n_tokens, n_used)).astype(np.int32)
    y = q.q2_0_mul_mat_id(_to(dev, w), n_expert, N, K, _to(dev, x), _to(dev, ids)).cpu().numpy()
    yo, acc, bad = oracle.matmul_id(w, n_expert, N, K, x, ids)
    assert bad == 0
    _assert_close(y.reshape(-1, N), yo.reshape(-1, N), acc.reshape(-1, N), TOL_SPLIT,
                  f"mul_mat_id {n_expert}x{N}x{K} tokens={n_tokens} used={n_used} n_x={n_x}")
    _no_device_error()


def test_mul_mat_id_moe_decode_sampled(dev):
    """A 128-expert layer of hidden 2048 (expert FFN 768), 8 experts per token:
    gate-shaped experts 768 x 2048 at 1 and 16 tokens, sampled rows."""
    n_expert, N, K, n_used = 128, 768, 2048, 8
    g = synth.rng(4102)
    w = _experts(g, n_expert, N, K)
    wd = _to(dev, w)
    for n_tokens in (1, 16):
        x = synth.activations(g, n_tokens, K).reshape(n_tokens, 1, K)
        ids = np.stack([g.permutation(n_expert)[:n_used] for _ in range(n_tokens)]).astype(np.int32)
        y = q.q2_0_mul_mat_id(wd, n_expert, N, K, _to(dev, x), _to(dev, ids)).cpu().numpy()
        rows = np.unique(np.concatenate([[0, 127, 128, N - 1], g.integers(0, N, 20)]))
        yo, acc, bad = oracle.matmul_id(w, n_expert, N, K, x, ids, rows=rows)
        assert bad == 0
        _assert_close(y[:, :, rows].reshape(-1, rows.size), yo.reshape(-1, rows.size),
                      acc.reshape(-1, rows.size), TOL_SPLIT, f"MoE decode tokens={n_tokens}")
    _no_device_error()


@pytest.mark.parametrize("K", [1024, 768])
def test_mul_mat_id_bad_ids(dev, K):
    """Out-of-range ids leave their slots unwritten and record BAD_ID; the other
    slots are correct."""
    n_expert, N, n_tokens, n_used = 3, 200, 2, 2
    g = synth.rng(4103, K)
    w = _experts(g, n_expert, N, K)
    x = synth.activations(g, n_tokens, K).reshape(n_tokens, 1, K)
    ids = np.array([[1, 3], [-2, 0]], dtype=np.int32)
    y = torch.full((n_tokens, n_used, N), 7.0, device=dev)
    q.q2_0_mul_mat_id(_to(dev, w), n_expert, N, K, _to(dev, x), _to(dev, ids), y=y)
    code, info = q.q2_0_get_error()
    assert code == q.Q2_0_DEVERR_BAD_ID and info in (1, 2)
    yh = y.cpu().numpy()
    assert np.all(yh[0, 1] == 7.0) and np.all(yh[1, 0] == 7.0)
    yo, acc, bad = oracle.matmul_id(w, n_expert, N, K, x, ids)
    assert bad == 2
    for t, i in ((0, 0), (1, 1)):
        _assert_close(yh[t, i][None], yo[t, i][None], acc[t, i][None], TOL_SPLIT, "good slots")


def test_mul_mat_id_unaligned_weights(dev):
    """Weights at an odd byte offset take the CUDA-core kernel."""
    n_expert, N, K = 2, 64, 512
    g = synth.rng(4104)
    w = _experts(g, n_expert, N, K)
    buf = torch.empty(w.size + 3, dtype=torch.uint8, device=dev)
    buf[3:] = _to(dev, w)
    x = synth.activations(g, 2, K).reshape(2, 1, K)
    ids = np.array([[1], [0]], dtype=np.int32)
    y = q.q2_0_mul_mat_id(buf[3:], n_expert, N, K, _to(dev, x), _to(dev, ids)).cpu().numpy()
    yo, acc, _ = oracle.matmul_id(w, n_expert, N, K, x, ids)
    _assert_close(y.reshape(-1, N), yo.reshape(-1, N), acc.reshape(-1, N), TOL_SPLIT, "unaligned")
    _no_device_error()


# ---------------------------------------------------------------------------
# Split layout (codes and scales in separate arrays)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("N,K", [(1, 64), (300, 1024), (129, 576), (2048, 2048)])
def test_split_layout_bit_exact_and_round_trip(dev, N, K):
    g = synth.rng(5101, N, K)
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    ref = oracle.raw_to_soa(w, N, K)
    dst = torch.full((q.q2_0_split_bytes(N, K),), 0xAB, dtype=torch.uint8, device=dev)
    q.q2_0_split_layout(_to(dev, w), N, K, dst=dst)
    got = dst.cpu().numpy()
    # the padding between and after the arrays is not written; compare the arrays
    nblk = N * (K // 64)
    d_off = -(-16 * nblk // 256) * 256
    assert np.array_equal(got[:16 * nblk], ref[:16 * nblk])
    assert np.array_equal(got[d_off:d_off + 2 * nblk], ref[d_off:d_off + 2 * nblk])
    back = q.q2_0_join_layout(dst, N, K).cpu().numpy()
    assert np.array_equal(back, w)


@pytest.mark.parametrize("N,K,ncols", [(300, 2048, 1), (2048, 6144, 1), (1000, 512, 1),
                                       (129, 576, 1), (257, 1024, 3), (64, 2048, 8)])
def test_matvec_split_parity(dev, N, K, ncols):
    g = synth.rng(5102, N, K, ncols)
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    x = synth.activations(g, ncols, K)
    soa = q.q2_0_split_layout(_to(dev, w), N, K)
    y = q.q2_0_mul_mat_vec_split(soa, _to(dev, x), N, K, ncols).cpu().numpy()
    yo, acc = oracle.matmul_soa(oracle.raw_to_soa(w, N, K), N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, f"split mat-vec {N}x{K} ncols={ncols}")
    _no_device_error()


def test_matvec_split_head_sampled_and_unaligned(dev):
    """The 151936 x 4096 head in the split layout (sampled rows), and the same
    buffer at an 8-byte offset, which takes the CUDA-core kernel."""
    N, K = 151936, 4096
    g = synth.rng(5103)
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    x = synth.activations(g, 1, K)
    soa = q.q2_0_split_layout(_to(dev, w), N, K)
    y = q.q2_0_mul_mat_vec_split(soa, _to(dev, x), N, K).cpu().numpy()
    rows = np.unique(np.concatenate([[0, 127, 128, N - 1], g.integers(0, N, 60)]))
    yo, acc = oracle.matmul(w, N, K, x, rows=rows)
    _assert_close(y[:, rows], yo, acc, TOL_SPLIT, "split head")
    nb = q.q2_0_split_bytes(N, K)
    buf = torch.empty(nb + 8, dtype=torch.uint8, device=dev)
    buf[8:] = soa
    y2 = q.q2_0_mul_mat_vec_split(buf[8:], _to(dev, x), N, K).cpu().numpy()
    _assert_close(y2[:, rows], yo, acc, TOL_SPLIT, "split head, unaligned")
    _no_device_error()


# ---------------------------------------------------------------------------
# Wide dynamic range inside one activation vector. The tolerance is relative to
# sum|w*x|, so a small element must keep its own relative precision even when
# it shares a vector (or a block of 64) with an element 10^5 times larger, and
# an element whose weight is zero (code 1) must contribute exactly nothing,
# however large it is. The inputs come from tests/wide_range.py.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("ncols", [1, 2, 4, 8])
@pytest.mark.parametrize("kind", wr.WIDE_KINDS)
def test_matvec_wide_range(dev, kind, ncols):
    g = synth.rng(2202, wr.WIDE_KINDS.index(kind), ncols)
    N, K = 260, 2048
    w, x = wr.wide_range_case(kind, g, N, K, ncols)
    y = q.q2_0_mul_mat_vec(_to(dev, w), _to(dev, x), N, K, ncols).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, f"mat-vec {kind} ncols={ncols}")
    _no_device_error()


@pytest.mark.parametrize("ncols", [1, 2, 3, 8])
def test_plan_wide_range(dev, ncols):
    g = synth.rng(2203, ncols)
    ents, host = [], []
    for i, (N, K) in enumerate([(300, 2048), (129, 6144), (1000, 1024)]):
        w, x = wr.wide_range_case(wr.WIDE_KINDS[i % len(wr.WIDE_KINDS)], g, N, K, ncols)
        ents.append((_to(dev, w), _to(dev, x), torch.empty((ncols, N), device=dev), N, K))
        host.append((w, x))
    plan = q.MvPlan(ents, ncols)
    plan.execute()
    torch.cuda.synchronize()
    for (w, x), (_, _, yd, N, K) in zip(host, ents):
        yo, acc = oracle.matmul(w, N, K, x)
        _assert_close(yd.cpu().numpy(), yo, acc, TOL_SPLIT, f"plan wide {N}x{K} ncols={ncols}")
    plan.close()
    _no_device_error()


@pytest.mark.parametrize("kind", wr.WIDE_KINDS)
def test_mul_mat_id_wide_range(dev, kind):
    n_expert, N, K, n_tokens, n_used = 3, 200, 1024, 2, 2
    g = synth.rng(2204, wr.WIDE_KINDS.index(kind))
    ws, xs = zip(*[wr.wide_range_case(kind, g, N, K, n_tokens) for _ in range(n_expert)])
    w = np.concatenate(ws)
    x = xs[0].reshape(n_tokens, 1, K)
    ids = np.array([[0, 2], [1, 0]], dtype=np.int32)
    y = q.q2_0_mul_mat_id(_to(dev, w), n_expert, N, K, _to(dev, x), _to(dev, ids)).cpu().numpy()
    yo, acc, bad = oracle.matmul_id(w, n_expert, N, K, x, ids)
    assert bad == 0
    _assert_close(y.reshape(-1, N), yo.reshape(-1, N), acc.reshape(-1, N), TOL_SPLIT,
                  f"mul_mat_id {kind}")
    _no_device_error()


@pytest.mark.parametrize("kind", wr.WIDE_KINDS)
def test_matvec_split_wide_range(dev, kind):
    g = synth.rng(2205, wr.WIDE_KINDS.index(kind))
    N, K = 300, 2048
    w, x = wr.wide_range_case(kind, g, N, K, 1)
    soa = q.q2_0_split_layout(_to(dev, w), N, K)
    y = q.q2_0_mul_mat_vec_split(soa, _to(dev, x), N, K, 1).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, f"split mat-vec {kind}")
    _no_device_error()


@pytest.mark.parametrize("ncols", [1, 2, 4])
def test_matvec_f16_wide_range(dev, ncols):
    g = synth.rng(2206, ncols)
    N, K = 260, 2048
    w, x = wr.wide_range_case("const_outliers", g, N, K, ncols)
    x16 = x.astype(np.float16)
    y = q.q2_0_mul_mat_vec_f16(_to(dev, w), _to(dev, x16), N, K, ncols).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x16.astype(np.float32))
    _assert_close(y, yo, acc, TOL_SPLIT, f"mat-vec f16 wide ncols={ncols}")
    _no_device_error()


@pytest.mark.parametrize("kind", wr.WIDE_KINDS)
def test_g128_matvec_wide_range(dev, kind):
    """The group-128 tensor-core path scales activations per 128 elements: small
    elements beside large ones and large elements under zero weights."""
    g = synth.rng(4104, wr.WIDE_KINDS.index(kind))
    N, K = 300, 4096
    w64, x = wr.wide_range_case(kind, g, N, K, 1)
    w = wr.to_g128(w64, N, K)
    y = q.q2_0_g128_mul_mat_vec(_to(dev, w), _to(dev, x), N, K, 1).cpu().numpy()
    yo, acc = oracle.matmul_g128(w, N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, f"g128 mat-vec {kind}")
    _no_device_error()


def test_g128_matvec_edge_blocks(dev):
    """Blocks with d = +-0, a subnormal d, all code 3 and d = 65504 on the
    group-128 tensor-core path."""
    g = synth.rng(4105)
    N, K = 260, 2048
    w = _g128_matrix(g, N, K)
    wb = w.reshape(N, K // 128, 34)
    for r in range(0, N, 5):
        b = r % (K // 128)
        kind = (r // 5) % 4
        if kind == 0:
            wb[r, b, :2] = [0x00, 0x80]       # -0
        elif kind == 1:
            wb[r, b, :2] = [0x01, 0x00]       # smallest subnormal
        elif kind == 2:
            wb[r, b, 2:] = 0xFF               # all code 3
        else:
            wb[r, b, :2] = [0xFF, 0x7B]       # 65504
            wb[r, b, 2:] = 0x24               # codes 0, 1, 2, 0
    x = synth.activations(g, 1, K, 0.001, 30.0)
    y = q.q2_0_g128_mul_mat_vec(_to(dev, w), _to(dev, x), N, K, 1).cpu().numpy()
    yo, acc = oracle.matmul_g128(w, N, K, x)
    assert np.all(np.isfinite(y))
    _assert_close(y, yo, acc, TOL_SPLIT, "g128 mat-vec edge blocks")
    _no_device_error()


def test_g128_matvec_head_sampled(dev):
    """A 151936 x 4096 group-128 head on the tensor-core path, checked on 512
    sampled rows (first, last, tile edges and random ones)."""
    g = synth.rng(4106)
    N, K = 151936, 4096
    nb = K // 128
    wb = np.empty((N, nb, 34), dtype=np.uint8)   # uniform codes 0..3 (byte draws)
    wb[:, :, 2:] = g.integers(0, 256, size=(N, nb, 32), dtype=np.uint8)
    d = g.uniform(0.005, 0.05, size=(N, nb)).astype(np.float16).view(np.uint16)
    wb[:, :, 0] = d & 0xFF
    wb[:, :, 1] = d >> 8
    w = wb.reshape(-1)
    x = synth.activations(g, 1, K, 0.001, 30.0)
    y = q.q2_0_g128_mul_mat_vec(_to(dev, w), _to(dev, x), N, K, 1).cpu().numpy()
    rows = np.unique(np.concatenate([[0, 127, 128, N - 129, N - 128, N - 1],
                                     g.integers(0, N, 506)])).astype(np.int64)
    yo, acc = oracle.matmul_g128(w, N, K, x, rows=rows)
    _assert_close(y[:, rows], yo, acc, TOL_SPLIT, "g128 head sampled rows")
    _no_device_error()


# ---------------------------------------------------------------------------
# GEMM: edge blocks, activations far from 1 (tiny, huge) and wide range
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("prec", [q.Q2_0_PREC_F16_SPLIT, q.Q2_0_PREC_F16])
def test_gemm_edge_blocks(dev, prec):
    """Rows seeded with the edge blocks (d = +-0, subnormal d, all code 3, all
    code 1, d = 65504 with codes 0..2): all finite in f32."""
    g = synth.rng(3201, prec)
    N, K, M = 300, 2048, 70
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    edges = synth.edge_blocks()
    wv = w.reshape(N, K // 64, 18)
    for r in range(0, N, 3):
        wv[r, r % (K // 64)] = edges[r % len(edges)]
        wv[r, (r + 7) % (K // 64)] = edges[(r + 1) % len(edges)]
    x = synth.activations(g, M, K, synth.PREFILL_OUTLIER_FRAC, synth.PREFILL_OUTLIER)
    y = q.q2_0_mul_mat(_to(dev, w), _to(dev, x), N, K, M, prec).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x)
    tol = TOL_SPLIT if prec == q.Q2_0_PREC_F16_SPLIT else TOL_F16
    _assert_close(y, yo, acc, tol, f"GEMM edge blocks prec={prec}")
    _no_device_error()


@pytest.mark.parametrize("prec", [q.Q2_0_PREC_F16_SPLIT, q.Q2_0_PREC_F16])
@pytest.mark.parametrize("scale", [1e-4, 1e-6, 1e-30, 1e5, 1e30])
def test_gemm_activation_magnitude(dev, prec, scale):
    """Activations scaled far below fp16's normal range and far above its
    largest value: the result keeps the stated tolerance."""
    g = synth.rng(3202, prec, int(np.log10(scale)) + 40)
    N, K, M = 260, 2048, 40
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    x = (synth.activations(g, M, K, synth.PREFILL_OUTLIER_FRAC, synth.PREFILL_OUTLIER)
         * np.float32(scale)).astype(np.float32)
    y = q.q2_0_mul_mat(_to(dev, w), _to(dev, x), N, K, M, prec).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x)
    tol = TOL_SPLIT if prec == q.Q2_0_PREC_F16_SPLIT else TOL_F16
    _assert_close(y, yo, acc, tol, f"GEMM x*{scale:g} prec={prec}")
    _no_device_error()


@pytest.mark.parametrize("kind", wr.WIDE_KINDS)
def test_gemm_wide_range(dev, kind):
    g = synth.rng(3203, wr.WIDE_KINDS.index(kind))
    N, K, M = 260, 2048, 24
    w, x = wr.wide_range_case(kind, g, N, K, M)
    y = q.q2_0_mul_mat(_to(dev, w), _to(dev, x), N, K, M).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, f"GEMM {kind}")
    _no_device_error()


@pytest.mark.parametrize("ncols", [1, 2, 4])
@pytest.mark.parametrize("scale", [1e-30, 1e30])
def test_matvec_activation_magnitude(dev, ncols, scale):
    g = synth.rng(2207, ncols, int(np.log10(scale)) + 40)
    N, K = 260, 2048
    w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    x = (synth.activations(g, ncols, K, 0.001, 30.0) * np.float32(scale)).astype(np.float32)
    y = q.q2_0_mul_mat_vec(_to(dev, w), _to(dev, x), N, K, ncols).cpu().numpy()
    yo, acc = oracle.matmul(w, N, K, x)
    _assert_close(y, yo, acc, TOL_SPLIT, f"mat-vec x*{scale:g} ncols={ncols}")
    _no_device_error()
