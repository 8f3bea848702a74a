#!/usr/bin/env python3
"""Benchmark of the Q2_0 hot path on one or more GB300s (one process per GPU).

One step = one pass of the whole hot path over one batch of synthetic input of
the 1.7B-class decoder (hidden 2048, 28 layers):
  1. get_rows: 512 seeded token ids from a 151936 x 2048 Q2_0 embedding table;
  2. prefill GEMM at M = 512 tokens over the layer's Q2_0 shapes gate/up
     (6144 x 2048, both reading one X) and down (2048 x 6144), F32
     activations, split fp16 hi+lo, as one grouped plan (the extras time the
     same products as separate calls and as two plans, gate+up then down);
  3. decode step: the 196 Q2_0 mat-vecs (q, k, v, o, gate, up, down x 28) at
     ncols = 1, each matrix with its own activation vector, as one batched plan.
value = packed-weight bytes of the decode step / the decode part's device time
(GB/s); the GEMM's TFLOP/s (2*M*N*K per product) and get_rows' bytes/s are
reported beside it. Inputs are resident in HBM before timing; the 396 MB of
packed decode weights streamed every step exceed the 129 MB L2, so no kernel
sees its inputs cached from the previous step. The timed steps replay CUDA
graphs of the three parts (captured from the same library calls); the e2e
figure times the plain public-API calls with host copies instead.

--impl reference runs the CPU oracle on bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "Q2_0 mat-vec weight GB/s (% of HBM peak); GEMM TFLOP/s at M=512"
WORKLOAD = "1.7B-class decoder, hidden 2048 x 28 layers: decode step (196 Q2_0 mat-vecs, ncols=1) " \
           "+ prefill GEMM M=512 (6144x2048, 6144x2048, 2048x6144) + get_rows 512 of 151936x2048"
VOCAB = 151936
HIDDEN = 2048
PREFILL_M = 512
GEMM_SHAPES = [("gate", 6144, 2048), ("up", 6144, 2048), ("down", 2048, 6144)]
N_IDS = 512
SEED = 1002


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def init_dist(world: int, backend: str):
    if world <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend=backend)
    return dist


def reduce_max(dist, value: float, device=None) -> float:
    """Max over ranks (identity with one rank)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def source_sha256(paths) -> str:
    import hashlib
    h = hashlib.sha256()
    for rel in paths:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def committed_traffic(kernel: str):
    """DRAM bytes per launch of `kernel` from the committed ncu summary
    (profiles/traffic.json), or None when absent or when the kernel's sources
    have changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            entry = json.load(f).get(kernel)
        if entry and source_sha256(entry["sources"]) == entry["sha256"]:
            return int(entry["bytes_per_launch"])
    except (OSError, ValueError, KeyError):
        pass
    return None


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"q2_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for nm, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        try:
            os.remove(self.path)
        except OSError:
            pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workload construction (host arrays; identical for both arms)
# ---------------------------------------------------------------------------
def decode_inputs(ncols: int = 1):
    mats = synth.decode_step_1p7b()
    out = []
    for idx, (layer, m) in enumerate(mats):
        g = synth.rng(SEED, idx)
        w = synth.packed_matrix(g, m.N, m.K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
        x = synth.activations(g, ncols, m.K)
        out.append((m, w, x))
    return out


def gemm_inputs():
    """The M = 512 prefill products (name, N, K, w, x). Gate and up read the same
    X, as both projections of a layer read its normed hidden state; down reads
    its own."""
    xs = {}
    out = []
    for i, (name, N, K) in enumerate(GEMM_SHAPES):
        g = synth.rng(SEED + 3, i)
        w = synth.packed_matrix(g, N, K, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
        if K not in xs:
            xs[K] = synth.activations(synth.rng(SEED + 4, K), PREFILL_M, K,
                                      synth.PREFILL_OUTLIER_FRAC, synth.PREFILL_OUTLIER)
        out.append((name, N, K, w, xs[K]))
    return out


def gemm_flops_512():
    return sum(2.0 * PREFILL_M * N * K for _, N, K in GEMM_SHAPES)


def gemm_device_entries(torch, dev, gm, M):
    """MmPlan entries (w, x, y, N, K, M) on the device; a shared X is copied once."""
    d_x, ents = {}, []
    for _, N, K, w, x in gm:
        if id(x) not in d_x:
            d_x[id(x)] = torch.from_numpy(x).to(dev)
        ents.append((torch.from_numpy(w).to(dev), d_x[id(x)],
                     torch.empty((M, N), dtype=torch.float32, device=dev), N, K, M))
    return ents


def rows_inputs():
    g = synth.rng(SEED + 5)
    table = synth.packed_matrix(g, VOCAB, HIDDEN, *synth.DECODE_SCALE, synth.DECODE_FRAC_CODE3)
    ids = synth.token_ids(g, N_IDS, VOCAB, 0.05)
    return table, ids


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch

    import bit_ternary_matmul_gb300 as q

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(world, "nccl")
    q.build()
    if q.q2_0_device_check() != q.Q2_0_OK:
        raise SystemExit("q2_0: current device is not compute capability 10.3")
    peaks = load_peaks()
    stream = torch.cuda.Stream(device=dev)

    # ---- resident inputs -------------------------------------------------
    # Decode activations and outputs live in two contiguous buffers (one slice
    # per matrix), as a runtime would lay out a step's vectors.
    nc = args.ncols
    dec = decode_inputs(nc)
    dec_bytes = sum(w.size for _, w, _ in dec)
    x_off, y_off, xo, yo = [], [], 0, 0
    for m, _, _ in dec:
        x_off.append(xo)
        y_off.append(yo)
        xo += nc * m.K
        yo += nc * m.N
    d_xall = torch.empty(xo, dtype=torch.float32, device=dev)
    d_yall = torch.empty(yo, dtype=torch.float32, device=dev)
    h_xall = torch.from_numpy(np.concatenate([x.reshape(-1) for _, _, x in dec]))
    d_xall.copy_(h_xall)
    d_dec = []
    for (m, w, _), xo_, yo_ in zip(dec, x_off, y_off):
        d_dec.append((torch.from_numpy(w).to(dev), d_xall[xo_:xo_ + nc * m.K].view(nc, m.K),
                      d_yall[yo_:yo_ + nc * m.N].view(nc, m.N), m.N, m.K))
    dec_x_bytes = d_xall.numel() * 4
    dec_y_bytes = d_yall.numel() * 4
    plan = q.MvPlan(d_dec, nc) if args.only in ("all", "decode") else None

    # The prefill part: the three M = 512 products as one grouped plan (one
    # prepass for the two distinct X, one tensor-core launch over all output
    # tiles, one stream-K reduction).
    gm = gemm_inputs()
    d_gm = gemm_device_entries(torch, dev, gm, PREFILL_M)
    gemm_flops = sum(2.0 * PREFILL_M * N * K for _, N, K, _, _ in gm)
    mm_plan = q.MmPlan(d_gm, q.Q2_0_PREC_F16_SPLIT) if args.only in ("all", "gemm") else None

    table, ids = rows_inputs()
    d_table = torch.from_numpy(table).to(dev)
    d_ids = torch.from_numpy(ids).to(dev)
    d_rows = torch.empty((N_IDS, HIDDEN), dtype=torch.float32, device=dev)
    rows_bytes = N_IDS * (HIDDEN // 64) * 18 + N_IDS * HIDDEN * 4
    del dec, gm, table
    torch.cuda.synchronize()

    launches_per_step = (1 if args.only in ("all", "get_rows") else 0) + \
        (mm_plan.launches if mm_plan is not None else 0) + \
        (plan.launches if plan is not None else 0)

    run_rows = args.only in ("all", "get_rows")
    run_gemm = args.only in ("all", "gemm")
    run_dec = args.only in ("all", "decode")

    def step(ev=None):
        with torch.cuda.stream(stream):
            if ev:
                ev[0].record(stream)
            if run_rows:
                q.q2_0_get_rows(d_table, VOCAB, HIDDEN, d_ids, out=d_rows, stream=stream)
            if ev:
                ev[1].record(stream)
            if run_gemm:
                mm_plan.execute(stream)
            if ev:
                ev[2].record(stream)
            if run_dec:
                plan.execute(stream)
            if ev:
                ev[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    code, info = q.q2_0_get_error(stream)
    if code != 0:
        raise SystemExit(f"device error word {code} (info {info}) after warm-up")

    # Device-side timing: each part of the step is captured once into a CUDA
    # graph (the same library calls), and the timed loop replays the three
    # graphs with events between them, so host-side call overhead is not timed.
    def capture(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            fn()
        return g

    # Between the GEMM part and the decode part the step reads a buffer twice
    # the size of L2: the GEMM part's outputs (about 29 MB at M = 512) are then
    # written back to HBM during that read rather than during the decode
    # part's weight stream. The read is inside the timed step but in neither
    # part's time.
    flush_buf = torch.ones(64 << 20, dtype=torch.float32, device=dev) if run_dec and run_gemm else None
    flush_out = torch.empty((), dtype=torch.float32, device=dev) if flush_buf is not None else None
    graphs = []
    with torch.cuda.stream(stream):
        if run_rows:
            graphs.append(("rows", capture(lambda: q.q2_0_get_rows(
                d_table, VOCAB, HIDDEN, d_ids, out=d_rows, stream=stream))))
        if run_gemm:
            graphs.append(("gemm", capture(lambda: mm_plan.execute(stream))))
        if flush_buf is not None:
            graphs.append(("flush", capture(lambda: torch.sum(flush_buf, dim=0, out=flush_out))))
        if run_dec:
            graphs.append(("dec", capture(lambda: plan.execute(stream))))
    gmap = dict(graphs)

    def graph_step(ev=None):
        with torch.cuda.stream(stream):
            if ev:
                ev[0].record(stream)
            if "rows" in gmap:
                gmap["rows"].replay()
            if ev:
                ev[1].record(stream)
            if "gemm" in gmap:
                gmap["gemm"].replay()
            if ev:
                ev[2].record(stream)
            if "flush" in gmap:
                gmap["flush"].replay()
            if ev:
                ev[3].record(stream)
            if "dec" in gmap:
                gmap["dec"].replay()
            if ev:
                ev[4].record(stream)

    for _ in range(args.warmup):
        graph_step()
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)  # first clock sample lands before the timed region
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for k in range(args.steps):
        graph_step(evs[k])
    t_end.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clk = clocks.stop()

    total_ms = t_start.elapsed_time(t_end)
    rows_ms = sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps
    gemm_ms = sum(e[1].elapsed_time(e[2]) for e in evs) / args.steps
    dec_ms = sum(e[3].elapsed_time(e[4]) for e in evs) / args.steps
    ms_per_step = total_ms / args.steps
    # max over ranks (each rank runs its own decoder replica: weak scaling)
    ms_per_step = reduce_max(dist, ms_per_step, dev)
    dec_ms = reduce_max(dist, dec_ms, dev)
    gemm_ms = reduce_max(dist, gemm_ms, dev)
    rows_ms = reduce_max(dist, rows_ms, dev)

    value = world * dec_bytes / (dec_ms * 1e-3) / 1e9
    gemm_tflops = world * gemm_flops / (gemm_ms * 1e-3) / 1e12
    rows_gbs = world * rows_bytes / (rows_ms * 1e-3) / 1e9

    # ---- end to end through the public API with host buffers --------------
    def make_plan(dx, dy):  # the same matrices over a second set of x and y buffers
        ents = []
        for (w, _, _, N, K), xo_, yo_ in zip(d_dec, x_off, y_off):
            ents.append((w, dx[xo_:xo_ + nc * K].view(nc, K), dy[yo_:yo_ + nc * N].view(nc, N), N, K))
        return q.MvPlan(ents, nc)

    e2e = measure_e2e(args, torch, stream, plan, h_xall, d_xall, d_yall, dec_bytes, make_plan) \
        if plan is not None else {"value": None, "unit": "GB/s"}
    e2e_val = reduce_sum(dist, e2e["value"], dev) if dist else e2e["value"]
    e2e["value"] = e2e_val

    extras = None
    configs = None
    if args.only == "all" and not args.no_extras:
        configs = measure_configs(torch, q, stream, dev, peaks["hbm_gbs"])
        extras = measure_extras(torch, q, stream, dev, peaks["hbm_gbs"])

    code, info = q.q2_0_get_error(stream)
    if code != 0:
        raise SystemExit(f"device error word {code} (info {info}) after timing")

    # ---- roofline of the dominant kernels -----------------------------------
    per_gpu_dec = dec_bytes / (dec_ms * 1e-3) / 1e9
    hbm = peaks["hbm_gbs"]
    roof_mv = {"bound": "hbm", "achieved": round(per_gpu_dec, 1), "peak": hbm, "unit": "GB/s",
               "frac": round(per_gpu_dec / hbm, 4),
               "traffic": committed_traffic("mv_t4_kernel/decoder_1p7b_step_ncols1"),
               "kernel": "mv_t4_kernel (decode mat-vec plan, incl. its activation prep launch)",
               "peak_source": peaks["source"]}
    per_gpu_gemm = gemm_flops / (gemm_ms * 1e-3) / 1e12
    # fp16 dense peak = measured bf16 peak (same nominal rate); split path does 2x tensor work.
    # The GEMM part is timed as sub-millisecond graph replays, so the burst peak applies.
    tpk = peaks["bf16_tflops"]
    roof_gemm = {"bound": "tensor", "achieved": round(per_gpu_gemm, 2), "peak": tpk,
                 "unit": "TFLOP/s", "frac": round(per_gpu_gemm / tpk, 4),
                 "traffic": committed_traffic("gemm_tc_kernel/prefill_1p7b_m512"),
                 "tensor_frac_hi_lo": round(2 * per_gpu_gemm / tpk, 4),
                 "kernel": "gemm_tc_kernel (one grouped plan over the three M=512 products, "
                           "fp16 hi+lo split, incl. its prepass and stream-K reduction)",
                 "peak_source": peaks["source"] + " bf16 (fp16 dense rate is the same)"}
    # The dominant kernel: the decode mat-vec kernel has the largest single-kernel
    # share of the step's launch list (the GEMM part is three kernels: prepass,
    # tensor-core kernel, stream-K reduction), and it carries the headline metric.
    dominant, other = roof_mv, roof_gemm

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "u8 weights (2-bit codes), f32 activations; tensor-core operands: decode "
                     "e2m1 (exact codes, 16 block-scaled activation pieces), GEMM fp16 hi+lo",
            "data": "synthetic (seeded; no trained weights)",
            "config": {"workload": WORKLOAD if nc == 1 else WORKLOAD.replace("ncols=1", f"ncols={nc}"),
                       "ncols": nc, "decode_matrices": len(d_dec),
                       "decode_weight_bytes": dec_bytes, "prefill_M": PREFILL_M,
                       "gemm_prec": "f16_split",
                       "gemm": "gate and up (6144x2048, one shared X) and down (2048x6144) as "
                               "one grouped plan",
                       "get_rows_ids": N_IDS,
                       "l2": "inputs larger than L2 (396 MB packed weights streamed per step); "
                             "a 256 MB read between the GEMM part and the decode part writes the "
                             "GEMM outputs back before the decode part (timed in the step, in "
                             "neither part)",
                       "timing": "CUDA-graph replay of each part, CUDA events on the launching stream",
                       "parallelism": f"replicas x{world}"},
            "hbm_frac": round(per_gpu_dec / hbm, 4),
            "gemm_tflops": round(gemm_tflops, 2),
            "get_rows_gbs": round(rows_gbs, 2),
            "parts_ms": {"get_rows": round(rows_ms, 5), "gemm": round(gemm_ms, 5),
                         "decode_matvec": round(dec_ms, 5)},
            "roofline": dominant, "roofline_other": other,
            "e2e": e2e, "gpu_launches": launches_per_step * args.steps,
            "clocks": clk, "cpu_baseline": cpu, "impl": "ours",
            "configs": configs,
            "extras": extras,
        }
        print(json.dumps(line), flush=True)
    if plan is not None:
        plan.close()
    if mm_plan is not None:
        mm_plan.close()
    if dist is not None:
        dist.destroy_process_group()


def measure_extras(torch, q, stream, dev, hbm_peak: float, reps: int = 20):
    """Side measurements outside the step, each a CUDA-graph replay timed with
    events on the launching stream:
      - the 151936 x 4096 output-head mat-vec (ncols 1), with F32 and with F16
        activations (175 MB of packed weights, above L2);
      - the same head mat-vec on the split layout (codes and scales in
        separate arrays), against the 18-byte layout, and the split itself;
      - the M = 512 prefill GEMMs with F16 activations (q2_0_mul_mat_f16);
      - the M = 512 split products as three q2_0_mul_mat calls, and as two
        plans in a layer's order (gate and up, then down);
      - the group-128 packing of the head-sized matrix: exact repack to the
        64-weight layout (bytes read + written) and the direct mat-vec;
      - the 8B-class decode step (253 matrices with the 151936 x 4096 head,
        2,128,527,360 packed bytes, ncols 1) as one plan;
      - the 8B-class prefill GEMMs at M = 2048 (4096x4096, 12288x4096,
        4096x12288), split fp16 hi+lo, as three calls and as one plan;
      - the expert mat-vec (q2_0_mul_mat_id) of one 128-expert layer with
        768 x 2048 experts, 8 experts per token, at 1 and 64 tokens.
    The 8B-class weights and activations are drawn on the device
    (synth.packed_matrix_device: the decode-step distribution, other bytes).
    Returns the GB/s and TFLOP/s figures."""
    g = synth.rng(SEED + 7)
    N, K = VOCAB, 4096
    w = torch.from_numpy(synth.packed_matrix(g, N, K, *synth.DECODE_SCALE,
                                             synth.DECODE_FRAC_CODE3)).to(dev)
    x = torch.from_numpy(synth.activations(g, 1, K)).to(dev)
    x16 = x.half()
    y = torch.empty((1, N), dtype=torch.float32, device=dev)
    head_bytes = w.numel()

    def timed(fn):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(gr, stream=stream):
                fn()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            gr.replay()
            a.record(stream)
            for _ in range(reps):
                gr.replay()
            b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps  # ms

    ms32 = timed(lambda: q.q2_0_mul_mat_vec(w, x, N, K, 1, y=y, stream=stream))
    ms16 = timed(lambda: q.q2_0_mul_mat_vec_f16(w, x16, N, K, 1, y=y, stream=stream))
    # the same head in the split layout (codes and scales apart), and the split itself
    split = q.q2_0_split_layout(w, N, K)
    ms_sp = timed(lambda: q.q2_0_mul_mat_vec_split(split, x, N, K, 1, y=y, stream=stream))
    ms_mk = timed(lambda: q.q2_0_split_layout(w, N, K, dst=split, stream=stream))
    split_bytes = split.numel()
    del w, split
    gm = []
    for name, Ng, Kg, wg, xg in gemm_inputs():
        ws = torch.empty(q.q2_0_mul_mat_workspace_size(PREFILL_M, Ng, Kg, q.Q2_0_PREC_F16),
                         dtype=torch.uint8, device=dev)
        gm.append((torch.from_numpy(wg).to(dev), torch.from_numpy(xg).to(dev).half(),
                   torch.empty((PREFILL_M, Ng), dtype=torch.float32, device=dev), Ng, Kg, ws))
    flops = sum(2.0 * PREFILL_M * Ng * Kg for _, _, _, Ng, Kg, _ in gm)

    def gemms():
        for wg, xg, yg, Ng, Kg, ws in gm:
            q.q2_0_mul_mat_f16(wg, xg, Ng, Kg, PREFILL_M, y=yg, workspace=ws, stream=stream)

    msg = timed(gemms)
    gemm_shapes = [[PREFILL_M, Ng, Kg] for _, _, _, Ng, Kg, _ in gm]
    del gm
    # The M = 512 split products of the step's prefill part two other ways: as
    # three separate calls (a prepass, a tensor-core launch and a reduction
    # each), and as a layer's MLP orders them: gate and up in one plan, then
    # down in a second (down reads the gated product, so it cannot share the
    # first launch).
    ents = gemm_device_entries(torch, dev, gemm_inputs(), PREFILL_M)
    wss = [torch.empty(q.q2_0_mul_mat_workspace_size(PREFILL_M, Ng, Kg), dtype=torch.uint8,
                       device=dev) for _, _, _, Ng, Kg, _ in ents]

    def per_call():
        for (wg, xg, yg, Ng, Kg, Mg), ws in zip(ents, wss):
            q.q2_0_mul_mat(wg, xg, Ng, Kg, Mg, q.Q2_0_PREC_F16_SPLIT, y=yg, workspace=ws,
                           stream=stream)

    ms_pc = timed(per_call)
    plan_gu, plan_dn = q.MmPlan(ents[:2]), q.MmPlan(ents[2:])

    def two_plans():
        plan_gu.execute(stream)
        plan_dn.execute(stream)

    ms_2p = timed(two_plans)
    plan_gu.close()
    plan_dn.close()
    del ents, wss
    # group-128 packing: the exact repack to the 64-weight layout, and the direct
    # CUDA-core mat-vec, on the head-sized matrix
    w128 = torch.from_numpy(synth.packed_matrix_g128(g, N, K, *synth.DECODE_SCALE)).to(dev)
    w64 = torch.empty(q.packed_bytes(N, K), dtype=torch.uint8, device=dev)
    ms_rp = timed(lambda: q.q2_0_g128_to_g64(w128, N, K, dst=w64, stream=stream))
    ms_g = timed(lambda: q.q2_0_g128_mul_mat_vec(w128, x, N, K, 1, y=y, stream=stream))
    rp_bytes = w128.numel() + w64.numel()
    g128_bytes = w128.numel()
    del w128, w64

    # 8B-class decode step, one plan over its 253 matrices
    gen = torch.Generator(device=dev)
    gen.manual_seed(SEED + 8)
    ents8 = []
    for _, m in synth.decode_step_8b(with_head=True):
        w8 = synth.packed_matrix_device(torch, gen, m.N, m.K, *synth.DECODE_SCALE,
                                        synth.DECODE_FRAC_CODE3, dev)
        x8 = torch.randn((1, m.K), generator=gen, device=dev)
        ents8.append((w8, x8, torch.empty((1, m.N), dtype=torch.float32, device=dev), m.N, m.K))
    bytes8 = sum(e[0].numel() for e in ents8)
    plan8 = q.MvPlan(ents8, 1)
    ms8 = timed(lambda: plan8.execute(stream))
    plan8.close()
    del ents8

    # 8B-class prefill GEMMs at M = 2048
    M2 = 2048
    g2 = []
    for Ng, Kg in [(4096, 4096), (12288, 4096), (4096, 12288)]:
        wg = synth.packed_matrix_device(torch, gen, Ng, Kg, *synth.DECODE_SCALE,
                                        synth.DECODE_FRAC_CODE3, dev)
        xg = torch.randn((M2, Kg), generator=gen, device=dev)
        out = torch.rand((M2, Kg), generator=gen, device=dev) < synth.PREFILL_OUTLIER_FRAC
        sign = torch.where(torch.rand((M2, Kg), generator=gen, device=dev) < 0.5, -1.0, 1.0)
        xg = torch.where(out, sign * synth.PREFILL_OUTLIER, xg)
        ws = torch.empty(q.q2_0_mul_mat_workspace_size(M2, Ng, Kg, q.Q2_0_PREC_F16_SPLIT),
                         dtype=torch.uint8, device=dev)
        g2.append((wg, xg, torch.empty((M2, Ng), dtype=torch.float32, device=dev), Ng, Kg, ws))
    flops2 = sum(2.0 * M2 * Ng * Kg for _, _, _, Ng, Kg, _ in g2)

    def gemms2():
        for wg, xg, yg, Ng, Kg, ws in g2:
            q.q2_0_mul_mat(wg, xg, Ng, Kg, M2, prec=q.Q2_0_PREC_F16_SPLIT, y=yg, workspace=ws,
                           stream=stream)

    ms2 = timed(gemms2)
    plan2 = q.MmPlan([(wg, xg, yg, Ng, Kg, M2) for wg, xg, yg, Ng, Kg, _ in g2])
    ms2p = timed(lambda: plan2.execute(stream))
    plan2.close()
    del g2

    # expert mat-vec: 128 experts of 768 x 2048, 8 per token
    n_exp, Ne, Ke, n_used = 128, 768, 2048, 8
    we = synth.packed_matrix_device(torch, gen, n_exp * Ne, Ke, *synth.DECODE_SCALE,
                                    synth.DECODE_FRAC_CODE3, dev)
    moe = {}
    for n_tok in (1, 64):
        xe = torch.randn((n_tok, 1, Ke), generator=gen, device=dev)
        ide = torch.stack([torch.randperm(n_exp, generator=gen, device=dev)[:n_used]
                           for _ in range(n_tok)]).to(torch.int32)
        ye = torch.empty((n_tok, n_used, Ne), dtype=torch.float32, device=dev)
        wse = torch.empty(max(1, q.q2_0_mul_mat_id_workspace_size(Ke, n_tok, 1)),
                          dtype=torch.uint8, device=dev)
        mse = timed(lambda: q.q2_0_mul_mat_id(we, n_exp, Ne, Ke, xe, ide, y=ye, workspace=wse,
                                              stream=stream))
        slot_bytes = n_tok * n_used * q.packed_bytes(Ne, Ke)
        distinct = int(torch.unique(ide).numel()) * q.packed_bytes(Ne, Ke)
        moe[f"tokens_{n_tok}"] = {"us": round(mse * 1e3, 2),
                                  "slot_weight_gbs": round(slot_bytes / (mse * 1e-3) / 1e9, 1),
                                  "distinct_expert_gbs": round(distinct / (mse * 1e-3) / 1e9, 1)}
    del we
    return {
        "moe_mul_mat_id_128x768x2048_top8": moe,
        "decode_8b_step_ncols1": {"bytes": bytes8, "us": round(ms8 * 1e3, 2),
                                  "gbs": round(bytes8 / (ms8 * 1e-3) / 1e9, 1),
                                  "hbm_frac": round(bytes8 / (ms8 * 1e-3) / 1e9 / hbm_peak, 4),
                                  "matrices": 253},
        "gemm_split_m2048_8b": {"tflops": round(flops2 / (ms2 * 1e-3) / 1e12, 2),
                                "us": round(ms2 * 1e3, 2),
                                "plan_tflops": round(flops2 / (ms2p * 1e-3) / 1e12, 2),
                                "plan_us": round(ms2p * 1e3, 2),
                                "shapes": [[M2, 4096, 4096], [M2, 12288, 4096], [M2, 4096, 12288]]},
        "gemm_split_m512_per_call": {"tflops": round(gemm_flops_512() / (ms_pc * 1e-3) / 1e12, 2),
                                     "us": round(ms_pc * 1e3, 2), "launches": 9},
        "gemm_split_m512_two_plans": {"tflops": round(gemm_flops_512() / (ms_2p * 1e-3) / 1e12, 2),
                                      "us": round(ms_2p * 1e3, 2), "launches": 6,
                                      "plans": "gate+up, then down"},
        "head_matvec_split_layout_151936x4096": {
            "split_bytes": split_bytes, "us": round(ms_sp * 1e3, 2),
            "gbs": round(head_bytes / (ms_sp * 1e-3) / 1e9, 1),
            "vs_18_byte_layout": round(ms32 / ms_sp, 3),
            "split_layout_us": round(ms_mk * 1e3, 2),
            "split_layout_gbs": round((head_bytes + split_bytes) / (ms_mk * 1e-3) / 1e9, 1)},
        "head_matvec_151936x4096": {"bytes": head_bytes,
                                    "f32_gbs": round(head_bytes / (ms32 * 1e-3) / 1e9, 1),
                                    "f16_gbs": round(head_bytes / (ms16 * 1e-3) / 1e9, 1),
                                    "f32_us": round(ms32 * 1e3, 2), "f16_us": round(ms16 * 1e3, 2)},
        "gemm_f16_m512": {"tflops": round(flops / (msg * 1e-3) / 1e12, 2),
                          "us": round(msg * 1e3, 2),
                          "shapes": gemm_shapes},
        "g128_151936x4096": {"repack_gbs": round(rp_bytes / (ms_rp * 1e-3) / 1e9, 1),
                             "repack_bytes": rp_bytes,
                             "direct_matvec_gbs": round(g128_bytes / (ms_g * 1e-3) / 1e9, 1),
                             "direct_matvec_us": round(ms_g * 1e3, 2)},
        "timing": "CUDA-graph replay, CUDA events on the launching stream, outside the step",
    }


def graph_ms(torch, stream, fn, reps: int = 20, warm: int = 3):
    """Mean time (ms) of one CUDA-graph replay of fn, CUDA events on the stream."""
    with torch.cuda.stream(stream):
        for _ in range(warm):
            fn()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(gr, stream=stream):
            fn()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        gr.replay()
        a.record(stream)
        for _ in range(reps):
            gr.replay()
        b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def graph_ms_each(torch, stream, fn, reps: int = 50):
    """Median time (ms) of single CUDA-graph replays of fn, each bracketed by events."""
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(gr, stream=stream):
            fn()
    ts = []
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            a.record(stream)
            gr.replay()
            b.record(stream)
            b.synchronize()
            ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def measure_configs(torch, q, stream, dev, hbm_peak: float):
    """The workloads of the configurations that the step does not cover, each
    timed as CUDA-graph replays with events on the launching stream:
      - one 2048 x 2048 mat-vec at ncols 1 (1,179,648 packed bytes, below L2):
        the single-launch latency (median of single replays, L2-warm), and
        the streaming rate of a graph of one call per distinct weight copy,
        with enough copies to exceed twice the L2 size (L2-cold);
      - the 1.7B-class decode step (196 matrices, 396,361,728 bytes) at
        ncols 2, 4 and 8, one plan each (ncols 1 is the step's own line);
      - get_rows of 512 seeded ids (about 5 % repeats) from the 151936 x 4096
        table whose first rows hold the edge blocks (d = +-0, subnormal d,
        all code 3, all code 1, d = 65504), against HBM and against the
        replay of one empty-sized kernel (the launch floor).
    Weights of the large cases are drawn on the device (the decode-step
    distribution, other bytes than the host stream)."""
    out = {}
    # ---- one 2048 x 2048 matrix, ncols 1 --------------------------------
    N1 = K1 = 2048
    g = synth.rng(1001)
    w1 = synth.packed_matrix(g, N1, K1, *synth.MATVEC_SMALL_SCALE)
    x1 = torch.from_numpy(synth.activations(g, 1, K1)).to(dev)
    y1 = torch.empty((1, N1), dtype=torch.float32, device=dev)
    ws1 = torch.empty(q.q2_0_mul_mat_vec_workspace_size(K1, 1), dtype=torch.uint8, device=dev)
    wd1 = torch.from_numpy(w1).to(dev)
    lat = graph_ms_each(torch, stream, lambda: q.q2_0_mul_mat_vec_ws(
        wd1, x1, N1, K1, 1, ws1, y=y1, stream=stream))
    l2 = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)) or (129 << 20)
    copies = 2 * l2 // w1.size + 2
    gen = torch.Generator(device=dev)
    gen.manual_seed(SEED + 11)
    wc = synth.packed_matrix_device(torch, gen, copies * N1, K1, *synth.MATVEC_SMALL_SCALE, 0.0,
                                    dev).view(copies, -1)

    def stream_all():
        for c in range(copies):
            q.q2_0_mul_mat_vec_ws(wc[c], x1, N1, K1, 1, ws1, y=y1, stream=stream)

    ms_c = graph_ms(torch, stream, stream_all, reps=5)
    per = ms_c / copies
    out["matvec_2048x2048_ncols1"] = {
        "bytes": int(w1.size), "latency_us": round(lat * 1e3, 2),
        "l2_cold_copies": int(copies), "l2_cold_us_per_call": round(per * 1e3, 2),
        "l2_cold_gbs": round(w1.size / (per * 1e-3) / 1e9, 1),
        "l2_cold_hbm_frac": round(w1.size / (per * 1e-3) / 1e9 / hbm_peak, 4)}
    del wc

    # ---- 1.7B-class decode step at ncols 2, 4, 8 -------------------------
    mats = synth.decode_step_1p7b()
    ws_dec = [synth.packed_matrix_device(torch, gen, m.N, m.K, *synth.DECODE_SCALE,
                                         synth.DECODE_FRAC_CODE3, dev) for _, m in mats]
    dbytes = sum(w.numel() for w in ws_dec)
    sweep = {}
    for nc in (2, 4, 8):
        ents = [(w, torch.randn((nc, m.K), generator=gen, device=dev),
                 torch.empty((nc, m.N), dtype=torch.float32, device=dev), m.N, m.K)
                for (_, m), w in zip(mats, ws_dec)]
        plan = q.MvPlan(ents, nc)
        ms = graph_ms(torch, stream, lambda: plan.execute(stream))
        plan.close()
        gbs = dbytes / (ms * 1e-3) / 1e9
        sweep[f"ncols_{nc}"] = {"us": round(ms * 1e3, 2), "gbs": round(gbs, 1),
                                "hbm_frac": round(gbs / hbm_peak, 4)}
        del ents
    out["decode_1p7b_step"] = {"bytes": dbytes, "matrices": len(mats), **sweep}
    del ws_dec

    # ---- get_rows from the 151936 x 4096 table ---------------------------
    V, H, n_ids = VOCAB, 4096, N_IDS
    table = synth.packed_matrix_device(torch, gen, V, H, *synth.DECODE_SCALE,
                                       synth.DECODE_FRAC_CODE3, dev)
    edges = synth.edge_blocks()
    head = np.arange(len(edges), dtype=np.int32) * 9973 % V
    tv = table.view(V, H // 64, 18)
    for i, r in enumerate(head):   # a whole row of each edge pattern
        tv[int(r)] = torch.from_numpy(np.ascontiguousarray(
            np.broadcast_to(edges[i], (H // 64, 18)))).to(dev)
    ids = torch.from_numpy(synth.token_ids(synth.rng(1005, 2), n_ids, V, 0.05, head)).to(dev)
    rows = torch.empty((n_ids, H), dtype=torch.float32, device=dev)
    ms_r = graph_ms(torch, stream, lambda: q.q2_0_get_rows(table, V, H, ids, out=rows,
                                                           stream=stream), reps=50)
    tiny = torch.zeros(1, device=dev)
    ms_floor = graph_ms(torch, stream, lambda: tiny.fill_(0.0), reps=50)
    rbytes = n_ids * (H // 64) * 18 + n_ids * H * 4
    out["get_rows_151936x4096_512ids"] = {
        "bytes": rbytes, "us": round(ms_r * 1e3, 2),
        "gbs": round(rbytes / (ms_r * 1e-3) / 1e9, 1),
        "hbm_frac": round(rbytes / (ms_r * 1e-3) / 1e9 / hbm_peak, 4),
        "launch_floor_us": round(ms_floor * 1e3, 2),
        "edge_rows": [int(r) for r in head]}
    del table
    out["timing"] = "CUDA-graph replay, CUDA events on the launching stream, outside the step"
    return out


def measure_e2e(args, torch, stream, plan, h_xall, d_xall, d_yall, dec_bytes, make_plan):
    """Decode steps through the public API with host buffers. Every step copies
    its 196 activation vectors from pinned host memory to the device, runs the
    plan, and copies all outputs back to pinned host memory. Steps are
    double-buffered, as a caller streaming steps would run them: step i's
    upload and step i - 1's download run on their own streams while step i - 1
    computes. Timed with CUDA events from before the first upload to after the
    last download."""
    hx = h_xall.pin_memory()
    hy = [torch.empty(d_yall.numel(), dtype=torch.float32).pin_memory() for _ in range(2)]
    dx = [d_xall, torch.empty_like(d_xall)]
    dy = [d_yall, torch.empty_like(d_yall)]
    plans = [plan, make_plan(dx[1], dy[1])]
    s_up = torch.cuda.Stream(device=d_xall.device)
    s_down = torch.cuda.Stream(device=d_xall.device)
    ev_up = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_down = [torch.cuda.Event() for _ in range(2)]
    steps = max(3, min(args.steps, 200))
    first = [True, True]

    def one(i):
        b = i & 1
        with torch.cuda.stream(s_up):
            if not first[b]:
                s_up.wait_event(ev_done[b])      # the buffer's previous step has read x
            dx[b].copy_(hx, non_blocking=True)
            ev_up[b].record(s_up)
        with torch.cuda.stream(stream):
            stream.wait_event(ev_up[b])
            if not first[b]:
                stream.wait_event(ev_down[b])    # the previous download of y[b] is done
            plans[b].execute(stream)
            ev_done[b].record(stream)
        with torch.cuda.stream(s_down):
            s_down.wait_event(ev_done[b])
            hy[b].copy_(dy[b], non_blocking=True)
            ev_down[b].record(s_down)
        first[b] = False

    for i in range(4):
        one(i)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b_ev = torch.cuda.Event(enable_timing=True)
    a.record(s_up)
    for i in range(steps):
        one(i)
    s_up.wait_stream(s_down)
    b_ev.record(s_up)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b_ev) / steps
    plans[1].close()
    return {"value": round(dec_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "h2d_bytes_per_step": hx.numel() * 4, "d2h_bytes_per_step": hy[0].numel() * 4,
            "ms_per_step": round(ms, 5), "steps": steps,
            "what": "decode steps: per step one pinned H2D of the 196 activation vectors, the "
                    "plan, one D2H of all outputs; double-buffered, uploads and downloads on "
                    "their own streams overlapping the neighbouring steps' plans"}


# ---------------------------------------------------------------------------
# CPU oracle timings (baseline leg and the reference arm)
# ---------------------------------------------------------------------------
class OracleDecodeSample:
    """The CPU oracle's mat-vec over the decode step's matrices, taken in step order
    and continuing cyclically from call to call; each call runs whole matrices
    until about budget_s seconds of CPU time are spent."""

    def __init__(self):
        import oracle
        oracle.build()
        self.oracle = oracle
        self.dec = decode_inputs(1)
        self.cursor = 0

    def run(self, budget_s: float):
        done_bytes, spent, n = 0, 0.0, 0
        while spent < budget_s or n == 0:
            m, w, x = self.dec[self.cursor]
            self.cursor = (self.cursor + 1) % len(self.dec)
            t0 = time.perf_counter()
            self.oracle.matmul(w, m.N, m.K, x)
            spent += time.perf_counter() - t0
            done_bytes += w.size
            n += 1
        return done_bytes, spent, n


def cpu_baseline(budget_s: float):
    s = OracleDecodeSample()
    b, t, n = s.run(budget_s)
    return {"value": round(b / t / 1e9, 4), "unit": "GB/s", "cores": s.oracle.num_threads(),
            "kind": "oracle",
            "sample": f"fp64 oracle mat-vec over {n} matrices of the decode step, in step order "
                      f"({b} packed bytes, {t:.1f} s of CPU time), OpenMP over rows"}


def run_reference(args):
    """The CPU oracle on the same workload and metric; the run is time-boxed to
    about --cpu-seconds * 6 in total whatever --steps/--warmup are."""
    rank, world, _ = dist_env()
    if rank != 0:
        return
    s = OracleDecodeSample()
    budget = max(0.01, 6.0 * args.cpu_seconds / (args.steps + args.warmup))
    for _ in range(args.warmup):
        s.run(budget)
    tot_b, tot_s, nmat = 0, 0.0, 0
    for _ in range(args.steps):
        b, t, n = s.run(budget)
        tot_b += b
        tot_s += t
        nmat += n
    value = tot_b / tot_s / 1e9
    sample = (f"each step: oracle mat-vec over ~{nmat / args.steps:.1f} decode-step matrices "
              f"(about {budget:.2f} s of CPU time), continuing through the step in order")
    line = {
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_s / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (CPU oracle)",
        "data": "synthetic (seeded; no trained weights)",
        "config": {"workload": WORKLOAD, "ncols": 1, "sample": sample},
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s",
                         "cores": s.oracle.num_threads(), "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the side measurements (head mat-vec F32/F16, F16 GEMM)")
    ap.add_argument("--ncols", type=int, default=1, choices=range(1, 9),
                    help="activation columns of the decode step (the headline runs 1)")
    ap.add_argument("--only", choices=["all", "decode", "gemm", "get_rows"], default="all",
                    help="run one part of the step (for profiling); the JSON line is the "
                         "benchmark only with the default 'all'")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
