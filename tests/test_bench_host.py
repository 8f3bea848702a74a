"""Host logic of bench.py without a GPU: the max/sum reductions over ranks with
two gloo processes, the clock-sample parser, the traffic bookkeeping and the
prefill part's inputs."""
import json
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    os.environ["RANK"] = str(rank)
    os.environ["WORLD_SIZE"] = str(world)
    os.environ["LOCAL_RANK"] = str(rank)
    r, w, lr = bench.dist_env()
    assert (r, w, lr) == (rank, world, rank)
    d = bench.init_dist(world, "gloo")
    mx = bench.reduce_max(d, 1.5 + rank)          # 1.5, 2.5 -> 2.5
    sm = bench.reduce_sum(d, 10.0 * (rank + 1))   # 10 + 20 -> 30
    d.barrier()
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"max": mx, "sum": sm}, f)
    d.destroy_process_group()


def test_reductions_over_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        got = json.load(open(tmp_path / f"r{r}.json"))
        assert got == {"max": 2.5, "sum": 30.0}


def test_single_rank_reductions_are_identity():
    assert bench.reduce_max(None, 3.0) == 3.0
    assert bench.reduce_sum(None, 4.0) == 4.0


def test_clock_sampler_parser(tmp_path, monkeypatch):
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "c.csv")
    with open(cs.path, "w") as f:
        f.write("0, 2070, 2070, 900.1, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 1950, 2070, 1300.0, 0x4, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 2010, 2070, 1200.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")

    class _P:
        def terminate(self):
            pass

        def wait(self, timeout=None):
            return 0

    cs.proc = _P()
    cs.fh = open(str(tmp_path / "dummy"), "w")
    got = cs.stop()
    assert got["sm_mhz"] == 2010 and got["sm_max_mhz"] == 2070
    assert got["reasons"] == ["sw_power_cap"] and got["samples"] == 3


def test_committed_traffic_tracks_sources():
    p = os.path.join(bench.ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        pytest.skip("no committed traffic counters")
    data = json.load(open(p))
    for name, entry in data.items():
        got = bench.committed_traffic(name)
        fresh = bench.source_sha256(entry["sources"]) == entry["sha256"]
        assert (got is not None) == fresh


def test_prefill_inputs_share_x_between_gate_and_up():
    """The prefill part's workload: gate and up read one X (M x 2048), down its
    own (M x 6144); the device entries copy a shared X once and every entry
    carries its own output of M x N."""
    gm = bench.gemm_inputs()
    names = [n for n, *_ in gm]
    assert names == ["gate", "up", "down"]
    (_, Ng, Kg, wg, xg), (_, Nu, Ku, wu, xu), (_, Nd, Kd, wd, xd) = gm
    assert (Ng, Kg, Nu, Ku, Nd, Kd) == (6144, 2048, 6144, 2048, 2048, 6144)
    assert xg is xu and xd is not xg
    assert xg.shape == (bench.PREFILL_M, 2048) and xd.shape == (bench.PREFILL_M, 6144)
    assert wg.size == 6144 * 2048 // 64 * 18 and not (wg == wu).all()
    ents = bench.gemm_device_entries(torch, torch.device("cpu"), gm, bench.PREFILL_M)
    assert ents[0][1] is ents[1][1] and ents[2][1] is not ents[0][1]
    assert [tuple(e[2].shape) for e in ents] == [(bench.PREFILL_M, 6144)] * 2 + [(bench.PREFILL_M, 2048)]
    assert [e[3:] for e in ents] == [(6144, 2048, bench.PREFILL_M)] * 2 + [(2048, 6144, bench.PREFILL_M)]
    assert bench.gemm_flops_512() == 2.0 * bench.PREFILL_M * (2 * 6144 * 2048 + 2048 * 6144)
