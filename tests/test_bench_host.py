"""Host logic of bench.py, on the CPU: the multi-rank reduction (gloo,
world size 2), the whole-job aggregate, the clock-sample parser and the
reference (oracle) arm's JSON line."""
import json
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    w, r, _ = bench.dist_env()
    dist = bench.init_dist(w, "gloo")
    my_ms = 10.0 + 5.0 * r          # rank 1 is the slowest
    bench.barrier(dist)
    worst = bench.max_over_ranks(dist, my_ms)
    value = bench.aggregate_tflops(1e12, 4, w, worst)
    with open(os.path.join(out_dir, "rank%d.json" % r), "w") as fh:
        json.dump({"worst": worst, "value": value}, fh)
    dist.destroy_process_group()


def test_two_rank_max_and_aggregate(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(world)]
    for r in res:
        assert r["worst"] == 15.0
        # 2 ranks x 4 steps x 1 TFLOP in 15 ms
        assert r["value"] == pytest.approx(2 * 4 * 1e12 / 15e-3 / 1e12)


def test_single_rank_helpers():
    assert bench.max_over_ranks(None, 3.5) == 3.5
    assert bench.aggregate_tflops(2.0 * 8192 ** 3, 10, 1, 6.0) == pytest.approx(
        2.0 * 8192 ** 3 * 10 / 6e-3 / 1e12)


def test_clock_parser():
    s = bench.ClockSampler(0)
    s.proc = type("P", (), {"terminate": lambda self: None, "wait": lambda self, timeout: 0})()
    s.t0, s.t1 = 100.0, 101.0
    row = "2026/12/02 10:00:00.000, 0, {mhz}, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, {pc}"
    s.lines = [(100.2, row.format(mhz=1800, pc="Active")), (100.5, row.format(mhz=1900, pc="Not Active")),
               (100.8, row.format(mhz=2000, pc="Not Active")), (300.0, row.format(mhz=10, pc="Not Active"))]
    out = s.stop()
    assert out["sm_mhz"] == 1900 and out["sm_max_mhz"] == 2070
    assert out["reasons"] == ["sw_power_cap"] and out["samples_in_window"] == 3


def test_fp32_alu_peak():
    assert bench.fp32_alu_peak_tflops(152, 2070.0) == pytest.approx(152 * 256 * 2.07e9 / 1e12)


def test_reference_arm_line(capsys):
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["metric"] == bench.METRIC
