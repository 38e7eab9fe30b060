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
    # a window that was opened but never closed: every sample is used, no error
    s.t1 = None
    out = s.stop()
    assert out["samples_in_window"] == 0 and out["samples"] == 4


def test_fp32_alu_peak():
    assert bench.fp32_alu_peak_tflops(152, 2070.0) == pytest.approx(152 * 256 * 2.07e9 / 1e12)


def test_reference_arm_line(capsys):
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["metric"] == bench.METRIC
    # the same workload as this library's arm, which adds its own keys to it
    cfg = dict(line["config"])
    assert cfg.pop("accumulate") == "f64 (the oracle)"
    assert cfg == bench.workload_config(1)
    assert line["higher_is_better"] is True and line["scaling"] == "weak"


def test_traffic_only_while_the_kernel_matches_its_profile(tmp_path, monkeypatch):
    """The line's roofline.traffic comes from the committed ncu summary and is
    reported only while the kernel's sources hash to the value recorded there;
    after any change to them it is null."""
    csrc = tmp_path / "dense_gemm_tcgen05_gb300" / "csrc"
    csrc.mkdir(parents=True)
    for name in bench.KERNEL_SOURCES:
        (csrc / name).write_text("// %s\n" % name)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    summary = tmp_path / "profiles" / "tc_gemm_f16_8192.txt"
    summary.write_text("kernel_source_sha256: %s\ntraffic_bytes_per_launch: 1259031552\n"
                       % bench.kernel_source_hash())
    assert bench.load_traffic() == 1259031552
    (csrc / bench.KERNEL_SOURCES[0]).write_text("// changed\n")
    assert bench.load_traffic() is None
    summary.unlink()
    assert bench.load_traffic() is None


def test_committed_profile_names_its_traffic():
    """The committed FP16 8192^3 summary carries the two fields the bench reads."""
    fields = {}
    for line in open(os.path.join(bench.ROOT, "profiles", "tc_gemm_f16_8192.txt")):
        if ":" in line:
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    assert len(fields["kernel_source_sha256"]) == 64
    assert int(float(fields["traffic_bytes_per_launch"])) > 384 << 20   # above the compulsory bytes


def test_compulsory_bytes():
    """A and B read once, C written once: 384 MiB at FP16 8192^3, 256 MiB for
    FP8 8192^3 with BF16 output, 384 MiB with FP32 output, about 22.6 MB for
    the ragged BF16 2047 x 3001 x 1023 case."""
    assert bench.compulsory_bytes("f16", 8192, 8192, 8192) == 384 << 20
    assert bench.compulsory_bytes("e4m3", 8192, 8192, 8192) == 256 << 20
    assert bench.compulsory_bytes("e4m3", 8192, 8192, 8192, out_f32=True) == 384 << 20
    assert bench.compulsory_bytes("bf16", 2047, 3001, 1023) == (2047 * 1023 + 3001 * 1023 +
                                                                2047 * 3001) * 2


def test_cpu_baseline_reports_all_cores_and_one():
    """The CPU baseline times the oracle on all its threads, then on one, and
    leaves the thread count as it found it."""
    import oracle

    before = oracle.num_threads()
    r = bench.cpu_baseline(M=256, N=256, K=256, budget_s=0.05, one_core_budget_s=0.05)
    assert r["kind"] == "oracle" and r["cores"] == before and r["value"] > 0
    assert r["one_core"]["cores"] == 1 and r["one_core"]["value"] > 0
    assert oracle.num_threads() == before


def test_tensor_peak_follows_the_window():
    """Burst for a short window or one without the power cap; sustained only
    for a window of seconds in which the sampler saw sw_power_cap."""
    burst, sustained = 1914.3, 1748.8
    # a driver-style run: 20 launches, 12 ms, clocks at max, no reason
    peak, regime, why = bench.tensor_peak(12.0, {"reasons": []}, burst, sustained)
    assert (peak, regime) == (burst, "burst") and "12 ms" in why
    assert 1837.6 / peak == pytest.approx(0.96, abs=0.001)
    # short, even if capped
    assert bench.tensor_peak(100.0, {"reasons": ["sw_power_cap"]}, burst, sustained)[1] == "burst"
    # long but not capped
    peak, regime, why = bench.tensor_peak(3000.0, {"reasons": []}, burst, sustained)
    assert regime == "burst" and "no sw_power_cap" in why
    # long and capped: the default 1000-step loop (0.67 s) at the power cap
    peak, regime, _ = bench.tensor_peak(667.0, {"reasons": ["sw_power_cap"]}, burst, sustained)
    assert (peak, regime) == (sustained, "sustained")
    # no clock record at all
    assert bench.tensor_peak(5000.0, None, burst, sustained)[1] == "burst"


def test_per_config_sets_exceed_l2():
    """Every per-configuration shape rotates over input sets whose bytes
    together exceed twice the 129 MB L2, with at least three sets."""
    for kind, (M, N, K), f32, _, _ in bench.PER_CONFIG:
        n = bench.sets_beyond_l2(kind, M, N, K, f32)
        assert n >= 3 and n * bench.compulsory_bytes(kind, M, N, K, f32) >= 2 * bench.L2_BYTES
    assert bench.sets_beyond_l2("bf16", 2047, 3001, 1023) == 12    # 22.6 MB a set
    shapes = {(k, s, f) for k, s, f, _, _ in bench.PER_CONFIG}
    for shape in [(4096, 4096, 4096), (4096, 14336, 4096), (4096, 4096, 14336),
                  (2047, 3001, 1023), (8191, 8191, 8191)]:
        assert ("bf16", shape, False) in shapes                    # the BF16 configuration
    for shape in [(8192, 8192, 8192), (4096, 14336, 4096), (16384, 4096, 4096)]:
        assert ("e4m3", shape, False) in shapes                    # the FP8 configuration
    for shape in [(8192, 8192, 8192), (8192, 28672, 8192), (8192, 10240, 8192),
                  (3072, 4096, 8192)]:
        assert ("e4m3", shape, True) in shapes                     # the FP8 page's Tables 1-4


def test_spread():
    s = bench.spread([1.0, 3.0, 2.0, 4.0])
    assert (s["mean_ms"], s["median_ms"], s["min_ms"], s["max_ms"], s["launches"]) == (
        2.5, 2.5, 1.0, 4.0, 4)


def test_ncu_case_spec():
    """--ncu-case: KIND:MxNxK with an optional third field of library options;
    workspace=0 drops the bench workspace."""
    assert bench.parse_ncu_case("bf16:128x8192x8192") == ("bf16", 128, 8192, 8192, {}, True)
    assert bench.parse_ncu_case("f16:16x8192x8192:half=3,workspace=0") == \
        ("f16", 16, 8192, 8192, {"half": 3}, False)
    assert bench.parse_ncu_case("e4m3:64X512X256:tile_q=192,pair=1") == \
        ("e4m3", 64, 512, 256, {"tile_q": 192, "pair": 1}, True)
    for bad in ("bf16", "bf16:1x2", "bf16:1x2x3:half", "bf16:1x2x3:a=1:b=2"):
        with pytest.raises(ValueError):
            bench.parse_ncu_case(bad)
