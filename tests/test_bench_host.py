"""bench.py host logic on the CPU: byte/FLOP model, roofline, peaks, clock
parsing, the committed-traffic lookup and the max-over-ranks timing with two
gloo ranks."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from dense_gemm_08_gb300.inputs import WORKLOADS
from golden.fixtures import read as read_fixture


def test_algorithmic_bytes_match_the_pages_and_the_configs():
    g = read_fixture("p5_4096_fp32_traffic.txt")
    # FP32 n^3, inputs read once, output written once: 12 n^2 bytes
    assert bench.algorithmic_bytes(4096, 4096, 4096, 4, 0.0) == int(g["Q_one_pass"])
    assert bench.algorithmic_bytes(8192, 8192, 8192, 2, 0.0) == 536_870_912
    mlp = WORKLOADS["bf16_mlp"]
    assert bench.algorithmic_bytes(mlp.M, mlp.N, mlp.K, 2, mlp.beta) == 1_124_073_472
    assert bench.algorithmic_bytes(4095, 4097, 1000, 4, -0.25) == 166_985_720
    assert bench.algorithmic_bytes(4095, 4097, 1000, 2, -0.25) == 150_601_720
    assert bench.algorithmic_bytes(1, 4096, 4096, 2, -0.25) == 33_595_392
    assert WORKLOADS["f32_4096"].flops == int(g["flops"])
    assert WORKLOADS["bf16_8192"].flops == 1_099_511_627_776
    assert WORKLOADS["bf16_mlp"].flops == 962_072_674_304


def test_roofline_is_min_of_peak_and_intensity_times_bandwidth():
    # intensity 0.5 FLOP/B at 6680.8 GB/s -> 3.34 TFLOP/s, below any peak
    assert bench.roofline_tflops(1.0, 2.0, 1886.0, 6680.8) == pytest.approx(3.3404)
    assert bench.roofline_tflops(2048.0, 1.0, 1886.0, 6680.8) == 1886.0
    # the page's hypothetical machine: P = 20 TFLOP/s, BW = 1 TB/s, T = 64 tile
    q64 = 8657043456
    assert bench.roofline_tflops(137438953472, q64, 20.0, 1000.0) == pytest.approx(15.875969, abs=1e-6)


def test_hbm_bound_shapes_report_against_bandwidth():
    compute = {"bound": "alu", "achieved": 0.3, "peak": 80.5, "unit": "TFLOP/s", "frac": 0.3 / 80.5}
    # FP32 1 x 4096 x 4096, beta != 0: 67,158,016 B in 20 us -> 3357.9 GB/s
    alg = bench.algorithmic_bytes(1, 4096, 4096, 4, -0.25)
    flops = 2 * 4096 * 4096
    roof_t = bench.roofline_tflops(flops, alg, 80.5, 6680.8)
    r = bench.hbm_bound_roof(dict(compute), alg, 20e-6, 6680.8, "measured", roof_t)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(alg / 20e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6680.8)
    assert r["compute"]["bound"] == "alu"
    # a compute-bound shape keeps its compute roofline
    big = bench.algorithmic_bytes(4096, 4096, 4096, 4, 0.0)
    roof_t = bench.roofline_tflops(2 * 4096 ** 3, big, 80.5, 6680.8)
    assert bench.hbm_bound_roof(dict(compute), big, 2.4e-3, 6680.8, "measured", roof_t) == compute


def test_fp32_peak_formula():
    assert bench.fp32_core_peak_tflops(152, 2070.0) == pytest.approx(80.54784)


def test_clock_summary():
    rows = [{"sm": 2070.0, "max": 2070.0, "power": 150.0, "reasons": []},
            {"sm": 1900.0, "max": 2070.0, "power": 1200.0, "reasons": ["sw_power_cap"]},
            {"sm": 1950.0, "max": 2070.0, "power": 1100.0, "reasons": []}]
    c = bench.clock_summary(rows)
    assert c["sm_mhz"] == 1925.0 and c["sm_max_mhz"] == 2070.0
    assert c["reasons"] == ["sw_power_cap"]
    assert bench.clock_summary([]) is None


def test_committed_traffic_needs_matching_source(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    (tmp_path / "profiles").mkdir()
    src = tmp_path / "k.cu"
    src.write_text("kernel v1")
    monkeypatch.setitem(bench.KERNEL_SOURCES, "kern", "k.cu")
    digest = bench.source_digest("k.cu")
    (tmp_path / "profiles" / "kern_w_traffic.md").write_text(
        f"traffic_bytes_per_launch: 123456\nsource_sha256_16: {digest}\n")
    assert bench.committed_traffic("kern", "w") == 123456.0
    src.write_text("kernel v2")  # the kernel changed since the capture
    assert bench.committed_traffic("kern", "w") is None
    assert bench.committed_traffic("kern", "other") is None


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [3.5, 7.25][rank]
        got = bench.max_over_ranks(elapsed, world, torch.device("cpu"))
        bench.barrier(world)
        out[rank] = got
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert dict(out) == {0: 7.25, 1: 7.25}


def test_rotation_copies_exceed_twice_l2():
    l2 = bench.L2_BYTES
    # FP32 256^3: A, B and D of 256 KiB each
    ws = 3 * 256 * 256 * 4
    n = bench.rotation_copies(ws, l2)
    assert n * ws >= 2 * l2 and (n - 1) * ws < 2 * l2
    # FP32 4096^3 (192 MiB) needs two copies; BF16 8192^3 (512 MiB) needs none
    assert bench.rotation_copies(192 * 2**20, l2) == 2
    assert bench.rotation_copies(512 * 2**20, l2) == 1
    assert bench.rotation_copies(2 * l2, l2) == 1


def test_region_clocks_take_the_samples_inside_the_timed_region():
    nvml = [{"t": 10.000, "sm": 1500.0, "max": 2070.0, "power": 200.0, "reasons": []},
            {"t": 10.004, "sm": 2070.0, "max": 2070.0, "power": 900.0, "reasons": []},
            {"t": 10.005, "sm": 2055.0, "max": 2070.0, "power": 1100.0,
             "reasons": ["sw_power_cap"]},
            {"t": 10.006, "sm": 2040.0, "max": 2070.0, "power": 1200.0, "reasons": []},
            {"t": 10.050, "sm": 1200.0, "max": 2070.0, "power": 150.0,
             "reasons": ["hw_slowdown"]}]
    smi = [{"t": 9.95, "sm": 1400.0, "max": 2070.0, "power": 180.0, "reasons": []}]
    c = bench.region_clocks(nvml, smi, 10.003, 10.010)
    assert c["samples"] == 3 and c["sm_mhz"] == 2055.0 and c["sm_mhz_min"] == 2040.0
    assert c["reasons"] == ["sw_power_cap"]  # the slowdown came after the region
    assert c["power_w_max"] == 1200.0 and c["sm_max_mhz"] == 2070.0
    assert c["source"].startswith("NVML")
    # no NVML samples: the run-wide nvidia-smi summary stands in
    c = bench.region_clocks([], smi, 10.003, 10.010)
    assert c["samples"] == 0 and c["sm_mhz"] == 1400.0


def test_reference_arm_prints_the_same_config_as_ours():
    w = WORKLOADS["bf16_8192"]
    ours = bench.workload_config(w, queue="gpu", l2="x")
    ref = bench.workload_config(w, queue="cpu")
    shared = set(ours) & set(ref)
    assert {"workload", "M", "N", "K", "alpha", "beta", "in_dtype", "acc_dtype", "out_dtype",
            "order_a", "order_b", "order_cd", "inputs"} <= shared
    assert all(ours[k] == ref[k] for k in shared if k != "queue")
    assert ours["order_b"] == "col" and ours["in_dtype"] == "bf16"


def test_pipeline_depth_fits_recover_their_models():
    # exact data of each model: the fit returns its parameters
    S = [2, 3, 4, 5, 6]
    P, kappa, rms = bench.fit_saturating(S, [2000 * s / (s + 1.5) for s in S])
    assert P == pytest.approx(2000, rel=1e-4) and kappa == pytest.approx(1.5, rel=1e-4)
    assert rms < 1e-3
    P, b, rms = bench.fit_littles_law(S, [min(1800.0, 400.0 * s) for s in S])
    assert P == pytest.approx(1800.0) and b == pytest.approx(400.0) and rms < 1e-9


def test_committed_pipeline_depth_sweep_refits_to_its_stated_fits():
    import re
    path = os.path.join(bench.ROOT, "profiles", "gemm_bf16_tc_pipeline_depth_sweep.md")
    text = open(path).read()
    stages = eval(re.search(r"^stages: (\[.*\])$", text, re.M).group(1))
    for wl in ("bf16_8192", "bf16_mlp"):
        med = eval(re.search(rf"^{wl}_tflops_median: (\[.*\])$", text, re.M).group(1))
        sat = dict(re.findall(r"(\w+)=([0-9.]+)",
                              re.search(rf"^fit_{wl}_saturating: (.*)$", text, re.M).group(1)))
        lit = dict(re.findall(r"(\w+)=([0-9.]+)",
                              re.search(rf"^fit_{wl}_littles_law: (.*)$", text, re.M).group(1)))
        P, kappa, rms = bench.fit_saturating(stages, med)
        assert P == pytest.approx(float(sat["P"]), rel=1e-3)
        assert kappa == pytest.approx(float(sat["kappa"]), rel=1e-3)
        assert rms == pytest.approx(float(sat["rms"]), rel=1e-3)
        P, b, rms = bench.fit_littles_law(stages, med)
        assert P == pytest.approx(float(lit["P"]), rel=1e-4)
        assert b == pytest.approx(float(lit["b"]), rel=1e-4)
        assert rms == pytest.approx(float(lit["rms"]), rel=1e-3)
        # the piecewise bound fits the measurements better than the smooth curve
        assert rms < float(sat["rms"])


def test_bf16_formula_peak():
    # 152 SMs x 8192 FLOP per clock x 2070 MHz
    assert bench.bf16_formula_tflops(152, 2070.0) == pytest.approx(2577.5, abs=0.1)
