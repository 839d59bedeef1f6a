"""The benchmark's roofline denominators and summaries, on the host: which peak a timed region is compared
with, the clock-normalised peak, the step-time percentiles and the committed DRAM-traffic lookup."""
import json
import os

import numpy as np
import pytest

import bench

PK = {"bf16_tflops": 1946.7, "bf16_tflops_sustained": 1744.3, "hbm_gbs": 6794.8}


def test_short_regions_use_the_burst_peak():
    assert bench.tensor_peak(PK, 0.072) == (1946.7, "burst")
    assert bench.tensor_peak(PK, bench.SUSTAINED_AFTER_S - 1e-6) == (1946.7, "burst")


def test_long_regions_use_the_sustained_peak():
    assert bench.tensor_peak(PK, bench.SUSTAINED_AFTER_S) == (1744.3, "sustained")
    assert bench.tensor_peak(PK, 4.0) == (1744.3, "sustained")


def test_sustained_peak_missing_falls_back_to_burst():
    pk = {"bf16_tflops": 1900.0}
    assert bench.tensor_peak(pk, 10.0) == (1900.0, "burst")


def test_fp8_peak_is_twice_the_bf16_peak_of_the_same_kind():
    peak, kind = bench.tensor_peak(PK, 0.1, dtype_factor=2.0)
    assert peak == pytest.approx(2 * 1946.7)
    assert kind == "2 x bf16 burst"


def test_clock_peak_is_flops_per_clock_times_sms_times_clock():
    # 8192 flop/clk/SM x 152 SMs x 2070 MHz
    assert bench.clock_peak(152, 2070.0) == pytest.approx(8192 * 152 * 2.07e9 / 1e12)
    assert bench.clock_peak(152, 1500.0, dtype_factor=2.0) == pytest.approx(2 * 8192 * 152 * 1.5e9 / 1e12)
    assert bench.clock_peak(152, None) is None
    assert bench.clock_peak(0, 2070.0) is None


def test_percentiles_of_step_times():
    ms = [float(x) for x in range(1, 101)]  # 1 .. 100
    p = bench.percentiles(ms)
    assert p["median"] == pytest.approx(np.median(ms))
    assert p["p10"] == pytest.approx(np.percentile(ms, 10))
    assert p["p90"] == pytest.approx(np.percentile(ms, 90))
    assert p["p10"] <= p["median"] <= p["p90"]


def test_traffic_lookup_follows_the_source_digest():
    path = os.path.join(bench.ROOT, "profiles", "dram_traffic.json")
    with open(path) as fh:
        table = json.load(fh)
    workload = table["workload"]
    for name, entry in table["segments"].items():
        got = bench.measured_traffic(name, workload)
        if entry["source_digest"] == bench.kernel_source_digest(name):
            assert got == entry["bytes_per_launch"]
            assert entry["bytes_per_launch"] == pytest.approx(entry["read"] + entry["write"])
        else:
            assert got is None  # a kernel changed since its capture reads as unmeasured
        assert bench.measured_traffic(name, workload + "_other") is None
    assert bench.measured_traffic("no_such_segment", workload) is None


def test_step_work_per_segment():
    from tensor_transformer_mlp_tp_gb300 import inputs
    w = inputs.WORKLOADS["sp_block_fwd_bwd"]  # T = 8192, d = 4096, F = 16384, N = 8
    segs = {name: (n, work, unit) for name, n, work, unit in bench.Step.kernels_of(w)}
    gemm = 2.0 * 8192 * 4096 * 16384  # 1.1 TFLOP
    assert [s for s in segs if s.startswith("gemm")] == [
        "gemm1_bias_gelu", "gemm2_shard_accum_rs_store", "gemm_dh_geluprime", "gemm_wgrad_b", "gemm_wgrad_a",
        "gemm_dx_shard_accum"]
    assert all(segs[s] == (1, gemm, "F") for s in segs if s.startswith("gemm"))
    assert segs["layernorm_gather"] == (1, 4.0 * 8192 * 4096, "B")      # read x, write the gathered row (bf16)
    assert segs["layernorm_backward"] == (2, 6.0 * 8192 * 4096, "B")    # read x, dy, write dx; two launches
    assert bench.useful_flops(w) == 6 * gemm


def test_forward_workloads_count_two_gemms():
    from tensor_transformer_mlp_tp_gb300 import inputs
    for name in ("gpt2_medium_fwd", "mlp7b_fwd", "sp_large_fwd"):
        w = inputs.WORKLOADS[name]
        names = [s[0] for s in bench.Step.kernels_of(w)]
        assert sum(n.startswith("gemm") for n in names) == 2
        assert ("layernorm_gather" in names) == w.sp
        assert bench.useful_flops(w) == 2 * 2.0 * w.T * w.d * w.F
