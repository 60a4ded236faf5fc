"""Host-side checks of bench.py's accounting (no GPU): the roofline of each step
kind, the algorithmic work credited to each kernel, and the peaks it divides by.

The expected values are written out from the definitions (bytes read once and
written once, 2 flops per multiply-add), not recomputed with bench.py's code.
"""
import importlib.util
import json
import os

import pytest

from dynamic_dilated_depthwise_gb300.inputs import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


PEAKS = {"hbm_gbs": 5000.0, "bf16_tflops": 2000.0, "bf16_tflops_sustained": 1800.0, "sm_max_mhz": 2000.0,
         "source": "test"}


def test_train_roofline_headline(bench):
    p = WORKLOADS["b1_c64_256x256_k3"]
    P, C, O = 65536, 64, 1728
    r = bench.step_roofline_us(p, 2, PEAKS, "train")
    flops = 4 * 2 * O * C * P                       # generator, recompute for dX, dY, dW
    nbytes = P * 6 * C * 2 + P * 8 * C * 2 + 4 * (O * C + O) * 2
    assert r["flops"] == flops
    assert r["bytes"] == nbytes
    assert r["tensor_us"] == pytest.approx(flops / 2000e12 * 1e6)
    assert r["hbm_us"] == pytest.approx(nbytes / 5000e9 * 1e6)
    assert r["roofline_us"] == pytest.approx(max(r["tensor_us"], r["hbm_us"]))
    # 57.98 GFLOP at the bf16 peak dominates 118 MB at the HBM peak
    assert r["roofline_us"] == r["tensor_us"]


def test_forward_and_filter_rooflines(bench):
    p = WORKLOADS["b1_c64_128x128_k5"]
    P, C, O = 16384, 64, 4800
    f = bench.step_roofline_us(p, 2, PEAKS, "forward")
    assert f["flops"] == 2 * O * C * P
    assert f["bytes"] == P * (2 * C + 4 * C) * 2 + (O * C + O) * 2
    t = bench.step_roofline_us(p, 4, PEAKS, "filter")
    assert t["flops"] == 0
    assert t["bytes"] == P * (C + O + 4 * C) * 4      # x and the taps in, 4C channels out
    assert t["roofline_us"] == pytest.approx(t["bytes"] / 5000e9 * 1e6)
    # filter fwd+bwd: x, taps and grad (4C) in; out (4C), dx (C) and dtaps (O) out
    ft = bench.step_roofline_us(p, 2, PEAKS, "filter_train")
    assert ft["flops"] == 0 and ft["bytes"] == P * (10 * C + 2 * O) * 2


def test_kernel_work(bench):
    p = WORKLOADS["b1_c64_256x256_k3"]
    P, C, O = 65536, 64, 1728
    assert bench.kernel_work("forward_tc", p, 2, 10) == ("tensor", 2.0 * O * C * P, "flops")
    assert bench.kernel_work("bwd_dx_tc_packed", p, 2, 10) == ("tensor", 2.0 * O * C * P, "flops")
    assert bench.kernel_work("bwd_dw_partial_simt", p, 4, 16) == ("alu", 2.0 * O * (C + 1) * P, "flops")
    assert bench.kernel_work("filter_pregenerated_simt", p, 2, 1) == ("hbm", P * (O + 5 * C) * 2, "bytes")
    assert bench.kernel_work("bwd_dw_reduce", p, 2, 10) == ("hbm", 10 * O * (C + 1) * 4 + O * (C + 1) * 2,
                                                            "bytes")
    assert bench.kernel_work("filter_bwd_dx", p, 2, 1) == ("hbm", P * (O + 5 * C) * 2, "bytes")
    assert bench.kernel_work("bwd_dw_tf32", p, 4, 16) == ("tensor_tf32", 2.0 * O * (C + 1) * P, "flops")
    assert bench.kernel_work("filter_bwd_dtaps", p, 4, 1) == ("hbm", P * (4 * C + O) * 4, "bytes")
    assert bench.kernel_work("no_such_kernel", p, 2, 1)[0] == "unknown"


def test_fp32_alu_ceiling(bench):
    # 152 SMs x 128 FP32 lanes x 2 flops x 2.07 GHz
    assert bench.fp32_alu_tflops({"sm_max_mhz": 2070.0}) == pytest.approx(80.5, abs=0.1)


def test_peaks_from_measured_file(bench):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    pk = bench.load_peaks()
    if os.path.exists(path):
        m = json.load(open(path))
        assert pk["source"] == "measured"
        assert pk["hbm_gbs"] == float(m["hbm_gbs"]) and pk["bf16_tflops"] == float(m["bf16_tflops"])
    else:
        assert pk["source"] == "fallback" and pk["hbm_gbs"] == 6800.0


def test_step_metrics_share_the_unit(bench):
    assert set(bench.STEP_METRIC) == {"train", "forward", "filter", "filter_train"}
    assert bench.STEP_METRIC["train"] == bench.METRIC


def test_stored_traffic_is_keyed_per_kernel(bench):
    # kernels sharing a source file share a digest; different files give different digests
    assert bench.kernel_source_digest("pack_chunks") == bench.kernel_source_digest("bwd_dx_tc_packed")
    assert bench.kernel_source_digest("bwd_dy_tc") != bench.kernel_source_digest("bwd_dw_tc")
    assert bench.kernel_source_digest("no_such_kernel") == "missing"
    t = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    for name, k in t["kernels"].items():
        want = k["dram_bytes_per_launch"] if k["source_digest"] == bench.kernel_source_digest(name) else None
        assert bench.stored_traffic(name, k["workload"]) == want
        assert bench.stored_traffic(name, "another_workload") is None
