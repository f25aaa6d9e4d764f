"""Host arithmetic of bench.py on CPU: the roofline figures, the per-launch
DRAM traffic lookup and the clock-sample summary."""
import os

import pytest

import bench
import workloads

PEAKS = {"hbm_gbs": 6000.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1600.0}


def test_hbm_kernel_roofline_uses_algorithmic_bytes():
    wl = workloads.WORKLOADS["c4"]
    te = wl.B * wl.H * wl.n * wl.d * wl.elem_bytes
    # 10 launches of the token kernel in 0.5 ms: 50 us per launch, 3 T e bytes each
    r = bench.roofline_for("tokens_tc", 0.5, 10, 1, wl, PEAKS, "measured")
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["algorithmic_bytes"] == 3 * te
    assert r["achieved"] == pytest.approx(3 * te / 50e-6 / 1e9)
    assert r["frac"] == pytest.approx(r["achieved"] / 6000.0)


def test_head_groups_split_the_bytes_of_a_launch():
    wl = workloads.WORKLOADS["c2"]
    one = bench.roofline_for("rows_tc", 1.0, 10, 1, wl, PEAKS, "measured")
    two = bench.roofline_for("rows_tc", 1.0, 10, 2, wl, PEAKS, "measured")
    assert two["algorithmic_bytes"] == one["algorithmic_bytes"] / 2


def test_pseudo_inverse_roofline_is_tf32_of_the_burst_peak():
    """Per-kernel times are short event-timed launches: the burst bf16 peak,
    scaled to tf32 by the nominal ratio (m <= 128: every product is tf32)."""
    wl = workloads.WORKLOADS["c4"]
    r = bench.roofline_for("pinv_tc", 1.0, 4, 1, wl, PEAKS, "measured")
    m, d = wl.m, wl.d
    flops = wl.heads * (2.0 * m * m * d + 8.0 * wl.iters * m ** 3 + 2.0 * m * m * d)
    assert r["bound"] == "tensor" and r["algorithmic_flops"] == flops
    assert r["peak"] == pytest.approx(1800.0 * 1.1 / 2.25)
    assert r["achieved"] == pytest.approx(flops / 250e-6 / 1e12)


def test_large_m_pseudo_inverse_peak_mixes_fp16_updates_and_tf32_rest():
    """m > 128: the update products run with fp16 operands (the bf16 rate),
    the scores and W = Z G in tf32; the peak is the flops over the time they
    take at those rates."""
    wl = workloads.WORKLOADS["c5"]
    r = bench.roofline_for("pinv_big", 1.0, 4, 1, wl, PEAKS, "measured")
    m, d = wl.m, wl.d
    upd = wl.heads * 8.0 * wl.iters * m ** 3
    rest = wl.heads * 4.0 * m * m * d
    t = upd / 1800e12 + rest / (1800e12 * 1.1 / 2.25)
    assert r["algorithmic_flops"] == upd + rest
    assert r["peak"] == pytest.approx((upd + rest) / t / 1e12)
    assert 1800.0 * 1.1 / 2.25 < r["peak"] < 1800.0


def test_pseudo_inverse_not_credited_with_w_when_w_tc_forms_it():
    wl = workloads.WORKLOADS["c3"]
    m, d = wl.m, wl.d
    r = bench.roofline_for("pinv_tc", 1.0, 4, 1, wl, PEAKS, "measured", w_separate=True)
    assert r["algorithmic_flops"] == wl.heads * (2.0 * m * m * d + 8.0 * wl.iters * m ** 3)
    w = bench.roofline_for("w_tc", 1.0, 4, 1, wl, PEAKS, "measured", w_separate=True)
    assert w["algorithmic_flops"] == wl.heads * 2.0 * m * m * d


def test_small_landmark_kernel_has_its_own_bytes():
    wl = workloads.WORKLOADS["c2"]
    te = wl.B * wl.H * wl.n * wl.d * wl.elem_bytes
    r = bench.roofline_for("landmarks_small", 0.2, 10, 1, wl, PEAKS, "measured")
    assert r["kernel"] == "landmarks_small" and r["algorithmic_bytes"] == 2 * te


def test_spread_of_regions():
    s = bench.spread([3.0, 1.0, 2.0, 5.0, 4.0])
    assert s["min"] == 1.0 and s["max"] == 5.0 and s["median"] == 3.0 and s["n"] == 5


def test_pass_roofline_is_the_slower_of_bytes_and_flops():
    wl = workloads.WORKLOADS["c3"]
    te = wl.B * wl.H * wl.n * wl.d * wl.elem_bytes
    r = bench.pass_roofline(wl, 0.1, PEAKS, "measured")
    # the method's minimum traffic: Q and V twice, K once, the output once
    assert r["bytes"] == 6 * te
    assert r["t_hbm_us"] == pytest.approx(6 * te / 6000e9 * 1e6)
    assert r["t_roofline_us"] == pytest.approx(max(r["t_hbm_us"], r["t_tensor_us"]))
    assert r["frac"] == pytest.approx(r["t_roofline_us"] / 100.0)
    # this schedule's traffic (K read twice) alongside
    assert r["bytes_7te"] == 7 * te
    assert r["frac_7te"] == pytest.approx(max(7 * te / 6000e9 * 1e6, r["t_tensor_us"]) / 100.0)


def test_traffic_is_used_only_while_the_kernel_source_is_unchanged(tmp_path, monkeypatch):
    wl = workloads.WORKLOADS["c4"]
    h = bench.kernel_source_hash("tokens_tc")
    assert h is not None
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic.txt").write_text(
        f"# kernel workload source-hash bytes\n"
        f"tokens_tc c4 {h} 1000\n"
        f"tokens_tc c5b1 {h} 300\n"
        f"pinv_tc c4 0000000000000000 5\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    # the source hash is read from the real tree; only the table moves
    monkeypatch.setattr(bench, "kernel_source_hash", lambda k: h if k == "tokens_tc" else "x")
    assert bench.measured_traffic("tokens_tc", wl) == 1000.0
    assert bench.measured_traffic("pinv_tc", wl) is None  # stale hash
    # a capture at batch 1 scales with the batch
    assert bench.measured_traffic("tokens_tc", workloads.WORKLOADS["c5"]) == 300.0 * 2


def test_clock_summary_flags_throttle_reasons():
    s = bench.ClockSampler(0)
    rows = [
        ["t", "0", "2070", "2070", "900", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"],
        ["t", "0", "1980", "2070", "1400", "0x4", "Not Active", "Not Active", "Not Active", "Active"],
        ["t", "1", "500", "2070", "100", "0x0", "Active", "Not Active", "Not Active", "Not Active"],
    ]
    s.samples = [(10.0 + i, r) for i, r in enumerate(rows)]
    out = s.summary(9.0, 20.0)
    assert out["sm_mhz"] == pytest.approx(2025.0)  # GPU 0 only
    assert out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"]
    assert out["samples_in_timed_region"] == 2


def test_kernel_sources_exist():
    src = os.path.join(bench.ROOT, "nystr_self_attention_gb300", "csrc")
    for kernel, f in bench.KERNEL_SOURCES.items():
        assert os.path.isfile(os.path.join(src, f)), kernel


@pytest.mark.parametrize("clocks,rejected", [
    ({"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": []}, False),
    ({"sm_mhz": 1900.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}, False),
    ({"sm_mhz": 2000.0, "sm_max_mhz": 2070.0, "reasons": ["hw_slowdown"]}, True),
    ({"sm_mhz": 2000.0, "sm_max_mhz": 2070.0, "reasons": ["sw_thermal_slowdown"]}, True),
    ({"sm_mhz": 1200.0, "sm_max_mhz": 2070.0, "reasons": []}, True),  # a leftover clock lock
    ({"sm_mhz": 1200.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"]}, False),
    ({"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}, False),  # no nvidia-smi
])
def test_clock_rejection_rule(clocks, rejected):
    assert bench.clocks_rejected(clocks) is rejected
