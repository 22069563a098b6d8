"""Host logic of bench.py's roofline accounting (no GPU).

The roofline object divides algorithmic bytes or flops by a measured time;
these tests pin the per-segment byte and flop counts to closed forms written
out independently for the default layer, and check the bound selection and
the summed-roofline fraction on hand-worked numbers.
"""

import pytest

import bench
from workloads import get_config

PEAKS = {"hbm_gbs": 6792.4, "bf16_tflops": 1945.7}


def test_expert_product_flops_are_twelve_dhm_in_total():
    cfg = get_config("qwen3-30b-a3b-t4k")
    M = 19707
    a = bench.algorithmic(cfg, M, gathered=True)
    D, H = cfg.D, cfg.H
    # G1 and G2: D x H per retained row each; G3 and G4: D x 2H each (x2 flops per MAC)
    assert a["fc2_dgrad"]["flops"] == a["fc2_wgrad"]["flops"] == 2 * M * D * H
    assert a["fc1_wgrad"]["flops"] == a["fc1_dgrad"]["flops"] == 4 * M * D * H
    assert sum(a[s]["flops"] for s in ("fc2_dgrad", "fc2_wgrad", "fc1_wgrad", "fc1_dgrad")) \
        == 12 * D * H * M


def test_weight_gradient_bytes_are_dominated_by_fp32_outputs():
    cfg = get_config("qwen3-30b-a3b-t4k")
    a = bench.algorithmic(cfg, 19707, gathered=True)
    E, D, H = cfg.E, cfg.D, cfg.H
    # dW_down (H x D) and dW_gate, dW_up (D x H each) in fp32, once per launch
    assert a["fc2_wgrad"]["bytes"] >= 4 * E * H * D
    assert a["fc1_wgrad"]["bytes"] >= 8 * E * D * H
    # the default layer: 1.61 GB of fp32 FC1 weight gradients plus the rows
    assert a["fc1_wgrad"]["bytes"] == 19707 * (D + 2 * H) * 2 + 8 * E * D * H


def test_score_reads_every_g_and_phi_row_once():
    cfg = get_config("qwen3-30b-a3b-t4k")
    a = bench.algorithmic(cfg, 1, gathered=True)
    N = cfg.T * cfg.K
    assert a["score"]["bytes"] == cfg.T * cfg.D * 2 + N * cfg.H * 2 + 12 * N


def test_gathered_compaction_moves_only_gradient_rows():
    cfg = get_config("qwen3-30b-a3b-t4k")
    M = 1000
    g = bench.algorithmic(cfg, M, gathered=True)["compact"]["bytes"]
    c = bench.algorithmic(cfg, M, gathered=False)["compact"]["bytes"]
    assert c - g == 2 * M * (2 * cfg.D + 3 * cfg.H) * 2 - 2 * M * cfg.D * 2


def test_roofline_picks_the_slower_bound():
    # 1 GB and 100 GFLOP: HBM takes 147 us, the tensor pipe 51 us -> HBM-bound
    r = bench.roofline_of({"bytes": 10 ** 9, "flops": 10 ** 11}, 0.2, PEAKS)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s"
    assert r["achieved"] == pytest.approx(5000.0, rel=1e-3)
    assert r["frac"] == pytest.approx(5000.0 / 6792.4, rel=1e-3)
    # 10 MB and 1 TFLOP: tensor-bound
    r = bench.roofline_of({"bytes": 10 ** 7, "flops": 10 ** 12}, 1.0, PEAKS)
    assert r["bound"] == "tensor" and r["achieved"] == pytest.approx(1000.0, rel=1e-3)


def test_roofline_time_is_the_larger_of_the_two_bounds():
    a = {"bytes": 6792.4e9 * 1e-3, "flops": 1945.7e12 * 2e-3}  # 1 ms of HBM, 2 ms of tensor
    assert bench.roofline_time_ms(a, PEAKS) == pytest.approx(2.0)
    assert bench.roofline_time_ms({"bytes": 6792.4e9 * 3e-3}, PEAKS) == pytest.approx(3.0)


def test_linear_fit_recovers_a_line_and_its_residuals():
    xs = [32818, 65569, 98353, 131072]
    ys = [1.87 + 4.972e-5 * x for x in xs]
    f = bench.linear_fit(xs, ys)
    assert f["a"] == pytest.approx(1.87, rel=1e-9)
    assert f["b"] == pytest.approx(4.972e-5, rel=1e-9)
    assert f["r2"] == pytest.approx(1.0)
    ys2 = [1.0, 3.0, 2.0, 4.0]  # hand-worked: slope 0.8, intercept 0.5, residuals +-0.3/0.6
    g = bench.linear_fit([1, 2, 3, 4], ys2)
    assert g["b"] == pytest.approx(0.8) and g["a"] == pytest.approx(0.5)
    assert g["max_abs_residual"] == pytest.approx(0.9)
    assert g["r2"] == pytest.approx(1 - 1.8 / 5.0)


def test_sweep_reports_the_fit_in_ns_per_row_and_the_fixed_bytes():
    cfg = get_config("glm45-106b-a12b-t16k")
    pts = [{"retained_rows": m, "ms_per_step": 2.0 + 5e-5 * m} for m in (1000, 2000, 4000)]
    s = bench.sweep_summary(cfg, pts, PEAKS)
    assert s["fit"]["ns_per_retained_row"] == pytest.approx(50.0)
    assert s["fit"]["intercept_ms"] == pytest.approx(2.0)
    fixed = s["intercept_reading"]["weights_in_and_fp32_weight_gradients_out_bytes"]
    assert fixed == 3 * 128 * 4096 * 1408 * 6  # BF16 weights in, FP32 gradients out
    assert s["routed_pairs"] == cfg.N


def test_headline_rate_is_the_middle_of_a_sweep():
    class A:
        rate = None
    assert bench.headline_rate(get_config("glm45-106b-a12b-t16k"), A()) == (1, 2)
    assert bench.headline_rate(get_config("qwen3-30b-a3b-t4k"), A()) == (3, 5)
    A.rate = "3/4"
    assert bench.headline_rate(get_config("glm45-106b-a12b-t16k"), A()) == (3, 4)


@pytest.mark.parametrize("name,score,fc1_dgrad,dispatch", [
    ("qwen3-30b-a3b-t4k", "score_upfront_kernel<8, 3>", "grouped_gemm_kernel<3, 1, 0>",
     "dispatch_fused_kernel"),
    ("qwen3-30b-a3b-t32k", "score_upfront_kernel<8, 3>", "grouped_gemm_kernel<3, 1, 0>",
     "dispatch_hist_kernel + dispatch_scan_kernel + dispatch_scatter_kernel"),
    ("glm45-106b-a12b-t16k", "score_upfront_kernel<16, 6>", "grouped_gemm_kernel<3, 1, 1>",
     "dispatch_fused_kernel"),
    ("stress-e256", "score_upfront_kernel<8, 2>", "grouped_gemm_kernel<3, 1, 0>",
     "dispatch_hist_kernel + dispatch_scan_kernel + dispatch_scatter_kernel"),
])
def test_segment_kernel_names_follow_the_launch_rules(name, score, fc1_dgrad, dispatch):
    # the names the launch list shows: score instantiation by chunks per lane
    # (D/8 and H/8 sixteen-byte chunks over 32 lanes), wide FC1 dgrad tiles when
    # 2H spans 32 or more 64-deep K blocks, three dispatch launches above 2^17 pairs
    cfg = get_config(name)
    assert bench.segment_kernels("score", cfg) == score
    assert bench.segment_kernels("fc1_dgrad", cfg) == fc1_dgrad
    assert bench.segment_kernels("dispatch", cfg) == dispatch
    assert bench.segment_kernels("fc1_wgrad", cfg) == "grouped_gemm_kernel<2, 0, 0>"
