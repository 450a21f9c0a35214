"""Host logic of bench.py (no GPU): the algorithmic work per launch that the
roofline divides by, the choice and labelling of the peaks, and the whole-job
throughput arithmetic."""
import json

import pytest

import bench
from sparse_moe_layer_topk_gb300 import inputs as I

# the bench workload: T=16384 tokens, d=4096, l=1024, E=896 experts, top-16, f=512, 2 shared
CFG = I.CONFIGS[4]
T, d, l, E, k, f, S = CFG.T, CFG.d, CFG.l, CFG.E, CFG.k, CFG.f, CFG.S
R = T * k


def test_bench_workload_shape():
    assert (T, d, l, E, k, f, S) == (16384, 4096, 1024, 896, 16, 512, 2)


@pytest.mark.parametrize("label,flops,nbytes", [
    # values worked out by hand from the shapes above (GFLOP, MB = 1e6 bytes)
    ("router_logits_gemm", 120.26, None),      # 2 * 16384 * 4096 * 896
    ("topk_sigmoid", 0, 61.87),                # 16384*896*4 + 16384*16*12
    ("latent_proj_gemm", 137.44, None),        # 2 * 16384 * 4096 * 1024
    # x 134.22 + [Wr | W_dn] 15.73 + fp32 logits 58.72 + bf16 z 33.55
    ("router_latent_gemm", 257.70, 242.22),    # 2 * 16384 * 4096 * (896 + 1024)
    ("permute_gather", 0, 571.47),             # 33.55 + 536.87 + 1.05
    ("combine", 0, 605.03),                    # 536.87 + 2*33.55 + 1.05
    ("expert_gemm1_swiglu", 549.76, None),     # 2 * 262144 * 1024 * 1024
    ("expert_wgrad1", 549.76, 4831.84),        # 536.87 + 536.87 + 896*1024*1024*4
    ("expert_wgrad2", 274.88, 2684.35),        # 268.44 + 536.87 + 896*512*1024*4
    # the router backward's dL has 16 nonzeros per token: 2 T k d per product
    ("down_proj_router_dgrad", 139.59, None),  # 2*16384*4096*1024 + 2*16384*16*4096
    ("router_wgrad", 2.15, 150.47),            # x 134.22 + 16 (value, id) pairs/token 1.57 + dWr 14.68
    # dy 536.87 + W2 939.52 + g,u,h in and dg,du,w*h out 1610.61 + d_row_w 1.05
    ("expert_dgrad2_swiglu_bwd", 274.88, 3088.06),
    ("routing_weight_grad_reduce", 0, 5.24),   # 4 fp32 partials in, 1 out, per row
    ("permute_hist", 0, 1.28),                 # ids 1.05 + 64 chunks x 896 counts 0.23
    ("permute_maps", 0, 5.48),                 # ids, weights 2.10 + prefixes 0.23 + maps out 3.15
    # dW2_sh: 4 slices of 1024 x 1024 fp32 in + out 20.97; dW13_sh: 2 of 1024 x 2048 25.17
    ("splitk_reduce", 0, 23.07),
])
def test_kernel_work_matches_hand_computed_values(label, flops, nbytes):
    fl, by = bench.kernel_work(CFG, T)[label]
    assert fl / 1e9 == pytest.approx(flops, abs=0.01)
    if nbytes is not None:
        assert by / 1e6 == pytest.approx(nbytes, abs=0.01)


def test_kernel_work_scales_with_tokens():
    """Every routed and dense term is linear in T except the weights: doubling T
    doubles the flops of every GEMM."""
    a, b = bench.kernel_work(CFG, 4096), bench.kernel_work(CFG, 8192)
    for label in a:
        assert b[label][0] == 2 * a[label][0], label
        assert b[label][1] >= a[label][1], label


def test_peaks_exact_names():
    p = {"hbm_gbs": 7100.0, "bf16_tflops": 2050.0, "bf16_tflops_sustained": 1750.0}
    hbm, hs, tc, ts = bench.roofline_peaks(p)
    assert (hbm, tc) == (7100.0, 1750.0)
    assert hs.startswith("measured") and ts == "measured (sustained)"


def test_peaks_nested_schema_and_value_objects():
    p = {"hbm": {"copy": {"gbs": 6900.0, "bytes": 1 << 30}, "util_pct": 88.0},
         "gemm": {"bf16": {"tflops": {"value": 2000.0}, "tflops_sustained": {"median": 1650.0}}},
         "clocks": {"sm_mhz": 2070}}
    hbm, hs, tc, ts = bench.roofline_peaks(p)
    assert hbm == 6900.0 and hs == "measured (copy)"
    assert tc == 1650.0 and ts == "measured (sustained)"


def test_peaks_burst_only_is_labelled_as_burst():
    hbm, hs, tc, ts = bench.roofline_peaks({"hbm_gbs": 7000, "bf16_tflops": 2000})
    assert tc == 2000.0 and "burst" in ts


def test_peaks_fallback_is_labelled_fallback():
    for p in ({}, {"note": "no data"}, {"hbm_gbs": 0, "bf16_tflops": None}):
        hbm, hs, tc, ts = bench.roofline_peaks(p)
        assert hbm == bench.FALLBACK_PEAKS["hbm_gbs"] and hs == "fallback (copy)"
        assert tc == bench.FALLBACK_PEAKS["bf16_tflops_sustained"] and ts == "fallback (sustained)"


def test_peaks_file_reading(tmp_path):
    path = tmp_path / "peaks.json"
    assert bench.load_peaks(str(path)) == {}
    path.write_text("not json")
    assert bench.load_peaks(str(path)) == {}
    path.write_text(json.dumps({"hbm_gbs": 7000}))
    assert bench.load_peaks(str(path)) == {"hbm_gbs": 7000}


def test_job_throughput_and_single_rank_time():
    # 2 replicas x 16384 tokens x 10 steps in 50 ms of the slowest rank
    assert bench.job_tokens_per_s(2, 16384, 10, 50.0) == pytest.approx(2 * 16384 * 10 / 0.05)
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5


def test_roofline_report_picks_the_dominant_kernel_and_its_bound():
    peaks = (8000.0, "measured (copy)", 2000.0, "measured (sustained)")
    work = {"mem_kernel": (1e9, 8e9),      # 0.5 ms of compute, 1.0 ms of memory at the peaks
            "tc_kernel": (4e12, 1e9),      # 2.0 ms of compute, 0.125 ms of memory
            "tiny": (0, 1e6)}
    # label -> (launches, total ms)
    per = {"mem_kernel": (2, 4.0), "tc_kernel": (1, 2.5), "tiny": (4, 0.4)}
    roof, br, gp = bench.roofline_report(per, work, peaks, lambda name: 123)
    assert roof["kernel"] == "mem_kernel" and roof["bound"] == "hbm"
    assert roof["achieved"] == pytest.approx(8e9 / 2e-3 / 1e9)       # 4000 GB/s per launch
    assert roof["frac"] == pytest.approx(0.5) and roof["traffic"] == 123
    assert roof["peak"] == 8000.0 and roof["peak_source"] == "measured (copy)"
    assert br["tc_kernel"]["roofline_frac"] == pytest.approx(2.0 / 2.5)
    assert br["tc_kernel"]["tflops"] == pytest.approx(1600.0)
    assert sum(v["share"] for v in br.values()) == pytest.approx(1.0, abs=1e-3)
    assert list(br) == ["mem_kernel", "tc_kernel", "tiny"]   # by total time
    assert gp is None                                          # no expert GEMM timed

    per = {"tc_kernel": (1, 2.5), "tiny": (1, 0.1)}
    roof, _, _ = bench.roofline_report(per, work, peaks, lambda name: None)
    assert roof["bound"] == "tensor" and roof["unit"] == "TFLOP/s"
    assert roof["frac"] == pytest.approx(0.8) and roof["peak_source"] == "measured (sustained)"


def test_roofline_report_grouped_gemm_percentage():
    peaks = (8000.0, "m", 2000.0, "m")
    work = {n: (1e12, 1e9) for n in bench.EXPERT_GEMMS}
    per = {n: (2, 2.0) for n in bench.EXPERT_GEMMS}             # 1 ms per launch
    _, _, gp = bench.roofline_report(per, work, peaks, lambda name: None)
    assert gp == pytest.approx(100.0 * 1000.0 / 2000.0)       # 1 PFLOP/s of 2


def test_kernel_work_bf16_weight_gradients():
    """With bf16 weight gradients only the gradient writes shrink, by half."""
    a, b = bench.kernel_work(CFG, T), bench.kernel_work(CFG, T, wgrad_bytes=2)
    grads = {"latent_proj_wgrad": d * l, "expert_wgrad2": E * f * l, "expert_wgrad1": E * l * 2 * f,
             "shared_wgrad2": S * f * l, "shared_wgrad1": S * l * 2 * f, "router_wgrad": d * E,
             # the split-K reduction writes the shared gradients (mean of its two launches)
             "splitk_reduce": (S * f * l + l * 2 * S * f) // 2}
    for label in a:
        assert a[label][0] == b[label][0], label
        assert a[label][1] - b[label][1] == 2 * grads.get(label, 0), label


def test_clock_samples_parsing():
    out = "\n".join([
        "2070, 2070, 910.55, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "2055, 2070, 1398.20, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "[N/A], 2070, [N/A], [N/A], [N/A], [N/A], [N/A], [N/A]",   # a sample nvidia-smi could not read
        "2040, 2070, 1401.00, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbage",
    ])
    c = bench.parse_clock_samples(out)
    assert c == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}
    hot = bench.parse_clock_samples(
        "1800, 2070, 1400, 0x28, Not Active, Active, Active, Not Active\n")
    assert hot["reasons"] == ["hw_thermal_slowdown", "sw_thermal_slowdown"]
    assert bench.parse_clock_samples("")["sm_mhz"] is None


def test_dram_traffic_only_for_the_sources_it_was_taken_on(monkeypatch):
    """The recorded ncu traffic is reported only while the GEMM engine's sources
    hash to the value it was captured on, and only for its own workload."""
    tab = json.load(open(bench.os.path.join(bench.ROOT, "profiles", "dram_traffic.json")))
    wl = "latentmoe_fwd_bwd_T16384_E896_top16"
    ent = tab[wl]["expert_wgrad1"]
    monkeypatch.setattr(bench, "source_hash", lambda: ent["source_hash"])
    assert bench.dram_traffic("expert_wgrad1", wl) == ent["bytes_per_launch"]
    assert bench.dram_traffic("expert_wgrad1", "another_workload") is None
    assert bench.dram_traffic("no_such_kernel", wl) is None
    monkeypatch.setattr(bench, "source_hash", lambda: "0" * 16)
    assert bench.dram_traffic("expert_wgrad1", wl) is None


def test_burst_peak_for_kernels_timed_alone():
    assert bench.burst_tc_peak({"bf16_tflops": 2050.0, "bf16_tflops_sustained": 1700.0}) == \
        (2050.0, "measured (burst)")
    assert bench.burst_tc_peak({"bf16_tflops_sustained": 1700.0}) == \
        (bench.FALLBACK_PEAKS["bf16_tflops"], "fallback (burst)")


def test_dense_router_backward_executed_flops_and_waste():
    """The dense GEMMs of the router backward execute 2 T E d flops per product;
    the breakdown reports that rate and the share of it that is waste next to
    the roofline fraction, which is taken on the sparse algorithmic cost."""
    ex = bench.dense_executed_flops(CFG, T)
    assert ex["router_wgrad"] / 1e9 == pytest.approx(120.26, abs=0.01)
    assert ex["down_proj_router_dgrad"] / 1e9 == pytest.approx(257.70, abs=0.01)
    work = bench.kernel_work(CFG, T)
    peaks = (6800.0, "m", 1700.0, "m")
    per = {"router_wgrad": (1, 0.082), "down_proj_router_dgrad": (1, 0.139)}
    _, br, _ = bench.roofline_report(per, work, peaks, lambda name: None, executed=ex)
    assert br["router_wgrad"]["executed_tflops"] == pytest.approx(120.26e9 / 82e-6 / 1e12, rel=1e-3)
    assert br["router_wgrad"]["executed_waste_frac"] == pytest.approx(1 - 16 / 896, abs=1e-4)
    # memory floor of router_wgrad: reading x once (plus dL's nonzeros and dWr)
    assert br["router_wgrad"]["roofline_frac"] == pytest.approx(150.47e6 / 6800e9 / 82e-6, rel=1e-2)
    # compute floor of the fused dgrad: its down-projection part plus the sparse router part
    assert br["down_proj_router_dgrad"]["roofline_frac"] == pytest.approx(
        139.59e9 / 1700e12 / 139e-6, rel=1e-2)
