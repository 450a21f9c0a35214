"""bench.py's GPU arm driven end to end on the CPU (no GPU needed): every CUDA
call, the library, the layer and the clock sampler are replaced by fakes, so the
host side (argument handling, timing arithmetic, roofline assembly, the JSON
line and its keys) runs as on a GB300."""
import io
import json
import sys
import types
from contextlib import redirect_stdout
from unittest import mock

import pytest
import torch

import bench
from sparse_moe_layer_topk_gb300 import _lib as M
from sparse_moe_layer_topk_gb300 import build as B
from sparse_moe_layer_topk_gb300 import inputs as I
import sparse_moe_layer_topk_gb300.layer as LY


# the library's launch labels of one step, and a per-launch time in us for a few
# of them (50 us for the rest)
LABELS = ["router_logits_gemm", "topk_sigmoid", "latent_proj_gemm", "permute_hist", "permute_scan",
          "permute_maps", "permute_gather", "expert_gemm1_swiglu", "expert_gemm2_rowscale",
          "shared_gemm1_swiglu", "shared_gemm2", "combine", "latent_proj_dgrad", "latent_proj_wgrad",
          "combine_bwd_gather", "expert_dgrad2_swiglu_bwd", "routing_weight_grad_reduce",
          "expert_wgrad2", "expert_dgrad1", "expert_wgrad1", "shared_dgrad2_swiglu_bwd",
          "shared_wgrad2", "splitk_reduce", "shared_dgrad1", "shared_wgrad1", "permute_bwd_sum",
          "router_bwd_dlogits", "down_proj_router_dgrad", "router_wgrad"]
US = {"expert_wgrad1": 786.0, "expert_dgrad2_swiglu_bwd": 575.0, "expert_gemm1_swiglu": 575.0}


class FakeEvent:
    """A CUDA event pair that measures 4.76 ms per step."""

    def __init__(self, enable_timing=False):
        pass

    def record(self, stream=None):
        pass

    def elapsed_time(self, other):
        return 4.76 * STEPS


class FakeLayer:
    def __init__(self, *a, **k):
        self.err = torch.zeros(1, dtype=torch.int32)

    def step(self, x, g):
        pass

    def capture_step(self, x, g):
        return types.SimpleNamespace(replay=lambda: None)

    def steps_from_host(self, xs, gs, dxs, graphs=True):
        pass


class FakeClocks:
    def __init__(self, uuid):
        pass

    def start(self):
        pass

    def stop(self):
        return {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 14}


def timing_report():
    """The library's per-label (launches, total ms) over STEPS steps."""
    rep = {}
    for lab in LABELS:
        n = STEPS * (2 if lab in ("latent_proj_gemm", "latent_proj_wgrad", "splitk_reduce") else 1)
        rep[lab] = (n, n * US.get(lab, 50.0) / 1000.0)
    return rep


def small_inputs(cfg, T=None):
    return {"cfg": cfg, "x": torch.zeros(4, 8, dtype=torch.bfloat16),
            "g": torch.zeros(4, 8, dtype=torch.bfloat16)}


STEPS = 50


def run(argv):
    """bench.run_ours with these command-line arguments and every GPU call faked;
    returns the JSON line it prints."""
    global STEPS
    with mock.patch.object(sys, "argv", ["bench.py"] + argv):
        args = bench.parse()
    STEPS = args.steps
    patches = [
        mock.patch.object(torch.cuda, "set_device", lambda *a: None),
        mock.patch.object(torch.cuda, "synchronize", lambda *a: None),
        mock.patch.object(torch.cuda, "current_stream", lambda *a: "stream"),
        mock.patch.object(torch.cuda, "Event", FakeEvent),
        mock.patch.object(torch.cuda, "empty_cache", lambda: None),
        mock.patch.object(torch.cuda, "get_device_properties", lambda i: types.SimpleNamespace(uuid="x")),
        mock.patch.object(torch.Tensor, "cuda", lambda self, *a, **k: self),
        mock.patch.object(torch.Tensor, "pin_memory", lambda self, *a, **k: self),
        mock.patch.object(B, "build_library", lambda *a, **k: None),
        mock.patch.object(M, "load", lambda *a, **k: None),
        mock.patch.object(M, "moe_timing_report", timing_report),
        mock.patch.object(M, "moe_timing_enable", lambda flag: None),
        mock.patch.object(I, "make_layer_inputs", small_inputs),
        mock.patch.object(LY, "LatentMoELayer", FakeLayer),
        mock.patch.object(LY, "weights_to_device", lambda inp: {}),
        mock.patch.object(bench, "ClockSampler", FakeClocks),
        mock.patch.object(bench, "oracle_sample_time", lambda inp, n: 11.5),
        mock.patch.object(bench, "load_peaks", lambda *a, **k: {}),  # no measured peaks
    ]
    for p in patches:
        p.start()
    try:
        buf = io.StringIO()
        with redirect_stdout(buf):
            bench.run_ours(args)
    finally:
        for p in patches:
            p.stop()
    line = json.loads(buf.getvalue().strip().splitlines()[-1])
    return line


CONTRACT_KEYS = ["metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                 "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                 "roofline", "cpu_baseline", "e2e", "gpu_launches", "clocks"]


def test_json_line_has_every_contract_key():
    d = run(["--no-secondary", "--steps", "10", "--warmup", "3"])
    assert [k for k in CONTRACT_KEYS if k not in d] == []
    assert d["steps"] == 10 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["ms_per_step"] == pytest.approx(4.76)
    assert d["value"] == pytest.approx(16384 / 4.76e-3)
    assert d["gpu_launches"] == sum(n for n, _ in timing_report().values())
    assert d["config"]["workload"] == "latentmoe_fwd_bwd_T16384_E896_top16"
    r = d["roofline"]
    assert r["kernel"] == "expert_wgrad1" and r["bound"] == "hbm"
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["clocks"]["sm_mhz"] > 0
    assert d["secondary_peak"] == {"tflops": 1900.0, "source": "fallback (burst)"}
    json.dumps(d)


def test_bf16_gradients_and_eager_timing():
    d = run(["--no-secondary", "--wgrad", "bf16", "--no-e2e", "--no-graph", "--no-cpu-baseline"])
    assert d["e2e"] is None and d["cpu_baseline"] is None
    assert d["roofline"]["traffic"] is None        # the capture on record used fp32 gradients
    assert d["timing"]["value"] == "eager launches"
    assert d["config"]["wgrad_dtype"] == "bf16"


def test_reference_arm_runs_on_rank_0_only(monkeypatch, capsys):
    """Under torchrun the oracle arm runs and prints on rank 0 alone; the other
    ranks return at once without work or output."""
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    with mock.patch.object(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"]):
        args = bench.parse()
    with mock.patch.object(bench, "oracle_sample_time", side_effect=AssertionError("work on rank 1")):
        assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""
