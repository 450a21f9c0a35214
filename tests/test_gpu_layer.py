"""Whole-layer parity of the libmoe forward/backward sequence against the fp64
oracle, on the seeded workloads (GPU).

Routing: the GPU decides on fp32 logits, the oracle on exact ones, so a token
whose k-th and (k+1)-th logits are closer than the fp32 rounding can pick a
different last expert. Such tokens must be rare and near-ties (oracle gap
< 1e-3); they are excluded from the per-token comparisons, and experts that
received a disagreeing token are excluded from the per-expert ones. Everything
else is compared with the bf16 I/O tolerances (max-abs 2e-2, relative
Frobenius 1e-2; weight gradients: max-abs relative to max|ref|)."""
import numpy as np
import pytest
import torch

import oracle as O
from sparse_moe_layer_topk_gb300 import _lib as M
from sparse_moe_layer_topk_gb300 import inputs as I
from sparse_moe_layer_topk_gb300.layer import LatentMoELayer, weights_to_device

from gpu_util import check_close, check_close_chunked, f64, need_gpu

pytestmark = pytest.mark.gpu

GRAD_NAMES = {"Wr": "dWr", "W_dn": "dW_dn", "W13": "dW13", "W2": "dW2", "W13_sh": "dW13_sh",
              "W2_sh": "dW2_sh", "W_up": "dW_up"}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _run(inp, T=None, wgrad=M.MOE_DTYPE_F32, backward=True, fused_gather=False):
    cfg = inp["cfg"]
    T = inp["x"].shape[0] if T is None else T
    layer = LatentMoELayer(weights_to_device(inp), T, cfg.k, wgrad, fused_gather=fused_gather)
    layer.forward(inp["x"].cuda())
    if backward:
        layer.backward(inp["g"].cuda())
    torch.cuda.synchronize()
    assert int(layer.err.item()) == 0
    return layer


def _routing_disagreement(layer, L_ref, k):
    """Tokens whose GPU selection differs from the oracle's; each must be a near-tie."""
    gi = layer.topk_idx.cpu().numpy()
    ri = O.topk_select(L_ref, k)
    bad = np.where((np.sort(gi, 1) != np.sort(ri, 1)).any(1))[0]
    if bad.size:
        Ls = -np.sort(-L_ref[bad], axis=1)
        gaps = Ls[:, k - 1] - Ls[:, k]
        assert np.all(gaps < 1e-3), gaps
    return bad, ri


@pytest.mark.parametrize("fused_gather", [True, False])
def test_layer_cfg0_forward_backward_all_outputs(fused_gather):
    inp = I.make_layer_inputs(0)
    cfg = inp["cfg"]
    layer = _run(inp, fused_gather=fused_gather)
    fwd = O.layer_forward(inp)
    bwd = O.layer_backward(inp, fwd)
    bad, _ = _routing_disagreement(layer, fwd["L"], cfg.k)
    assert bad.size == 0
    np.testing.assert_array_equal(layer.counts.cpu().numpy(), fwd["counts"])
    np.testing.assert_array_equal(layer.offsets.cpu().numpy(), fwd["offsets"])
    np.testing.assert_array_equal(layer.slot_of.cpu().numpy(), fwd["slot_of"])
    np.testing.assert_array_equal(layer.token_of.cpu().numpy(), fwd["token_of"])
    check_close("w", f64(layer.topk_w), fwd["w"], max_abs=1e-5, rel_fro=1e-5)
    for name in ("z", "y_lat", "out"):
        check_close(name, f64(getattr(layer, name)), fwd[name])
    if not fused_gather:
        check_close("z_perm", f64(layer.z_perm), fwd["z_perm"])
    check_close("dx", f64(layer.dx), bwd["dx"])
    check_close("d_w", f64(layer.d_topk_w), bwd["d_w"])
    for wn, gn in GRAD_NAMES.items():
        check_close(gn, f64(layer.grads[wn]), bwd[gn], scale_by_max=True)


def test_layer_cfg0_bf16_wgrad():
    inp = I.make_layer_inputs(0)
    layer = _run(inp, wgrad=M.MOE_DTYPE_BF16)
    fwd = O.layer_forward(inp)
    bwd = O.layer_backward(inp, fwd)
    for wn, gn in GRAD_NAMES.items():
        assert layer.grads[wn].dtype == torch.bfloat16
        check_close(gn, f64(layer.grads[wn]), bwd[gn], scale_by_max=True)


def test_layer_ragged_token_count():
    """T not a multiple of any tile (ragged tails everywhere), cfg0 widths."""
    inp = I.make_layer_inputs(0, T=77)
    layer = _run(inp)
    fwd = O.layer_forward(inp)
    bwd = O.layer_backward(inp, fwd)
    bad, _ = _routing_disagreement(layer, fwd["L"], inp["cfg"].k)
    assert bad.size == 0
    check_close("out", f64(layer.out), fwd["out"])
    check_close("dx", f64(layer.dx), bwd["dx"])
    for wn, gn in GRAD_NAMES.items():
        check_close(gn, f64(layer.grads[wn]), bwd[gn], scale_by_max=True)


def test_layer_single_token():
    inp = I.make_layer_inputs(0, T=1)
    layer = _run(inp)
    fwd = O.layer_forward(inp)
    bwd = O.layer_backward(inp, fwd)
    check_close("out", f64(layer.out), fwd["out"])
    check_close("dx", f64(layer.dx), bwd["dx"])
    check_close("dW13", f64(layer.grads["W13"]), bwd["dW13"], scale_by_max=True)
    # all but k experts are empty: their gradients are exact zeros
    empty = np.where(fwd["counts"] == 0)[0]
    assert not layer.grads["W13"][empty].any() and not layer.grads["W2"][empty].any()


def _gpu_logits(layer):
    """The fp32 router logits the GPU selected on (they stay in the route
    workspace after the forward)."""
    T, E = layer.T, layer.E
    return layer.ws["route"][: T * E * 4].view(torch.float32).view(T, E).cpu().numpy()


def _check_routing_staged(layer, k, L_ref, max_bad, bias=None):
    """Staged routing parity at full size: the oracle's selection step run on the
    values the GPU decides on (its own fp32 logits, plus the bias in fp32 when
    there is one) must give the GPU's ids bit for bit, and its weights (sigmoid
    and renormalisation of those fp32 values) to fp32 rounding; those values
    must be within fp32 accumulation error of the fp64 logits L_ref (bias
    included); and against L_ref only rare near-ties may select another expert.
    Returns the GPU's ids and the tokens whose selection differs from the fp64
    one."""
    v32 = _gpu_logits(layer)
    if bias is not None:
        v32 = (v32 + bias.numpy()[None, :]).astype(np.float32)
    v32 = v32.astype(np.float64)
    assert np.abs(v32 - L_ref).max() < 1e-3
    gi = layer.topk_idx.cpu().numpy()
    np.testing.assert_array_equal(gi, O.topk_select(v32, k))
    w32, s32 = O.routing_weights(v32, gi)
    np.testing.assert_allclose(layer.topk_s.cpu().numpy(), s32, rtol=2e-6, atol=1e-7)
    np.testing.assert_allclose(layer.topk_w.cpu().numpy(), w32, rtol=3e-6, atol=1e-7)
    bad, _ = _routing_disagreement(layer, L_ref, k)
    assert bad.size <= max_bad, bad.size
    return gi, bad


def _check_maps(layer, gi, E):
    """Counts, offsets, slot and token maps, tile schedule and permuted routing
    weights of the GPU's permute against the oracle's counting sort of the GPU's
    ids: bit for bit."""
    slot_of, token_of, offsets = O.permutation_maps(gi, E)
    counts = np.diff(offsets)
    np.testing.assert_array_equal(layer.counts.cpu().numpy(), counts)
    np.testing.assert_array_equal(layer.offsets.cpu().numpy(), offsets)
    np.testing.assert_array_equal(layer.slot_of.cpu().numpy(), slot_of)
    np.testing.assert_array_equal(layer.token_of.cpu().numpy(), token_of)
    np.testing.assert_array_equal(layer.tile_sched.cpu().numpy(), O.m_tiles_schedule(counts, 128))
    row_w = np.empty(gi.size, dtype=np.float32)
    row_w[slot_of.reshape(-1)] = layer.topk_w.cpu().numpy().reshape(-1)
    np.testing.assert_array_equal(layer.row_w.cpu().numpy(), row_w)
    return counts


@pytest.mark.parametrize("cfg_id", [1, 2])
def test_layer_full_size_forward(cfg_id):
    inp = I.make_layer_inputs(cfg_id)
    cfg = inp["cfg"]
    layer = _run(inp, backward=False)
    fwd = O.layer_forward(inp)
    gi, bad = _check_routing_staged(layer, cfg.k, fwd["L"], max(2, cfg.T // 1000), inp["bias"])
    counts = _check_maps(layer, gi, cfg.E)
    keep = np.setdiff1d(np.arange(cfg.T), bad)
    check_close("out", f64(layer.out)[keep], fwd["out"][keep])
    check_close("y_lat", f64(layer.y_lat)[keep], fwd["y_lat"][keep])
    if cfg.skew:
        assert (counts <= 2).sum() >= 150 and (counts == 0).sum() > 0


@pytest.mark.parametrize("cfg_id", [1, 2])
def test_layer_T2048_E896_every_output_and_gradient(cfg_id):
    """The layer at the 896-expert shapes (d=4096, l=1024, E=896 top-16, S=2,
    f=512) with T=2048 tokens, uniform (1) and Zipf-skewed (2) routing: every
    output and every gradient (out, dx, d_w, dWr, dW_dn, dW13, dW2, dW13_sh,
    dW2_sh, dW_up) against the full fp64 oracle on the same inputs. This runs
    the router's 896 columns (three 256-wide tiles and a 128-wide tail) in the
    logits and in dWr, the K-split shared-expert weight gradients (2 slices at
    K = 2048), and, skewed, empty experts (exact-zero gradients) next to
    experts of many row tiles. Routing is staged: the GPU's ids are checked bit
    for bit against the oracle's selection on the values the GPU decided on,
    and the oracle then runs on those ids, so no token is excluded from any
    comparison."""
    inp = I.make_layer_inputs(cfg_id, T=2048)
    cfg = inp["cfg"]
    layer = _run(inp)
    L = O.router_logits(inp["x"], inp["Wr"], inp["bias"])
    gi, _ = _check_routing_staged(layer, cfg.k, L, 4, inp["bias"])
    counts = _check_maps(layer, gi, cfg.E)
    if cfg.skew:
        empty = np.where(counts == 0)[0]
        assert empty.size > 0 and counts.max() > 4 * 128
        assert not layer.grads["W13"][empty].any() and not layer.grads["W2"][empty].any()
    fwd = O.layer_forward(inp, idx=gi)
    check_close("w", f64(layer.topk_w), fwd["w"], max_abs=1e-5, rel_fro=1e-5)
    for name in ("z", "y_lat", "out"):
        check_close(name, f64(getattr(layer, name)), fwd[name])
    check_close_chunked("z_perm", layer.z_perm, fwd["z_perm"], chunk=4096)
    check_close_chunked("y_perm", layer.y_perm, fwd["y_perm"], chunk=4096)
    bwd = O.layer_backward(inp, fwd)
    check_close("dx", f64(layer.dx), bwd["dx"])
    # |d_w| reaches ~25 at l = 1024: max-abs relative to max|ref| (like a weight gradient)
    check_close("d_w", f64(layer.d_topk_w), bwd["d_w"], scale_by_max=True)
    for wn, gn in GRAD_NAMES.items():
        check_close_chunked(gn, layer.grads[wn], bwd[gn], scale_by_max=True)


def test_ep_rank_grouped_gemm_and_return():
    """One expert-parallel rank: 14 experts over 65536 pre-permuted rows, then
    the weighted return to arrival order (combine with k = 1)."""
    inp = I.make_ep_rank_inputs()
    cfg = inp["cfg"]
    counts = inp["counts"].numpy()
    offsets = O.expert_offsets(counts)
    sched = O.m_tiles_schedule(counts, 128)
    R, l, f, E = cfg.R, cfg.l, cfg.f, cfg.E
    gu = torch.empty(R, 2 * f, dtype=torch.bfloat16, device="cuda")
    h = torch.empty(R, f, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(R, l, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(R, l, dtype=torch.bfloat16, device="cuda")
    M.moe_grouped_swiglu(inp["z_perm"].cuda(), inp["W13"].cuda(), inp["W2"].cuda(),
                         torch.from_numpy(offsets).int().cuda(), torch.from_numpy(sched).int().cuda(),
                         inp["w"].cuda(), E, R, l, f, None, h, y)
    perm = inp["perm"].numpy()
    inv = np.empty(R, dtype=np.int32)
    inv[perm] = np.arange(R, dtype=np.int32)        # slot of arrival row t
    M.moe_unpermute_combine(y, torch.from_numpy(inv).reshape(R, 1).cuda(), None, R, 1, l, out)
    torch.cuda.synchronize()
    ref = O.ep_rank_forward(inp["z_perm"], counts, inp["W13"], inp["W2"], inp["w"], perm)
    check_close("ep_out", f64(out), ref)


def test_layer_fwd_bwd_T16384_sampled():
    """The benchmark workload at full size (T=16384).
    - Routing and maps: staged, bit for bit, over all tokens.
    - Every output and input gradient of sampled tokens (out, z, y_lat, dy_lat,
      dz, d_w, dx) against the oracle run on exactly those tokens.
    - Expert weight gradients of sampled experts against the oracle run on the
      tokens they hold.
    - The shared experts' weight gradients (and z, dy_lat, dz_sh over all
      tokens) against the full fp64 oracle: they do not depend on the routing.
    - dWr (896 columns: three 256-wide tiles and a 128-wide tail) against the
      oracle's router backward fed the GPU's routing-weight gradients (checked
      on the sampled tokens above) and x^T dL in fp64.
    - dW_up and dW_dn against their defining products of the layer's own
      y_lat and dz (both checked per token above)."""
    inp = I.make_layer_inputs(4)
    cfg = inp["cfg"]
    layer = _run(inp)
    L = O.router_logits(inp["x"], inp["Wr"], inp["bias"])
    gpu_idx, bad = _check_routing_staged(layer, cfg.k, L, 20)
    _check_maps(layer, gpu_idx, cfg.E)
    ref_idx = O.topk_select(L, cfg.k)
    rng = np.random.default_rng(0)
    toks = np.setdiff1d(rng.choice(cfg.T, 96, replace=False), bad)
    sub = dict(inp)
    sub["x"], sub["g"] = inp["x"][toks], inp["g"][toks]
    fwd = O.layer_forward(sub)
    bwd = O.layer_backward(sub, fwd)
    for name in ("out", "z", "y_lat"):
        check_close(name, f64(getattr(layer, name))[toks], fwd[name])
    for name in ("dz", "dx"):
        check_close(name, f64(getattr(layer, name))[toks], bwd[name])
    # internal gradients with values far above 1 (|dy_lat| up to ~8, |d_w| up to
    # ~25): max-abs relative to max|ref|, like the weight gradients
    check_close("dy_lat", f64(layer.dy_lat)[toks], bwd["dy_lat"], scale_by_max=True)
    check_close("d_w", f64(layer.d_topk_w)[toks], bwd["d_w"], scale_by_max=True)
    # sampled experts whose token set is the same on both sides
    touched = set(np.unique(gpu_idx[bad])) | set(np.unique(ref_idx[bad]))
    cand = [e for e in rng.permutation(cfg.E) if e not in touched][:6]
    for e in cand:
        te = np.where((ref_idx == e).any(1))[0]
        sub = dict(inp)
        sub["x"], sub["g"] = inp["x"][te], inp["g"][te]
        fe = O.layer_forward(sub)
        be = O.layer_backward(sub, fe)
        check_close(f"dW13[{e}]", f64(layer.grads["W13"][e]), be["dW13"][e], scale_by_max=True)
        check_close(f"dW2[{e}]", f64(layer.grads["W2"][e]), be["dW2"][e], scale_by_max=True)
    # shared experts over all tokens: full oracle
    x, g = f64(inp["x"]), f64(inp["g"])
    z_ref = x @ f64(inp["W_dn"])
    dy_ref = g @ f64(inp["W_up"]).T
    check_close("z (all tokens)", f64(layer.z), z_ref)
    check_close("dy_lat (all tokens)", f64(layer.dy_lat), dy_ref, scale_by_max=True)
    dz_sh = np.zeros_like(z_ref)
    for s in range(cfg.S):
        dzs, dW13s, dW2s = O.swiglu_expert_backward(z_ref, inp["W13_sh"][s], inp["W2_sh"][s],
                                                    dy_ref)
        dz_sh += dzs
        check_close(f"dW13_sh[{s}]", f64(layer.grads["W13_sh"][s]), dW13s, scale_by_max=True)
        check_close(f"dW2_sh[{s}]", f64(layer.grads["W2_sh"][s]), dW2s, scale_by_max=True)
    check_close("dz_sh (all tokens)", f64(layer.dz_sh), dz_sh)
    del dz_sh, z_ref, dy_ref
    # router weight gradient: the oracle's router backward on the GPU's d_w
    dL = O.router_backward(f64(layer.d_topk_w), f64(layer.topk_w), f64(layer.topk_s), gpu_idx,
                           cfg.E)
    check_close("dWr", f64(layer.grads["Wr"]), x.T @ dL, scale_by_max=True)
    # dense weight gradients = their defining products on the layer's activations
    check_close("dW_up", f64(layer.grads["W_up"]), f64(layer.y_lat).T @ g, scale_by_max=True)
    check_close("dW_dn", f64(layer.grads["W_dn"]), x.T @ f64(layer.dz), scale_by_max=True)


def test_layer_cfg0_with_aux_balance_loss():
    """aux_scale * (negative routing entropy) added to the loss: the aux loss and
    the router's gradients (dx, dWr) against the oracle with the aux term."""
    inp = I.make_layer_inputs(0)
    cfg = inp["cfg"]
    layer = LatentMoELayer(weights_to_device(inp), cfg.T, cfg.k, M.MOE_DTYPE_F32, aux_scale=0.5)
    layer.forward(inp["x"].cuda())
    layer.backward(inp["g"].cuda())
    torch.cuda.synchronize()
    fwd = O.layer_forward(inp)
    bwd = O.layer_backward(inp, fwd)
    p_ref, loss_ref = O.aux_balance_loss(fwd["L"])
    np.testing.assert_allclose(layer.p_mean.cpu().numpy(), p_ref, rtol=1e-4)
    assert abs(layer.aux_loss.item() - loss_ref) < 1e-4 * abs(loss_ref)
    dL_aux = O.aux_balance_loss_backward(fwd["L"], None, scale=0.5)
    x = f64(inp["x"])
    check_close("dx", f64(layer.dx), bwd["dx"] + dL_aux @ f64(inp["Wr"]).T)
    check_close("dWr", f64(layer.grads["Wr"]), bwd["dWr"] + x.T @ dL_aux, scale_by_max=True)


@pytest.mark.parametrize("graphs", [True, False])
def test_steps_from_host_pipeline_matches_step(graphs):
    """The pipelined host-driven steps (copies on their own streams, double-
    buffered device inputs, CUDA-graph replays or eager launches) give the same
    input gradients as plain steps."""
    inp = I.make_layer_inputs(0)
    cfg = inp["cfg"]
    layer = LatentMoELayer(weights_to_device(inp), cfg.T, cfg.k, M.MOE_DTYPE_F32)
    g0 = torch.Generator().manual_seed(9)
    xs = [torch.randn(cfg.T, cfg.d, generator=g0).to(torch.bfloat16).pin_memory() for _ in range(3)]
    gs = [torch.randn(cfg.T, cfg.d, generator=g0).to(torch.bfloat16).pin_memory() for _ in range(3)]
    outs = [torch.empty(cfg.T, cfg.d, dtype=torch.bfloat16).pin_memory() for _ in range(3)]
    layer.steps_from_host(xs, gs, outs, graphs=graphs)
    torch.cuda.synchronize()
    ref = LatentMoELayer(weights_to_device(inp), cfg.T, cfg.k, M.MOE_DTYPE_F32)
    for i in range(3):
        dx = ref.step(xs[i].cuda(), gs[i].cuda())
        torch.cuda.synchronize()
        assert torch.equal(dx.cpu(), outs[i]), i


def test_captured_step_replays_bit_identical():
    """A step captured as a CUDA graph and replayed on new contents of its input
    buffers gives the eager step's outputs and gradients bit for bit."""
    inp = I.make_layer_inputs(0)
    cfg = inp["cfg"]
    layer = LatentMoELayer(weights_to_device(inp), cfg.T, cfg.k, M.MOE_DTYPE_F32)
    x = inp["x"].cuda()
    g = inp["g"].cuda()
    layer.step(x, g)  # eager first: kernel attributes are set outside the capture
    graph = layer.capture_step(x, g)
    gen = torch.Generator().manual_seed(21)
    x.copy_(torch.randn(cfg.T, cfg.d, generator=gen).to(torch.bfloat16))
    g.copy_(torch.randn(cfg.T, cfg.d, generator=gen).to(torch.bfloat16))
    graph.replay()
    torch.cuda.synchronize()
    assert int(layer.err.item()) == 0
    got = {"out": layer.out.clone(), "dx": layer.dx.clone(),
           **{n: t.clone() for n, t in layer.grads.items()}}
    ref = LatentMoELayer(weights_to_device(inp), cfg.T, cfg.k, M.MOE_DTYPE_F32)
    ref.step(x, g)
    torch.cuda.synchronize()
    want = {"out": ref.out, "dx": ref.dx, **ref.grads}
    for n in got:
        assert torch.equal(got[n], want[n]), n
