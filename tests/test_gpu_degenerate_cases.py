"""Degenerate cases of the method (GPU): the empty batch through the whole layer,
every expert selected (k = E), and every token routed to one expert."""
import numpy as np
import pytest
import torch

import oracle as O
from sparse_moe_layer_topk_gb300 import _lib as M
from sparse_moe_layer_topk_gb300 import inputs as I
from sparse_moe_layer_topk_gb300.layer import LatentMoELayer, weights_to_device

from gpu_util import check_close, dev, f64, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.mark.parametrize("wgrad", [M.MOE_DTYPE_F32, M.MOE_DTYPE_BF16])
def test_layer_with_no_tokens(wgrad):
    """T = 0: empty output and input gradient, zero rows for every expert, no
    device error, and every weight gradient exactly zero (stale contents are
    overwritten)."""
    inp = I.make_layer_inputs(0)
    cfg = inp["cfg"]
    layer = LatentMoELayer(weights_to_device(inp), 0, cfg.k, wgrad)
    for g in layer.grads.values():
        g.fill_(1.0)
    for t in (layer.counts, layer.offsets, layer.tile_sched):
        t.fill_(-1)
    x = torch.empty(0, cfg.d, dtype=torch.bfloat16, device="cuda")
    dout = torch.empty(0, cfg.d, dtype=torch.bfloat16, device="cuda")
    out = layer.forward(x)
    dx = layer.backward(dout)
    torch.cuda.synchronize()
    assert tuple(out.shape) == (0, cfg.d) and tuple(dx.shape) == (0, cfg.d)
    assert int(layer.err.item()) == 0
    for name in ("counts", "offsets", "tile_sched"):
        assert not getattr(layer, name).any(), name
    for name, g in layer.grads.items():
        assert not g.any(), name


@pytest.mark.parametrize("T,E", [(64, 32), (100, 16)])
def test_topk_selects_every_expert_when_k_equals_E(T, E):
    """k = E: every expert is selected, in (logit desc, id asc) order, and the
    weights are the sigmoids renormalised over all experts."""
    k = E
    L = I.make_logits(5 + T, T, E, ties=True)
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    s = torch.empty(T, k, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_topk_from_logits(dev(L), None, T, E, k, idx, w, s, err)
    torch.cuda.synchronize()
    v = L.numpy().astype(np.float64)
    ref_idx = O.topk_select(v, k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    assert np.array_equal(np.sort(ref_idx, axis=1), np.tile(np.arange(E), (T, 1)))
    ref_w, ref_s = O.routing_weights(v, ref_idx)
    np.testing.assert_allclose(s.cpu().numpy(), ref_s, rtol=2e-6, atol=1e-7)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=3e-6, atol=1e-7)
    assert int(err.item()) == 0


def test_every_token_on_one_expert():
    """All T tokens pick the same expert (k = 1): the permute gives that expert
    every row in token order and the others none, and the grouped experts run
    one segment of T rows next to empty ones."""
    T, E, l, f, hot = 300, 64, 128, 64, 37
    idx = torch.full((T, 1), hot, dtype=torch.int32)
    z = (torch.randn(T, l, generator=torch.Generator().manual_seed(41))).to(torch.bfloat16)
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    slot_of = torch.empty(T, 1, dtype=torch.int32, device="cuda")
    token_of = torch.empty(T, dtype=torch.int32, device="cuda")
    tile_sched = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    row_w = torch.empty(T, dtype=torch.float32, device="cuda")
    z_perm = torch.empty(T, l, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    tw = torch.full((T, 1), 1.0)
    wsb = M.moe_workspace_size(M.MOE_OP_PERMUTE, T=T, E=E)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    M.moe_permute(dev(z), dev(idx), dev(tw), T, l, E, 1, z_perm, counts, offsets, slot_of,
                  token_of, tile_sched, row_w, ws, wsb, err)
    torch.cuda.synchronize()
    ref_counts = np.zeros(E, dtype=np.int64)
    ref_counts[hot] = T
    np.testing.assert_array_equal(counts.cpu().numpy(), ref_counts)
    np.testing.assert_array_equal(offsets.cpu().numpy(), O.expert_offsets(ref_counts))
    np.testing.assert_array_equal(tile_sched.cpu().numpy(), O.m_tiles_schedule(ref_counts, 128))
    np.testing.assert_array_equal(token_of.cpu().numpy(), np.arange(T))
    np.testing.assert_array_equal(slot_of.cpu().numpy().ravel(), np.arange(T))
    assert torch.equal(z_perm.cpu(), z)
    assert int(err.item()) == 0
    # the grouped experts on that permutation
    W13 = (torch.randn(E, l, 2 * f, generator=torch.Generator().manual_seed(42)) * 0.02).to(
        torch.bfloat16)
    W2 = (torch.randn(E, f, l, generator=torch.Generator().manual_seed(43)) * 0.02).to(
        torch.bfloat16)
    gu = torch.empty(T, 2 * f, dtype=torch.bfloat16, device="cuda")
    h = torch.empty(T, f, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(T, l, dtype=torch.bfloat16, device="cuda")
    M.moe_grouped_swiglu(z_perm, dev(W13), dev(W2), offsets, tile_sched, row_w, E, T, l, f, gu, h,
                         y)
    torch.cuda.synchronize()
    ref_y = O.grouped_swiglu(f64(z), W13, W2, O.expert_offsets(ref_counts), np.ones(T))
    check_close("y_perm", f64(y), ref_y)
