"""The empty batch (T = 0 tokens) through the whole layer (GPU): the forward
output and input gradient are empty, the permute reports zero rows for every
expert, no device error is raised, and every weight gradient is exactly zero
(stale contents are overwritten)."""
import pytest
import torch

from sparse_moe_layer_topk_gb300 import _lib as M
from sparse_moe_layer_topk_gb300 import inputs as I
from sparse_moe_layer_topk_gb300.layer import LatentMoELayer, weights_to_device

from gpu_util import need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


@pytest.mark.parametrize("wgrad", [M.MOE_DTYPE_F32, M.MOE_DTYPE_BF16])
def test_layer_with_no_tokens(wgrad):
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
