"""Out-of-bounds write checks (GPU): every output of an entry point lives inside
a larger buffer whose 4 KB before and after it hold a byte pattern, and the
pattern must be intact after the call. The shapes are the ragged ones (row
counts that are not multiples of the tile, N tails narrower than a tile, an
odd number of 128-row blocks for the CTA pairs, empty and one-row experts)
where a clipped TMA store or a scattered index write would spill first."""
import math

import numpy as np
import pytest
import torch

import oracle as O
from sparse_moe_layer_topk_gb300 import _lib as M
from sparse_moe_layer_topk_gb300 import inputs as I

from gpu_util import dev, need_gpu

pytestmark = pytest.mark.gpu

PAD = 4096    # guard bytes on each side (a multiple of 16: the inner tensor stays aligned)
CANARY = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


class Guarded:
    """Output tensors carved out of padded buffers, and the check of their guards."""

    def __init__(self):
        self.bufs = []

    def empty(self, *shape, dtype):
        n = math.prod(shape)
        es = torch.empty(0, dtype=dtype).element_size()
        raw = torch.full((2 * PAD + n * es,), CANARY, dtype=torch.uint8, device="cuda")
        self.bufs.append((raw, n * es))
        return raw[PAD:PAD + n * es].view(dtype).view(*shape)

    def check(self):
        torch.cuda.synchronize()
        for i, (raw, nbytes) in enumerate(self.bufs):
            head, tail = raw[:PAD], raw[PAD + nbytes:]
            bad_h = int((head != CANARY).sum().item())
            bad_t = int((tail != CANARY).sum().item())
            assert bad_h == 0 and bad_t == 0, f"buffer {i}: {bad_h} bytes before, {bad_t} after"


def _bf16(seed, *shape, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


@pytest.mark.parametrize("M_,K,N", [(300, 256, 192), (1100, 256, 512), (129, 384, 256)])
def test_latent_proj_writes_stay_in_bounds(M_, K, N):
    g = Guarded()
    x, W, dout = _bf16(1, M_, K), _bf16(2, K, N, std=0.02), _bf16(3, M_, N)
    out = g.empty(M_, N, dtype=torch.bfloat16)
    din = g.empty(M_, K, dtype=torch.bfloat16)
    dW = g.empty(K, N, dtype=torch.float32)
    dWb = g.empty(K, N, dtype=torch.bfloat16)
    M.moe_latent_proj(dev(x), dev(W), M_, K, N, out)
    M.moe_latent_proj_bwd(dev(dout), dev(x), dev(W), M_, K, N, din, dW, M.MOE_DTYPE_F32)
    M.moe_latent_proj_bwd(dev(dout), dev(x), dev(W), M_, K, N, None, dWb, M.MOE_DTYPE_BF16)
    g.check()


def test_router_and_topk_writes_stay_in_bounds():
    T, d, E, k = 333, 512, 192, 16
    g = Guarded()
    L = g.empty(T, E, dtype=torch.float32)
    idx = g.empty(T, k, dtype=torch.int32)
    w = g.empty(T, k, dtype=torch.float32)
    s = g.empty(T, k, dtype=torch.float32)
    M.moe_router_logits(dev(_bf16(4, T, d)), dev(_bf16(5, d, E, std=0.02)), T, d, E, L)
    M.moe_topk_from_logits(L, None, T, E, k, idx, w, s, None)
    g.check()


def test_permute_and_combine_writes_stay_in_bounds():
    T, E, k, l = 300, 37, 5, 128
    R = T * k
    idx = dev(I.make_topk_ids(331, T, E, k, skew=2.0))
    z = dev(_bf16(9, T, l))
    tw = dev(torch.rand(T, k, generator=torch.Generator().manual_seed(2)))
    g = Guarded()
    z_perm = g.empty(R, l, dtype=torch.bfloat16)
    counts = g.empty(E, dtype=torch.int32)
    offsets = g.empty(E + 1, dtype=torch.int32)
    slot_of = g.empty(T, k, dtype=torch.int32)
    token_of = g.empty(R, dtype=torch.int32)
    tile_sched = g.empty(E + 1, dtype=torch.int32)
    row_w = g.empty(R, dtype=torch.float32)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    wsb = M.moe_workspace_size(M.MOE_OP_PERMUTE, T=T, E=E)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    M.moe_permute(z, idx, tw, T, l, E, k, z_perm, counts, offsets, slot_of, token_of, tile_sched,
                  row_w, ws, wsb, err)
    y_sh = dev(_bf16(13, T, l))
    y = g.empty(T, l, dtype=torch.bfloat16)
    M.moe_unpermute_combine(z_perm, slot_of, y_sh, T, k, l, y)
    dy_perm = g.empty(R, l, dtype=torch.bfloat16)
    M.moe_unpermute_combine_bwd(y_sh, token_of, T, k, l, dy_perm)
    dz = g.empty(T, l, dtype=torch.bfloat16)
    M.moe_permute_bwd(dy_perm, slot_of, y_sh, T, k, l, dz)
    g.check()
    assert int(err.item()) == 0


def test_grouped_swiglu_writes_stay_in_bounds():
    counts = np.array([0, 1, 127, 128, 129, 300, 0, 256, 5])
    E, l, f = len(counts), 128, 64
    offsets = O.expert_offsets(counts)
    sched = O.m_tiles_schedule(counts, 128)
    R = int(offsets[-1])
    z_perm = dev(_bf16(20, R, l))
    W13, W2 = dev(_bf16(21, E, l, 2 * f, std=0.02)), dev(_bf16(22, E, f, l, std=0.02))
    row_w = dev(torch.rand(R, generator=torch.Generator().manual_seed(3)) * 0.2 + 0.01)
    off_d = dev(torch.from_numpy(offsets).int())
    sch_d = dev(torch.from_numpy(sched).int())
    g = Guarded()
    gu = g.empty(R, 2 * f, dtype=torch.bfloat16)
    h = g.empty(R, f, dtype=torch.bfloat16)
    y = g.empty(R, l, dtype=torch.bfloat16)
    M.moe_grouped_swiglu(z_perm, W13, W2, off_d, sch_d, row_w, E, R, l, f, gu, h, y)
    dy = dev(_bf16(23, R, l))
    dz = g.empty(R, l, dtype=torch.bfloat16)
    d_row_w = g.empty(R, dtype=torch.float32)
    dW13 = g.empty(E, l, 2 * f, dtype=torch.float32)
    dW2 = g.empty(E, f, l, dtype=torch.float32)
    wsb = M.moe_workspace_size(M.MOE_OP_GROUPED_SWIGLU_BWD, T=R, k=1, f=f)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    M.moe_grouped_swiglu_bwd(dy, z_perm, W13, W2, gu, h, row_w, off_d, sch_d, E, R, l, f, dz,
                             d_row_w, dW13, dW2, M.MOE_DTYPE_F32, ws, wsb)
    g.check()


def test_grouped_swiglu_fp8cache_writes_stay_in_bounds():
    """The FP8 cache's bytes and scales (32-byte TMA rows, per-thread stores for the
    ragged row blocks) and the backward that reads them."""
    counts = np.array([0, 1, 63, 64, 65, 127, 129, 300, 0, 5])
    E, l, f = len(counts), 128, 128
    offsets = O.expert_offsets(counts)
    sched = O.m_tiles_schedule(counts, 128)
    R = int(offsets[-1])
    z_perm = dev(_bf16(30, R, l))
    W13, W2 = dev(_bf16(31, E, l, 2 * f, std=0.02)), dev(_bf16(32, E, f, l, std=0.02))
    row_w = dev(torch.rand(R, generator=torch.Generator().manual_seed(4)) * 0.2 + 0.01)
    off_d = dev(torch.from_numpy(offsets).int())
    sch_d = dev(torch.from_numpy(sched).int())
    g = Guarded()
    gu8 = g.empty(R, 2 * f, dtype=torch.uint8)
    sc = g.empty(R, 2 * f // O.FP8_BLOCK, dtype=torch.float32)
    h = g.empty(R, f, dtype=torch.bfloat16)
    y = g.empty(R, l, dtype=torch.bfloat16)
    M.moe_grouped_swiglu_fp8cache(z_perm, W13, W2, off_d, sch_d, row_w, E, R, l, f, gu8, sc, h, y)
    dy = dev(_bf16(33, R, l))
    dz = g.empty(R, l, dtype=torch.bfloat16)
    d_row_w = g.empty(R, dtype=torch.float32)
    dW13 = g.empty(E, l, 2 * f, dtype=torch.float32)
    dW2 = g.empty(E, f, l, dtype=torch.float32)
    wsb = M.moe_workspace_size(M.MOE_OP_GROUPED_SWIGLU_BWD, T=R, k=1, f=f)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    M.moe_grouped_swiglu_bwd_fp8cache(dy, z_perm, W13, W2, gu8, sc, h, row_w, off_d, sch_d, E, R,
                                      l, f, dz, d_row_w, dW13, dW2, M.MOE_DTYPE_F32, ws, wsb)
    g.check()


@pytest.mark.parametrize("T,l,f,S", [(77, 256, 128, 3), (1100, 512, 256, 2)])
def test_shared_swiglu_writes_stay_in_bounds(T, l, f, S):
    z = dev(_bf16(30, T, l))
    W13, W2 = dev(_bf16(31, S, l, 2 * f, std=0.02)), dev(_bf16(32, S, f, l, std=0.02))
    g = Guarded()
    gu = g.empty(T, S * 2 * f, dtype=torch.bfloat16)
    h = g.empty(T, S * f, dtype=torch.bfloat16)
    y = g.empty(T, l, dtype=torch.bfloat16)
    M.moe_shared_swiglu(z, W13, W2, T, l, f, S, gu, h, y)
    dy = dev(_bf16(33, T, l))
    dz = g.empty(T, l, dtype=torch.bfloat16)
    dW13 = g.empty(S, l, 2 * f, dtype=torch.float32)
    dW2 = g.empty(S, f, l, dtype=torch.float32)
    wsb = M.moe_workspace_size(M.MOE_OP_SHARED_SWIGLU_BWD, T=T, l=l, f=f, S=S)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    M.moe_shared_swiglu_bwd(dy, z, W13, W2, gu, h, T, l, f, S, dz, dW13, dW2, M.MOE_DTYPE_F32, ws,
                            wsb)
    g.check()


def test_bounded_wait_gives_up_sets_the_flag_and_leaves_the_gpu_usable():
    """The library's mbarrier wait, with a 1 ms limit, on a barrier that nothing
    arrives at: the kernel returns, MOE_FLAG_TIMEOUT is set, the wait lasted at
    least the limit (and not unboundedly longer), and a layer step right after
    still matches the fp64 oracle with a clean error word."""
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    M.moe_diag_wait_timeout(1_000_000, err, waited)
    torch.cuda.synchronize()
    assert int(err.item()) == M.MOE_FLAG_TIMEOUT
    assert 1_000_000 <= int(waited.item()) < 200_000_000
    with pytest.raises(M.MoEError):
        M.moe_diag_wait_timeout(10, err, waited)   # limit out of range: nothing launched

    from sparse_moe_layer_topk_gb300.layer import LatentMoELayer, weights_to_device
    from gpu_util import check_close, f64
    inp = I.make_layer_inputs(0)
    cfg = inp["cfg"]
    layer = LatentMoELayer(weights_to_device(inp), cfg.T, cfg.k, M.MOE_DTYPE_F32)
    out = layer.forward(inp["x"].cuda())
    dx = layer.backward(inp["g"].cuda())
    torch.cuda.synchronize()
    assert int(layer.err.item()) == 0
    fwd = O.layer_forward(inp)
    bwd = O.layer_backward(inp, fwd)
    check_close("out", f64(out), fwd["out"])
    check_close("dx", f64(dx), bwd["dx"])
