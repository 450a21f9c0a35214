"""The FP8 cache of the GMM outputs (moe_grouped_swiglu[_bwd]_fp8cache and
LatentMoELayer(fp8_cache=True)) against the oracle's FP8 cache on the same
seeded inputs (GPU). The cached bytes and scales are decoded here from the
E4M3 format's bit fields; gradients use the bf16 I/O tolerances."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from sparse_moe_layer_topk_gb300 import _lib as M
from sparse_moe_layer_topk_gb300 import inputs as I
from sparse_moe_layer_topk_gb300.layer import LatentMoELayer, weights_to_device

from gpu_util import check_close, dev, f64, need_gpu

pytestmark = pytest.mark.gpu

GRAD_NAMES = {"Wr": "dWr", "W_dn": "dW_dn", "W13": "dW13", "W2": "dW2", "W13_sh": "dW13_sh",
              "W2_sh": "dW2_sh", "W_up": "dW_up"}


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _bf16(seed, *shape, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


def _e4m3_values():
    """Value of every E4M3 byte: sign, 4 exponent bits (bias 7), 3 mantissa bits;
    exponent 0 is subnormal, exponent 15 with mantissa 7 is NaN."""
    lut = np.zeros(256)
    for c in range(256):
        sgn, e, m = c >> 7, (c >> 3) & 15, c & 7
        v = np.nan if (e == 15 and m == 7) else (m * 2.0 ** -9 if e == 0
                                                 else (1 + m / 8) * 2.0 ** (e - 7))
        lut[c] = -v if sgn else v
    return lut


def _decode(gu8, scale):
    """The cache's g|u values ([R][2f]: g, then u): each row's bytes hold 16-feature
    groups of g and u in turn (32 bytes per 16 features); E4M3 byte value times its
    block's scale."""
    b = gu8.cpu().numpy()
    R, f2 = b.shape
    grp = b.reshape(R, f2 // 32, 2, 16)
    vals = _e4m3_values()[np.concatenate([grp[:, :, 0, :].reshape(R, -1),
                                          grp[:, :, 1, :].reshape(R, -1)], axis=1)]
    return vals * np.repeat(scale.cpu().numpy().astype(np.float64), O.FP8_BLOCK, axis=1)


def _oracle_cache(z, W13, W2, offsets, f):
    """The oracle's FP8 cache of every expert's g and u (dequantized) and scales."""
    R = int(offsets[-1])
    g_d, u_d = np.zeros((R, f)), np.zeros((R, f))
    sc = np.ones((R, 2 * f // O.FP8_BLOCK))
    nb = f // O.FP8_BLOCK
    for e in range(len(offsets) - 1):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b == a:
            continue
        _, g, u, _ = O.swiglu_expert(z[a:b], W13[e], W2[e], True)
        qg, sg = O.fp8_block_quantize(g)
        qu, su = O.fp8_block_quantize(u)
        g_d[a:b], u_d[a:b] = O.fp8_block_dequantize(qg, sg), O.fp8_block_dequantize(qu, su)
        sc[a:b, :nb], sc[a:b, nb:] = sg, su
    return g_d, u_d, sc


@pytest.mark.parametrize("counts,l,f", [
    ([0, 1, 63, 64, 65, 127, 128, 129, 300, 0, 256, 5], 256, 128),
    ([300, 0, 555, 1, 40], 1024, 512),
])
def test_grouped_swiglu_fp8cache_forward_and_backward(counts, l, f):
    counts = np.asarray(counts)
    E = len(counts)
    offsets = O.expert_offsets(counts)
    sched = O.m_tiles_schedule(counts, 128)
    R = int(offsets[-1])
    z = _bf16(30, R, l)
    W13 = _bf16(31, E, l, 2 * f, std=0.02)
    W2 = _bf16(32, E, f, l, std=0.02)
    row_w = torch.rand(R, generator=torch.Generator().manual_seed(33)) * 0.2 + 0.01
    off_d, sch_d = dev(torch.from_numpy(offsets).int()), dev(torch.from_numpy(sched).int())
    zd, W13d, W2d, rwd = dev(z), dev(W13), dev(W2), dev(row_w)
    bf = lambda *s: torch.empty(*s, dtype=torch.bfloat16, device="cuda")  # noqa: E731
    gu, h0, y0, h1, y1 = bf(R, 2 * f), bf(R, f), bf(R, l), bf(R, f), bf(R, l)
    gu8 = torch.empty(R, 2 * f, dtype=torch.uint8, device="cuda")
    sc = torch.empty(R, 2 * f // O.FP8_BLOCK, dtype=torch.float32, device="cuda")
    M.moe_grouped_swiglu(zd, W13d, W2d, off_d, sch_d, rwd, E, R, l, f, gu, h0, y0)
    M.moe_grouped_swiglu_fp8cache(zd, W13d, W2d, off_d, sch_d, rwd, E, R, l, f, gu8, sc, h1, y1)
    torch.cuda.synchronize()
    # h and y do not depend on how g|u is cached
    assert torch.equal(h0, h1) and torch.equal(y0, y1)
    # the cache against the oracle's: scales equal, values equal but for rare
    # rounding ties that fp32 and fp64 accumulation put on different sides
    zr = f64(z)
    g_ref, u_ref, sc_ref = _oracle_cache(zr, W13, W2, offsets, f)
    np.testing.assert_array_equal(sc.cpu().numpy(), sc_ref)
    got = _decode(gu8, sc)
    ref = np.concatenate([g_ref, u_ref], axis=1)
    assert np.all(np.isfinite(got))
    same = got == ref
    assert same.mean() > 0.999, same.mean()
    step = np.abs(ref) * 2.0 ** -3 + np.repeat(sc_ref, O.FP8_BLOCK, axis=1) * 2.0 ** -9
    assert np.all(np.abs(got - ref) <= step)
    # backward reading the cache
    dy = _bf16(34, R, l)
    dz = torch.empty(R, l, dtype=torch.bfloat16, device="cuda")
    drw = torch.empty(R, dtype=torch.float32, device="cuda")
    dW13 = torch.empty(E, l, 2 * f, dtype=torch.float32, device="cuda")
    dW2 = torch.empty(E, f, l, dtype=torch.float32, device="cuda")
    wsb = M.moe_workspace_size(M.MOE_OP_GROUPED_SWIGLU_BWD, T=R, k=1, f=f)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    M.moe_grouped_swiglu_bwd_fp8cache(dev(dy), zd, W13d, W2d, gu8, sc, h1, rwd, off_d, sch_d, E,
                                      R, l, f, dz, drw, dW13, dW2, M.MOE_DTYPE_F32, ws, wsb)
    torch.cuda.synchronize()
    dyr, rw = f64(dy), f64(row_w)
    ref_dz, ref_dw = np.zeros((R, l)), np.zeros(R)
    ref_dW13, ref_dW2 = np.zeros((E, l, 2 * f)), np.zeros((E, f, l))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b == a:
            continue
        o = O.swiglu_expert(zr[a:b], W13[e], W2[e])
        ref_dw[a:b] = np.einsum("rc,rc->r", dyr[a:b], o)
        ref_dz[a:b], ref_dW13[e], ref_dW2[e] = O.swiglu_expert_backward(
            zr[a:b], W13[e], W2[e], dyr[a:b] * rw[a:b, None], (g_ref[a:b], u_ref[a:b]))
    check_close("dz_perm", f64(dz), ref_dz)
    check_close("d_row_w", f64(drw), ref_dw, scale_by_max=True)  # a sum over l columns
    check_close("dW13", f64(dW13), ref_dW13, scale_by_max=True)
    check_close("dW2", f64(dW2), ref_dW2, scale_by_max=True)
    for e in range(E):
        if counts[e] == 0:
            assert not dW13[e].any() and not dW2[e].any()


def test_fp8cache_needs_128_wide_expert_ffn():
    x = torch.zeros(64, dtype=torch.uint8, device="cuda")
    with pytest.raises(M.MoEError, match="UNSUPPORTED|unsupported"):
        M.moe_grouped_swiglu_fp8cache(x, x, x, x, x, None, 2, 8, 64, 64, x, x, x, x)


def test_layer_fp8cache_every_output_and_gradient():
    """The whole layer with the routed experts' g|u kept in FP8 against the
    oracle layer with the same cache (a tiny configuration with f = 128)."""
    cfg = dataclasses.replace(I.CONFIGS[0], name="tiny_T256_E64_top4_f128", f=128)
    inp = I.make_layer_inputs(cfg)
    layer = LatentMoELayer(weights_to_device(inp), cfg.T, cfg.k, M.MOE_DTYPE_F32, fp8_cache=True)
    layer.forward(inp["x"].cuda())
    layer.backward(inp["g"].cuda())
    torch.cuda.synchronize()
    assert int(layer.err.item()) == 0
    fwd = O.layer_forward(inp)
    gi = layer.topk_idx.cpu().numpy()
    np.testing.assert_array_equal(np.sort(gi, 1), np.sort(O.topk_select(fwd["L"], cfg.k), 1))
    check_close("out", f64(layer.out), fwd["out"])
    # Staged backward: the cache puts g and u on a grid of 2^-3 relative steps,
    # so a 2^-9 difference in the latent z they come from (the GPU keeps z in
    # bf16, the oracle does not round it) moves a few per cent of them to the
    # neighbouring grid point. The oracle's backward therefore starts from the
    # GPU's z, which puts both caches' rounding decisions on the same values.
    z_gpu = f64(layer.z)
    staged = dict(fwd, z=z_gpu, z_perm=z_gpu[fwd["token_of"]])
    bwd = O.layer_backward(inp, staged, fp8_cache=True)
    check_close("dx", f64(layer.dx), bwd["dx"])
    check_close("d_w", f64(layer.d_topk_w), bwd["d_w"])
    for wn, gn in GRAD_NAMES.items():
        check_close(gn, f64(layer.grads[wn]), bwd[gn], scale_by_max=True)
