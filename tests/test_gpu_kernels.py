"""Per-entry-point parity of libmoe against the fp64 oracle on identical
seeded inputs (GPU). Integer outputs bit-exact, floats within the bf16 I/O
tolerances (max-abs 2e-2, relative Frobenius 1e-2)."""
import numpy as np
import pytest
import torch

import oracle as O
from sparse_moe_layer_topk_gb300 import _lib as M
from sparse_moe_layer_topk_gb300 import inputs as I

from gpu_util import check_close, dev, f64, need_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    need_gpu()


def _bf16(seed, *shape, std=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(*shape, generator=g) * std).to(torch.bfloat16)


# ---------------------------------------------------------------- GEMM engine

@pytest.mark.parametrize("M_,K,N", [(300, 256, 192), (128, 64, 64), (1000, 512, 1024), (5, 128, 256),
                                    (700, 1024, 512), (2000, 1024, 768), (1100, 256, 512),
                                    (129, 384, 256)])
def test_latent_proj_and_bwd(M_, K, N):
    """Every operand layout of the tcgen05 engine: A K-major / B MN-major
    (forward), B K-major (dgrad), A and B MN-major (wgrad); ragged M and an
    N tail narrower than the tile; 256-wide tiles run on CTA pairs, including
    an odd number of 128-row blocks (the last pair's second CTA has no rows)."""
    x = _bf16(1, M_, K)
    W = _bf16(2, K, N, std=0.02)  # |out| ~ 1: bf16 output rounding stays below 2e-2
    dout = _bf16(3, M_, N)
    out = torch.empty(M_, N, dtype=torch.bfloat16, device="cuda")
    M.moe_latent_proj(dev(x), dev(W), M_, K, N, out)
    din = torch.empty(M_, K, dtype=torch.bfloat16, device="cuda")
    dW = torch.empty(K, N, dtype=torch.float32, device="cuda")
    M.moe_latent_proj_bwd(dev(dout), dev(x), dev(W), M_, K, N, din, dW, M.MOE_DTYPE_F32)
    dWb = torch.empty(K, N, dtype=torch.bfloat16, device="cuda")
    M.moe_latent_proj_bwd(dev(dout), dev(x), dev(W), M_, K, N, None, dWb, M.MOE_DTYPE_BF16)
    torch.cuda.synchronize()
    xr, Wr, dr = f64(x), f64(W), f64(dout)
    check_close("out", f64(out), xr @ Wr)
    check_close("din", f64(din), dr @ Wr.T)
    check_close("dW", f64(dW), xr.T @ dr, scale_by_max=True)
    check_close("dW_bf16", f64(dWb), xr.T @ dr, scale_by_max=True)


def test_router_logits():
    T, d, E = 333, 512, 192
    x = _bf16(4, T, d)
    Wr = _bf16(5, d, E, std=0.02)
    L = torch.empty(T, E, dtype=torch.float32, device="cuda")
    M.moe_router_logits(dev(x), dev(Wr), T, d, E, L)
    torch.cuda.synchronize()
    ref = O.router_logits(x, Wr)
    err = np.abs(f64(L) - ref).max()
    assert err < 1e-4, err



@pytest.mark.parametrize("T,d,E,l,k", [(300, 256, 256, 256, 4), (1100, 512, 384, 512, 8),
                                       (2048, 4096, 896, 1024, 16), (100, 256, 256, 256, 4),
                                       (300, 256, 64, 256, 4), (1, 128, 128, 64, 2)])
def test_route_topk_latent_equals_the_separate_calls(T, d, E, l, k):
    """The router and the latent down-projection as one GEMM over [Wr | W_dn]
    (T > 128, E a multiple of 128: columns of the 256-wide tile that straddles E
    come from both weights) give the separate calls' logits, z and selection bit
    for bit; the other shapes take the separate calls inside the entry point.
    The logits against the oracle as in test_router_logits."""
    x = dev(_bf16(40, T, d))
    Wr = dev(_bf16(41, d, E, std=0.02))
    W_dn = dev(_bf16(42, d, l, std=0.02))
    wsb = M.moe_workspace_size(M.MOE_OP_ROUTE_TOPK, T=T, d=d, E=E, k=k)
    ws0 = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    ws1 = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    out = []
    for ws, fused in ((ws0, False), (ws1, True)):
        idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
        w = torch.empty(T, k, dtype=torch.float32, device="cuda")
        sg = torch.empty(T, k, dtype=torch.float32, device="cuda")
        z = torch.empty(T, l, dtype=torch.bfloat16, device="cuda")
        if fused:
            M.moe_route_topk_latent(x, Wr, None, W_dn, T, d, E, k, l, idx, w, sg, z, ws, wsb)
        else:
            M.moe_route_topk(x, Wr, None, T, d, E, k, idx, w, sg, ws, wsb)
            M.moe_latent_proj(x, W_dn, T, d, l, z)
        out.append((ws[: T * E * 4].view(torch.float32).view(T, E).clone(), idx, w, sg, z))
    torch.cuda.synchronize()
    for name, a, b in zip(("logits", "topk_idx", "topk_w", "topk_s", "z"), out[0], out[1]):
        assert torch.equal(a, b), name
    err = np.abs(f64(out[1][0]) - O.router_logits(x.cpu(), Wr.cpu())).max()
    assert err < 1e-4, err

# ---------------------------------------------------------------- top-k

@pytest.mark.parametrize("T,E,k,ties,bias", [
    (513, 64, 4, False, False), (300, 896, 16, False, True), (257, 896, 16, True, False),
    (64, 40, 32, False, False), (100, 1024, 32, True, True), (33, 17, 1, False, False)])
def test_topk_from_logits_bit_exact(T, E, k, ties, bias):
    L = I.make_logits(7 + T, T, E, ties=ties)
    b = (torch.randn(E, generator=torch.Generator().manual_seed(3)) * 0.5).float() if bias else None
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    s = torch.empty(T, k, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_topk_from_logits(dev(L), dev(b) if bias else None, T, E, k, idx, w, s, err)
    torch.cuda.synchronize()
    # the selection is decided on the fp32 value logit + bias on both sides
    v32 = (L.numpy() + b.numpy()[None, :]).astype(np.float32) if bias else L.numpy()
    ref_idx = O.topk_select(v32.astype(np.float64), k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    ref_w, ref_s = O.routing_weights(v32.astype(np.float64), ref_idx)
    np.testing.assert_allclose(s.cpu().numpy(), ref_s, rtol=2e-6, atol=1e-7)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=3e-6, atol=1e-7)
    assert int(err.item()) == 0


@pytest.mark.parametrize("neg_zero_bias", [False, True])
def test_topk_signed_zero_ties(neg_zero_bias):
    """-0.0 and +0.0 are equal logits: when they tie at the k-th place the
    lower expert id wins, whatever the signs. With a bias of -0.0 the summed
    value keeps the sign of the logit (-0 + -0 = -0), so signed zeros reach
    the selection itself."""
    T, E, k = 97, 64, 4
    rng = np.random.default_rng(5)
    L = -rng.uniform(1.0, 5.0, size=(T, E)).astype(np.float32)
    for t in range(T):
        top = rng.choice(E, size=k - 1, replace=False)
        L[t, top] = rng.uniform(1.0, 2.0, size=k - 1)
        rest = np.setdiff1d(np.arange(E), top)
        zeros = rng.choice(rest, size=6, replace=False)
        L[t, zeros] = np.where(rng.random(6) < 0.5, np.float32(-0.0), np.float32(0.0))
    # the lowest-id zero of some tokens is a -0.0 that an order with -0 < +0 would skip
    assert any(np.signbit(L[t, np.where(L[t] == 0)[0].min()]) for t in range(T))
    b = torch.full((E,), -0.0, dtype=torch.float32) if neg_zero_bias else None
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    s = torch.empty(T, k, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_topk_from_logits(dev(torch.from_numpy(L)), dev(b) if b is not None else None, T, E, k,
                           idx, w, s, err)
    torch.cuda.synchronize()
    ref_idx = O.topk_select(L.astype(np.float64), k)
    np.testing.assert_array_equal(idx.cpu().numpy(), ref_idx)
    ref_w, ref_s = O.routing_weights(L.astype(np.float64), ref_idx)
    np.testing.assert_allclose(s.cpu().numpy(), ref_s, rtol=2e-6, atol=1e-7)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=3e-6, atol=1e-7)
    assert int(err.item()) == 0


def test_topk_flags_nonfinite():
    L = I.make_logits(1, 16, 64)
    L[3, 5] = float("nan")
    idx = torch.empty(16, 4, dtype=torch.int32, device="cuda")
    w = torch.empty(16, 4, dtype=torch.float32, device="cuda")
    s = torch.empty(16, 4, dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    M.moe_topk_from_logits(dev(L), None, 16, 64, 4, idx, w, s, err)
    torch.cuda.synchronize()
    assert int(err.item()) & M.MOE_FLAG_NONFINITE


# ---------------------------------------------------------------- permute

def _run_permute(idx, E, l, z=None, topk_w=None):
    T, k = idx.shape
    R = T * k
    out = dict(
        counts=torch.empty(E, dtype=torch.int32, device="cuda"),
        offsets=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
        slot_of=torch.empty(T, k, dtype=torch.int32, device="cuda"),
        token_of=torch.empty(R, dtype=torch.int32, device="cuda"),
        tile_sched=torch.empty(E + 1, dtype=torch.int32, device="cuda"),
        row_w=torch.empty(R, dtype=torch.float32, device="cuda"),
        z_perm=torch.empty(R, l, dtype=torch.bfloat16, device="cuda"),
        err=torch.zeros(1, dtype=torch.int32, device="cuda"),
    )
    wsb = M.moe_workspace_size(M.MOE_OP_PERMUTE, T=T, E=E)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    M.moe_permute(dev(z) if z is not None else None, dev(idx), dev(topk_w) if topk_w is not None
                  else None, T, l, E, k, out["z_perm"], out["counts"], out["offsets"],
                  out["slot_of"], out["token_of"], out["tile_sched"], out["row_w"], ws, wsb,
                  out["err"])
    torch.cuda.synchronize()
    return {n: v.cpu() for n, v in out.items()}


@pytest.mark.parametrize("T,E,k,skew", [(256, 64, 4, 0.0), (4096, 896, 16, 0.0),
                                        (4096, 896, 16, 1.1), (300, 37, 5, 2.0),
                                        (1, 896, 16, 0.0), (700, 8, 8, 0.0)])
def test_permute_bit_exact(T, E, k, skew):
    idx = I.make_topk_ids(31 + T, T, E, k, skew=skew)
    l = 128
    z = _bf16(9, T, l)
    tw = torch.rand(T, k, generator=torch.Generator().manual_seed(2))
    g = _run_permute(idx, E, l, z, tw)
    slot_of, token_of, offsets = O.permutation_maps(idx.numpy(), E)
    counts = O.expert_counts(idx.numpy(), E)
    np.testing.assert_array_equal(g["counts"].numpy(), counts)
    np.testing.assert_array_equal(g["offsets"].numpy(), offsets)
    np.testing.assert_array_equal(g["slot_of"].numpy(), slot_of)
    np.testing.assert_array_equal(g["token_of"].numpy(), token_of)
    np.testing.assert_array_equal(g["tile_sched"].numpy(), O.m_tiles_schedule(counts, 128))
    row_w = np.empty(T * k, dtype=np.float32)
    row_w[slot_of.reshape(-1)] = tw.numpy().reshape(-1)
    np.testing.assert_array_equal(g["row_w"].numpy(), row_w)
    np.testing.assert_array_equal(g["z_perm"].view(torch.int16).numpy(),
                                  z[torch.from_numpy(token_of)].view(torch.int16).numpy())
    assert int(g["err"].item()) == 0


def test_permute_flags_bad_ids():
    idx = I.make_topk_ids(5, 64, 32, 4)
    idx[7, 2] = 40          # out of range
    idx[9, 1] = idx[9, 0]   # repeated id
    g = _run_permute(idx, 32, 64)
    assert int(g["err"].item()) & M.MOE_FLAG_BAD_EXPERT
    assert g["slot_of"][7, 2].item() == -1


def test_permute_then_combine_identity():
    """Unit weights and identity experts: combine(permute(z)) == k z exactly
    (sums of k equal bf16 values are exact in fp32 for k a power of two)."""
    T, E, k, l = 500, 64, 4, 256
    idx = I.make_topk_ids(8, T, E, k)
    z = _bf16(10, T, l)
    g = _run_permute(idx, E, l, z)
    y = torch.empty(T, l, dtype=torch.bfloat16, device="cuda")
    M.moe_unpermute_combine(dev(g["z_perm"]), dev(g["slot_of"]), None, T, k, l, y)
    torch.cuda.synchronize()
    assert torch.equal(y.cpu(), (z.float() * k).to(torch.bfloat16))


def test_combine_and_gather_rows():
    T, k, l, R = 300, 6, 192, 300 * 6
    idx = I.make_topk_ids(11, T, 50, k)
    slot_of, token_of, _ = O.permutation_maps(idx.numpy(), 50)
    y_perm = _bf16(12, R, l)
    y_sh = _bf16(13, T, l)
    y = torch.empty(T, l, dtype=torch.bfloat16, device="cuda")
    M.moe_unpermute_combine(dev(y_perm), dev(torch.from_numpy(slot_of).int()), dev(y_sh), T, k, l,
                            y)
    dy_perm = torch.empty(R, l, dtype=torch.bfloat16, device="cuda")
    M.moe_unpermute_combine_bwd(dev(y_sh), dev(torch.from_numpy(token_of).int()), T, k, l, dy_perm)
    torch.cuda.synchronize()
    ref = O.combine(y_perm, slot_of, y_sh)
    # fp32 sum of bf16 terms, one final bf16 rounding (half an ulp = 2^-9 relative)
    assert np.all(np.abs(f64(y) - ref) <= 2.0 ** -8 * np.abs(ref) + 1e-6)
    assert torch.equal(dy_perm.cpu(), y_sh[torch.from_numpy(token_of)])


# ---------------------------------------------------------------- experts

def _segments(counts):
    counts = np.asarray(counts)
    offsets = O.expert_offsets(counts)
    sched = O.m_tiles_schedule(counts, 128)
    return offsets, sched


@pytest.mark.parametrize("counts,l,f", [
    ([0, 1, 127, 128, 129, 300, 0, 256, 5], 128, 64),
    ([73] * 20 + [0, 2, 1], 256, 128),
    ([300, 0, 555, 1], 1024, 512),
])
def test_grouped_swiglu_fwd_bwd(counts, l, f):
    E = len(counts)
    offsets, sched = _segments(counts)
    R = int(offsets[-1])
    z_perm = _bf16(20, R, l)
    W13 = _bf16(21, E, l, 2 * f, std=0.02)
    W2 = _bf16(22, E, f, l, std=0.02)
    row_w = torch.rand(R, generator=torch.Generator().manual_seed(3)) * 0.2 + 0.01
    gu = torch.empty(R, 2 * f, dtype=torch.bfloat16, device="cuda")
    h = torch.empty(R, f, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(R, l, dtype=torch.bfloat16, device="cuda")
    off_d = dev(torch.from_numpy(offsets).int())
    sch_d = dev(torch.from_numpy(sched).int())
    M.moe_grouped_swiglu(dev(z_perm), dev(W13), dev(W2), off_d, sch_d, dev(row_w), E, R, l, f, gu,
                         h, y)
    torch.cuda.synchronize()
    zr = f64(z_perm)
    ref_y = O.grouped_swiglu(zr, W13, W2, offsets, row_w)
    check_close("y_perm", f64(y), ref_y)
    # g/u/h against the oracle's expert pieces
    ref_g = np.zeros((R, f)); ref_u = np.zeros((R, f)); ref_h = np.zeros((R, f))
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if b > a:
            _, ref_g[a:b], ref_u[a:b], ref_h[a:b] = O.swiglu_expert(zr[a:b], W13[e], W2[e], True)
    check_close("g", f64(gu[:, :f]), ref_g)
    check_close("u", f64(gu[:, f:]), ref_u)
    check_close("h", f64(h), ref_h)
    # backward on the GPU's own forward activations
    dy = _bf16(23, R, l)
    dz = torch.empty(R, l, dtype=torch.bfloat16, device="cuda")
    d_row_w = torch.empty(R, dtype=torch.float32, device="cuda")
    dW13 = torch.empty(E, l, 2 * f, dtype=torch.float32, device="cuda")
    dW2 = torch.empty(E, f, l, dtype=torch.float32, device="cuda")
    wsb = M.moe_workspace_size(M.MOE_OP_GROUPED_SWIGLU_BWD, T=R, k=1, f=f)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    M.moe_grouped_swiglu_bwd(dev(dy), dev(z_perm), dev(W13), dev(W2), gu, h, dev(row_w), off_d,
                             sch_d, E, R, l, f, dz, d_row_w, dW13, dW2, M.MOE_DTYPE_F32, ws, wsb)
    torch.cuda.synchronize()
    dyr = f64(dy)
    ref_dz = np.zeros((R, l)); ref_dw = np.zeros(R)
    ref_dW13 = np.zeros((E, l, 2 * f)); ref_dW2 = np.zeros((E, f, l))
    for e in range(E):
        a, b = offsets[e], offsets[e + 1]
        if b == a:
            continue
        o = O.swiglu_expert(zr[a:b], W13[e], W2[e])
        ref_dw[a:b] = np.einsum("rc,rc->r", dyr[a:b], o)
        ref_dz[a:b], ref_dW13[e], ref_dW2[e] = O.swiglu_expert_backward(
            zr[a:b], W13[e], W2[e], dyr[a:b] * f64(row_w)[a:b, None])
    check_close("dz_perm", f64(dz), ref_dz)
    check_close("d_row_w", f64(d_row_w), ref_dw)
    check_close("dW13", f64(dW13), ref_dW13, scale_by_max=True)
    check_close("dW2", f64(dW2), ref_dW2, scale_by_max=True)
    for e in range(E):
        if counts[e] == 0:
            assert not dW13[e].any() and not dW2[e].any()


@pytest.mark.parametrize("T,l,f,S", [(256, 128, 64, 1), (1000, 1024, 512, 2), (77, 256, 128, 3),
                                     (4096, 1024, 512, 2), (1100, 512, 256, 2)])
def test_shared_swiglu_fwd_bwd(T, l, f, S):
    """Dense SwiGLU experts on all tokens (CTA pairs for the 256-wide tiles; T=1100
    has an odd number of 128-row blocks)."""
    z = _bf16(30, T, l)
    W13 = _bf16(31, S, l, 2 * f, std=0.02)
    W2 = _bf16(32, S, f, l, std=0.02)
    gu = torch.empty(T, S * 2 * f, dtype=torch.bfloat16, device="cuda")
    h = torch.empty(T, S * f, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(T, l, dtype=torch.bfloat16, device="cuda")
    M.moe_shared_swiglu(dev(z), dev(W13), dev(W2), T, l, f, S, gu, h, y)
    dy = _bf16(33, T, l)
    dz = torch.empty(T, l, dtype=torch.bfloat16, device="cuda")
    dW13 = torch.empty(S, l, 2 * f, dtype=torch.float32, device="cuda")
    dW2 = torch.empty(S, f, l, dtype=torch.float32, device="cuda")
    wsb = M.moe_workspace_size(M.MOE_OP_SHARED_SWIGLU_BWD, T=T, l=l, f=f, S=S)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    M.moe_shared_swiglu_bwd(dev(dy), dev(z), dev(W13), dev(W2), gu, h, T, l, f, S, dz, dW13, dW2,
                            M.MOE_DTYPE_F32, ws, wsb)
    torch.cuda.synchronize()
    zr, dyr = f64(z), f64(dy)
    ref = sum(O.swiglu_expert(zr, W13[s], W2[s]) for s in range(S))
    check_close("y_sh", f64(y), ref)
    for s in range(S):
        _, g_, u_, h_ = O.swiglu_expert(zr, W13[s], W2[s], True)
        check_close("h_sh", f64(h[:, s * f:(s + 1) * f]), h_)
        check_close("g_sh", f64(gu[:, s * 2 * f:s * 2 * f + f]), g_)
        check_close("u_sh", f64(gu[:, s * 2 * f + f:(s + 1) * 2 * f]), u_)
    ref_dz = np.zeros((T, l))
    for s in range(S):
        dzs, dW13s, dW2s = O.swiglu_expert_backward(zr, W13[s], W2[s], dyr)
        ref_dz += dzs
        check_close("dW13_sh", f64(dW13[s]), dW13s, scale_by_max=True)
        check_close("dW2_sh", f64(dW2[s]), dW2s, scale_by_max=True)
    check_close("dz_sh", f64(dz), ref_dz)


def test_route_topk_bwd():
    T, d, E, k = 300, 256, 64, 4
    x = _bf16(40, T, d)
    Wr = _bf16(41, d, E, std=0.02)
    L = O.router_logits(x, Wr)
    idx = O.topk_select(L, k)
    w, s = O.routing_weights(L, idx)
    slot_of, token_of, _ = O.permutation_maps(idx, E)
    R = T * k
    d_row_w = torch.randn(R, generator=torch.Generator().manual_seed(4)).float()
    dx = _bf16(42, T, d)
    dx_d = dev(dx)
    dWr = torch.empty(d, E, dtype=torch.float32, device="cuda")
    d_topk_w = torch.empty(T, k, dtype=torch.float32, device="cuda")
    wsb = M.moe_workspace_size(M.MOE_OP_ROUTE_TOPK_BWD, T=T, E=E)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    M.moe_route_topk_bwd(dev(d_row_w), dev(torch.from_numpy(slot_of).int()),
                         dev(torch.from_numpy(idx).int()), dev(torch.from_numpy(w).float()),
                         dev(torch.from_numpy(s).float()), dev(x), dev(Wr), T, d, E, k, d_topk_w,
                         dx_d, dWr, M.MOE_DTYPE_F32, None, None, None, 0.0, None, None, 0, ws, wsb)
    torch.cuda.synchronize()
    dw = f64(d_row_w)[slot_of]
    np.testing.assert_array_equal(d_topk_w.cpu().numpy(), d_row_w.numpy()[slot_of])
    w32, s32 = w.astype(np.float32), s.astype(np.float32)   # the values the GPU was given
    dL = O.router_backward(dw, w32, s32, idx, E)
    check_close("dx", f64(dx_d), f64(dx) + dL @ f64(Wr).T)
    check_close("dWr", f64(dWr), f64(x).T @ dL, scale_by_max=True)


def test_host_argument_errors_do_not_launch():
    with pytest.raises(M.MoEError, match="invalid argument"):
        M.moe_latent_proj(None, None, 4, 64, 64, None)
    x = torch.empty(64, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(M.MoEError, match="misaligned"):
        M.moe_latent_proj(x, x, 64, 64, 96, x)
    with pytest.raises(M.MoEError, match="workspace"):
        M.moe_route_topk(x, x, None, 64, 64, 64, 4, x, x, x, x, 16)


@pytest.mark.parametrize("T,E,k,l,f,skew", [(300, 37, 4, 128, 64, 1.5), (2048, 64, 8, 1024, 512, 0.0),
                                             (1, 16, 4, 256, 128, 0.0)])
def test_gather_fused_grouped_gemms_equal_explicit_permute(T, E, k, l, f, skew):
    """moe_grouped_swiglu[_bwd]_gather (rows copied into the GEMMs' shared-memory
    stages by the gather warps) produce bit-identical results to the explicit
    permute followed by the plain grouped calls: the same bytes land in the same
    shared-memory tiles."""
    idx = I.make_topk_ids(50 + T, T, E, k, skew=skew)
    z = _bf16(51, T, l)
    dy_lat = _bf16(52, T, l)
    tw = torch.rand(T, k, generator=torch.Generator().manual_seed(5)) * 0.2 + 0.01
    g = _run_permute(idx, E, l, z, tw)
    R = T * k
    W13 = dev(_bf16(53, E, l, 2 * f, std=0.02))
    W2 = dev(_bf16(54, E, f, l, std=0.02))
    off, sch, tok, roww = (dev(g["offsets"]), dev(g["tile_sched"]), dev(g["token_of"]),
                           dev(g["row_w"]))
    outs = []
    for fused in (False, True):
        gu = torch.empty(R, 2 * f, dtype=torch.bfloat16, device="cuda")
        h = torch.empty(R, f, dtype=torch.bfloat16, device="cuda")
        y = torch.empty(R, l, dtype=torch.bfloat16, device="cuda")
        dz = torch.empty(R, l, dtype=torch.bfloat16, device="cuda")
        drw = torch.empty(R, dtype=torch.float32, device="cuda")
        dW13 = torch.empty(E, l, 2 * f, dtype=torch.float32, device="cuda")
        dW2 = torch.empty(E, f, l, dtype=torch.float32, device="cuda")
        wsb = M.moe_workspace_size(M.MOE_OP_GROUPED_SWIGLU_BWD, T=R, k=1, f=f)
        ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
        if fused:
            M.moe_grouped_swiglu_gather(dev(z), tok, T, W13, W2, off, sch, roww, E, R, l, f, gu, h,
                                        y)
            M.moe_grouped_swiglu_bwd_gather(dev(dy_lat), dev(z), tok, T, W13, W2, gu, h, roww, off,
                                            sch, E, R, l, f, dz, drw, dW13, dW2, M.MOE_DTYPE_F32,
                                            ws, wsb)
        else:
            dy_perm = torch.empty(R, l, dtype=torch.bfloat16, device="cuda")
            M.moe_unpermute_combine_bwd(dev(dy_lat), tok, T, k, l, dy_perm)
            M.moe_grouped_swiglu(dev(g["z_perm"]), W13, W2, off, sch, roww, E, R, l, f, gu, h, y)
            M.moe_grouped_swiglu_bwd(dy_perm, dev(g["z_perm"]), W13, W2, gu, h, roww, off, sch, E,
                                     R, l, f, dz, drw, dW13, dW2, M.MOE_DTYPE_F32, ws, wsb)
        torch.cuda.synchronize()
        outs.append([t.cpu() for t in (gu, h, y, dz, drw, dW13, dW2)])
    for name, a, b in zip(("gu", "h", "y", "dz", "d_row_w", "dW13", "dW2"), *outs):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a,
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b), name


@pytest.mark.parametrize("T,E,bias", [(333, 64, False), (4096, 896, True), (1, 64, False)])
def test_router_aux_loss_and_gradient(T, E, bias):
    L = I.make_logits(60 + T, T, E)
    b = (torch.randn(E, generator=torch.Generator().manual_seed(6)) * 0.5).float() if bias else None
    p_mean = torch.empty(E, dtype=torch.float32, device="cuda")
    loss = torch.empty(1, dtype=torch.float32, device="cuda")
    wsb = M.moe_workspace_size(M.MOE_OP_ROUTER_AUX, T=T, E=E)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    Ld, bd = dev(L), (dev(b) if bias else None)
    M.moe_router_aux_loss(Ld, bd, T, E, p_mean, loss, ws, wsb)
    torch.cuda.synchronize()
    ref_p, ref_loss = O.aux_balance_loss(L.numpy(), b.numpy() if bias else None)
    np.testing.assert_allclose(p_mean.cpu().numpy(), ref_p, rtol=2e-5, atol=1e-9)
    assert abs(loss.item() - ref_loss) < 2e-5 * abs(ref_loss)
    # gradient through moe_route_topk_bwd: zero routing-weight gradient, so dL is the aux term
    k = 4
    idx = O.topk_select(L.numpy() + (b.numpy()[None, :] if bias else 0), k)
    slot_of, _, _ = O.permutation_maps(idx, E)
    d = 128
    x = _bf16(61, T, d)
    Wr = _bf16(62, d, E, std=0.02)
    dWr = torch.empty(d, E, dtype=torch.float32, device="cuda")
    wsb2 = M.moe_workspace_size(M.MOE_OP_ROUTE_TOPK_BWD, T=T, E=E)
    ws2 = torch.empty(wsb2, dtype=torch.uint8, device="cuda")
    ones = torch.full((T, k), 0.25, dtype=torch.float32)
    M.moe_route_topk_bwd(dev(torch.zeros(T * k)), dev(torch.from_numpy(slot_of).int()),
                         dev(torch.from_numpy(idx).int()), dev(ones), dev(ones), dev(x), dev(Wr), T,
                         d, E, k, None, None, dWr, M.MOE_DTYPE_F32, Ld, bd, p_mean, 3.0, None, None,
                         0, ws2, wsb2)
    torch.cuda.synchronize()
    dL = O.aux_balance_loss_backward(L.numpy(), b.numpy() if bias else None, scale=3.0)
    check_close("dWr_aux", f64(dWr), f64(x).T @ dL, scale_by_max=True)


@pytest.mark.parametrize("case", ["page", "zipf", "ep"])
def test_replica_plan_bit_exact(case):
    if case == "page":
        counts, P = np.array([12, 1, 2, 9, 0, 3, 4, 1]), 8
    elif case == "zipf":
        idx = I.make_topk_ids(70, 4096, 896, 16, skew=1.1).numpy()
        counts, P = O.expert_counts(idx, 896), 64
    else:
        counts, P = I.make_ep_rank_inputs()["counts"].numpy(), 14
    E = len(counts)
    pieces = torch.full(((2 * E + P), 4), -1, dtype=torch.int32, device="cuda")
    n = torch.zeros(1, dtype=torch.int32, device="cuda")
    load = torch.empty(P, dtype=torch.int32, device="cuda")
    M.moe_replica_plan(dev(torch.from_numpy(np.asarray(counts)).int()), E, P, pieces, n, load)
    torch.cuda.synchronize()
    ref_pieces, ref_load = O.replica_plan(counts, P)
    assert int(n.item()) == len(ref_pieces)
    assert pieces[: len(ref_pieces)].cpu().tolist() == [list(p) for p in ref_pieces]
    assert load.cpu().tolist() == ref_load


@pytest.mark.parametrize("skew", [0.0, 1.1, 2.0])
def test_bucket_order_and_ordered_grouped_gemm(skew):
    T, E, k, l, f = 2048, 128, 8, 256, 128
    idx = I.make_topk_ids(80, T, E, k, skew=skew)
    z = _bf16(81, T, l)
    tw = torch.rand(T, k, generator=torch.Generator().manual_seed(8)) * 0.2 + 0.01
    g = _run_permute(idx, E, l, z, tw)
    counts = g["counts"].numpy()
    order = torch.empty(E, dtype=torch.int32, device="cuda")
    sched_o = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    M.moe_expert_buckets(dev(g["counts"]), E, order, sched_o)
    torch.cuda.synchronize()
    ref_order, ref_sched = O.bucket_order(counts)
    np.testing.assert_array_equal(order.cpu().numpy(), ref_order)
    np.testing.assert_array_equal(sched_o.cpu().numpy(), ref_sched)
    R = T * k
    W13 = dev(_bf16(82, E, l, 2 * f, std=0.02))
    W2 = dev(_bf16(83, E, f, l, std=0.02))
    outs = []
    for ordered in (False, True):
        h = torch.empty(R, f, dtype=torch.bfloat16, device="cuda")
        y = torch.empty(R, l, dtype=torch.bfloat16, device="cuda")
        if ordered:
            M.moe_grouped_swiglu_ordered(dev(g["z_perm"]), W13, W2, dev(g["offsets"]), sched_o, order,
                                         dev(g["row_w"]), E, R, l, f, None, h, y)
        else:
            M.moe_grouped_swiglu(dev(g["z_perm"]), W13, W2, dev(g["offsets"]), dev(g["tile_sched"]),
                                 dev(g["row_w"]), E, R, l, f, None, h, y)
        torch.cuda.synchronize()
        outs.append((h.cpu().view(torch.int16), y.cpu().view(torch.int16)))
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])


@pytest.mark.parametrize("T", [500, 300])
def test_route_topk_bwd_fused_down_projection_dgrad(T):
    """dx = dz W_dn^T + dL Wr^T as one K-concatenated GEMM (K = l + E), on CTA
    pairs; T=300 leaves the last pair's second CTA without rows."""
    d, E, k, l = 512, 128, 4, 256
    x = _bf16(90, T, d)
    Wr = _bf16(91, d, E, std=0.02)
    W_dn = _bf16(92, d, l, std=0.02)
    dz = _bf16(93, T, l)
    L = O.router_logits(x, Wr)
    idx = O.topk_select(L, k)
    w, s = O.routing_weights(L, idx)
    slot_of, _, _ = O.permutation_maps(idx, E)
    d_row_w = torch.randn(T * k, generator=torch.Generator().manual_seed(9)).float()
    dx = torch.empty(T, d, dtype=torch.bfloat16, device="cuda")
    wsb = M.moe_workspace_size(M.MOE_OP_ROUTE_TOPK_BWD, T=T, E=E)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    M.moe_route_topk_bwd(dev(d_row_w), dev(torch.from_numpy(slot_of).int()),
                         dev(torch.from_numpy(idx).int()), dev(torch.from_numpy(w).float()),
                         dev(torch.from_numpy(s).float()), dev(x), dev(Wr), T, d, E, k, None, dx,
                         None, M.MOE_DTYPE_F32, None, None, None, 0.0, dev(dz), dev(W_dn), l, ws, wsb)
    torch.cuda.synchronize()
    dL = O.router_backward(f64(d_row_w)[slot_of], w.astype(np.float32), s.astype(np.float32), idx, E)
    check_close("dx", f64(dx), f64(dz) @ f64(W_dn).T + dL @ f64(Wr).T)
