"""Pins of the fp64 oracle against things other than itself: a hand-worked
example, brute force on tiny inputs, closed forms, invariants, textbook
library routines and central finite differences. CPU only."""
import json
import math
import os
import types

import numpy as np
import pytest
import torch

import oracle as O
from sparse_moe_layer_topk_gb300 import inputs as I

HERE = os.path.dirname(os.path.abspath(__file__))


def _ln3_matrix(a):
    a = np.asarray(a, dtype=np.float64)
    return a[..., 0] + a[..., 1] * math.log(3.0)


def _worked():
    with open(os.path.join(HERE, "golden", "worked_example.json")) as fh:
        spec = json.load(fh)
    cfg = types.SimpleNamespace(E=3, k=2, S=1, f=1)
    inp = {n: _ln3_matrix(spec[n]) for n in
           ("x", "Wr", "W_dn", "W13", "W2", "W13_sh", "W2_sh", "W_up")}
    inp["cfg"] = cfg
    inp["bias"] = None
    return inp, spec["expected"]


def test_worked_example():
    """Hand derivation: L[0] = [ln3, 0, -ln3] -> experts (0, 1), sigmoid (3/4, 1/2)
    -> w = (0.6, 0.4); L[1] = [0, -ln3, ln3] -> experts (2, 0), same weights.
    silu(ln3) = 3/4 ln3, silu(0) = 0, silu(-ln3) = -ln3/4, and the expert and
    shared outputs give y_lat = ln3 * [[1.65, -0.3], [-0.6, -0.6]]; W_up = I."""
    inp, exp = _worked()
    fwd = O.layer_forward(inp)
    assert fwd["idx"].tolist() == exp["idx"]
    np.testing.assert_allclose(fwd["w"], exp["w"], rtol=0, atol=1e-15)
    assert fwd["counts"].tolist() == exp["counts"]
    assert fwd["offsets"].tolist() == exp["offsets"]
    assert fwd["slot_of"].tolist() == exp["slot_of"]
    assert fwd["token_of"].tolist() == exp["token_of"]
    np.testing.assert_allclose(fwd["out"], np.asarray(exp["out_ln3"]) * math.log(3.0),
                               rtol=0, atol=1e-14)


# ---------------------------------------------------------------- routing

def _brute_topk(row, k):
    return sorted(range(len(row)), key=lambda e: (-row[e], e))[:k]


@pytest.mark.parametrize("ties", [False, True])
def test_topk_matches_brute_force(ties):
    L = I.make_logits(11, 64, 40, ties=ties).numpy().astype(np.float64)
    for k in (1, 4, 16, 40):
        idx = O.topk_select(L, k)
        for t in range(L.shape[0]):
            assert idx[t].tolist() == _brute_topk(L[t].tolist(), k)


def test_topk_equal_columns_lower_id_wins():
    # bf16-valued operands: every product is exact in fp64 and so is every
    # partial sum, so equal columns give bit-equal logits in any summation order
    g = torch.Generator().manual_seed(5)
    x = I.to_f64(torch.randn(32, 16, generator=g).to(torch.bfloat16))
    Wr = I.to_f64(torch.randn(16, 10, generator=g).to(torch.bfloat16))
    Wr[:, 7] = Wr[:, 3]             # experts 3 and 7 always tie
    Wr[:, 9] = Wr[:, 3]
    L = O.router_logits(x, Wr)
    idx = O.topk_select(L, 10)
    for t in range(32):
        pos = {e: p for p, e in enumerate(idx[t])}
        assert pos[3] < pos[7] < pos[9]
        assert pos[7] == pos[3] + 1 and pos[9] == pos[3] + 2


def test_topk_signed_zeros_are_one_value():
    """-0.0 == +0.0, so zeros of either sign tie and the lower id goes first."""
    L = np.array([[0.0, -0.0, 1.0, -0.0, 0.0, -2.0],
                  [-0.0, 0.0, -1.0, 0.0, -0.0, 3.0]])
    assert O.topk_select(L, 4).tolist() == [[2, 0, 1, 3], [5, 0, 1, 3]]
    rng = np.random.default_rng(8)
    M = rng.choice(np.array([-0.0, 0.0, 1.0, -1.0]), size=(50, 12))
    for k in (1, 3, 12):
        idx = O.topk_select(M, k)
        for t in range(50):
            assert idx[t].tolist() == _brute_topk(M[t].tolist(), k)


def test_topk_k_equals_E_is_full_order():
    L = I.make_logits(3, 8, 12).numpy().astype(np.float64)
    idx = O.topk_select(L, 12)
    for t in range(8):
        assert sorted(idx[t].tolist()) == list(range(12))
        assert np.all(np.diff(L[t, idx[t]]) <= 0)


def test_weights_invariants():
    L = I.make_logits(4, 128, 64).numpy().astype(np.float64)
    idx = O.topk_select(L, 8)
    w, s = O.routing_weights(L, idx)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
    sig = 1.0 / (1.0 + np.exp(-np.take_along_axis(L, idx, 1)))
    np.testing.assert_allclose(s, sig, rtol=1e-15)
    ratio = w / sig
    np.testing.assert_allclose(ratio, ratio[:, :1].repeat(8, 1), rtol=1e-13)
    # the first selected id has the largest weight
    assert np.all(w[:, 0] >= w.max(1) - 1e-15)


def test_renorm_jacobian_closed_form():
    """d w_i / d s_j = (delta_ij - w_i) / sum(s): the vector-Jacobian product
    written in the oracle's backward equals the explicit Jacobian."""
    rng = np.random.default_rng(9)
    s = rng.uniform(0.05, 0.95, 6)
    dw = rng.standard_normal(6)
    S = s.sum()
    w = s / S
    J = (np.eye(6) - w[:, None]) / S            # J[i, j] = dw_i / ds_j
    ds_explicit = J.T @ dw
    ds_oracle = (dw - (w * dw).sum()) / S      # form used by layer_backward
    np.testing.assert_allclose(ds_oracle, ds_explicit, rtol=1e-13, atol=1e-15)
    # and J against finite differences of w(s)
    h = 1e-7
    for j in range(6):
        sp, sm = s.copy(), s.copy()
        sp[j] += h
        sm[j] -= h
        np.testing.assert_allclose((sp / sp.sum() - sm / sm.sum()) / (2 * h), J[:, j],
                                   rtol=1e-6, atol=1e-9)


# ---------------------------------------------------------------- permute

def _brute_maps(idx, E):
    T, k = idx.shape
    rows = {e: [] for e in range(E)}
    for t in range(T):
        for j in range(k):
            rows[int(idx[t, j])].append((t, j))
    slot_of = np.full((T, k), -1)
    token_of = []
    for e in range(E):
        for (t, j) in rows[e]:
            slot_of[t, j] = len(token_of)
            token_of.append(t)
    return slot_of, np.asarray(token_of)


@pytest.mark.parametrize("skew", [0.0, 1.1])
def test_counts_offsets_maps(skew):
    T, E, k = 300, 37, 5
    idx = I.make_topk_ids(21, T, E, k, skew=skew).numpy()
    counts = O.expert_counts(idx, E)
    np.testing.assert_array_equal(counts, np.bincount(idx.reshape(-1), minlength=E))
    assert counts.sum() == T * k
    offsets = O.expert_offsets(counts)
    assert offsets[0] == 0 and offsets[-1] == T * k and np.all(np.diff(offsets) >= 0)
    slot_of, token_of, off2 = O.permutation_maps(idx, E)
    np.testing.assert_array_equal(off2, offsets)
    bs, bt = _brute_maps(idx, E)
    np.testing.assert_array_equal(slot_of, bs)
    np.testing.assert_array_equal(token_of, bt)
    # bijection and inverse relation
    assert sorted(slot_of.reshape(-1).tolist()) == list(range(T * k))
    for t in range(T):
        for j in range(k):
            assert token_of[slot_of[t, j]] == t
            e = idx[t, j]
            assert offsets[e] <= slot_of[t, j] < offsets[e + 1]
    for e in range(E):
        seg = token_of[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)
    if skew:
        assert (counts == 0).any() or counts.max() > 3 * counts.mean()


def test_tile_schedule_brute():
    counts = np.array([0, 1, 127, 128, 129, 300, 0, 256])
    sched = O.m_tiles_schedule(counts, 128)
    acc, ref = 0, [0]
    for c in counts:
        n = 0
        while n * 128 < c:
            n += 1
        acc += n
        ref.append(acc)
    assert sched.tolist() == ref


def test_permute_unpermute_identity():
    """Identity experts with unit weights: combine(permute(z)) = k z exactly."""
    T, E, k, l = 50, 9, 3, 16
    idx = I.make_topk_ids(2, T, E, k).numpy()
    z = I.to_f64(torch.randn(T, l, generator=torch.Generator().manual_seed(0))
                 .to(torch.bfloat16))
    slot_of, token_of, _ = O.permutation_maps(idx, E)
    zp = O.permute_rows(z, token_of)
    np.testing.assert_array_equal(O.combine(zp, slot_of), k * z)
    # with k = 1 the combine is an exact inverse permutation
    slot1, tok1, _ = O.permutation_maps(idx[:, :1], E)
    np.testing.assert_array_equal(O.combine(O.permute_rows(z, tok1), slot1), z)


# ---------------------------------------------------------------- experts

def test_shared_expert_is_textbook_swiglu():
    g = torch.Generator().manual_seed(1)
    z = torch.randn(40, 32, generator=g, dtype=torch.float64)
    W13 = torch.randn(32, 2 * 24, generator=g, dtype=torch.float64) * 0.1
    W2 = torch.randn(24, 32, generator=g, dtype=torch.float64) * 0.1
    ref = (torch.nn.functional.silu(z @ W13[:, :24]) * (z @ W13[:, 24:])) @ W2
    np.testing.assert_allclose(O.swiglu_expert(z, W13, W2), ref.numpy(), rtol=1e-13, atol=1e-15)


def test_single_group_equals_dense():
    g = torch.Generator().manual_seed(2)
    z = torch.randn(20, 16, generator=g, dtype=torch.float64)
    W13 = torch.randn(1, 16, 12, generator=g, dtype=torch.float64)
    W2 = torch.randn(1, 6, 16, generator=g, dtype=torch.float64)
    y = O.grouped_swiglu(z, W13, W2, np.array([0, 20]))
    ref = (torch.nn.functional.silu(z @ W13[0, :, :6]) * (z @ W13[0, :, 6:])) @ W2[0]
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-13, atol=1e-14)


def test_sparse_equals_dense_cfg0():
    """Evaluate every expert on every token and mask by the top-k choice."""
    inp = I.make_layer_inputs(0)
    cfg = inp["cfg"]
    fwd = O.layer_forward(inp)
    x = I.to_f64(inp["x"])
    z = x @ I.to_f64(inp["W_dn"])
    L = x @ I.to_f64(inp["Wr"])
    dense = np.zeros_like(z)
    for e in range(cfg.E):
        W13 = I.to_f64(inp["W13"][e])
        W2 = I.to_f64(inp["W2"][e])
        gate = z @ W13[:, :cfg.f]
        up = z @ W13[:, cfg.f:]
        o = ((gate / (1 + np.exp(-gate))) * up) @ W2
        for t in range(cfg.T):
            row = L[t]
            rank = int(np.sum(row > row[e]) + np.sum((row == row[e]) & (np.arange(cfg.E) < e)))
            if rank < cfg.k:
                top = sorted(range(cfg.E), key=lambda q: (-row[q], q))[:cfg.k]
                sg = 1 / (1 + np.exp(-row[top]))
                dense[t] += (1 / (1 + np.exp(-row[e])) / sg.sum()) * o[t]
    for sidx in range(cfg.S):
        W13 = I.to_f64(inp["W13_sh"][sidx])
        W2 = I.to_f64(inp["W2_sh"][sidx])
        gate = z @ W13[:, :cfg.f]
        dense += ((gate / (1 + np.exp(-gate))) * (z @ W13[:, cfg.f:])) @ W2
    np.testing.assert_allclose(fwd["y_lat"], dense, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(fwd["out"], dense @ I.to_f64(inp["W_up"]), rtol=1e-11, atol=1e-13)


def test_ep_rank_forward_brute():
    rng = np.random.default_rng(3)
    E, R, l, f = 4, 40, 8, 6
    counts = np.array([10, 0, 25, 5])
    z = rng.standard_normal((R, l))
    W13 = rng.standard_normal((E, l, 2 * f)) * 0.3
    W2 = rng.standard_normal((E, f, l)) * 0.3
    w = rng.uniform(0.01, 0.2, R)
    perm = rng.permutation(R)
    out = O.ep_rank_forward(z, counts, W13, W2, w, perm)
    starts = np.concatenate([[0], np.cumsum(counts)])
    for r in range(R):
        e = int(np.searchsorted(starts, r, side="right") - 1)
        g = z[r] @ W13[e][:, :f]
        u = z[r] @ W13[e][:, f:]
        o = ((g / (1 + np.exp(-g))) * u) @ W2[e]
        np.testing.assert_allclose(out[perm[r]], w[r] * o, rtol=1e-12, atol=1e-14)


# ---------------------------------------------------------------- backward

def _tiny_inputs(seed=7):
    cfg = types.SimpleNamespace(T=6, d=8, l=6, E=5, k=2, S=1, f=4)
    rng = np.random.default_rng(seed)
    inp = {
        "cfg": cfg,
        "x": rng.standard_normal((cfg.T, cfg.d)),
        "Wr": rng.standard_normal((cfg.d, cfg.E)) * 0.5,
        "bias": rng.standard_normal(cfg.E) * 0.1,
        "W_dn": rng.standard_normal((cfg.d, cfg.l)) * 0.4,
        "W13": rng.standard_normal((cfg.E, cfg.l, 2 * cfg.f)) * 0.4,
        "W2": rng.standard_normal((cfg.E, cfg.f, cfg.l)) * 0.4,
        "W13_sh": rng.standard_normal((cfg.S, cfg.l, 2 * cfg.f)) * 0.4,
        "W2_sh": rng.standard_normal((cfg.S, cfg.f, cfg.l)) * 0.4,
        "W_up": rng.standard_normal((cfg.l, cfg.d)) * 0.4,
        "g": rng.standard_normal((cfg.T, cfg.d)),
    }
    return inp


def test_backward_finite_differences():
    inp = _tiny_inputs()
    fwd = O.layer_forward(inp)
    Ls = np.sort(fwd["L"], axis=1)[:, ::-1]
    k = inp["cfg"].k
    assert np.min(Ls[:, k - 1] - Ls[:, k]) > 1e-3   # no near-ties: routing is fixed
    grads = O.layer_backward(inp, fwd)
    names = {"x": "dx", "Wr": "dWr", "W_dn": "dW_dn", "W13": "dW13", "W2": "dW2",
             "W13_sh": "dW13_sh", "W2_sh": "dW2_sh", "W_up": "dW_up"}
    rng = np.random.default_rng(0)
    h = 1e-6

    def loss(p):
        return float(np.sum(O.layer_forward(p)["out"] * inp["g"]))

    for pname, gname in names.items():
        base = inp[pname]
        flat_idx = rng.choice(base.size, size=min(12, base.size), replace=False)
        for fi in flat_idx:
            pp = dict(inp)
            pm = dict(inp)
            a, b = base.copy(), base.copy()
            a.flat[fi] += h
            b.flat[fi] -= h
            pp[pname], pm[pname] = a, b
            fd = (loss(pp) - loss(pm)) / (2 * h)
            an = grads[gname].flat[fi]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (pname, fi, fd, an)
    # empty experts get exactly zero gradient
    for e in range(inp["cfg"].E):
        if fwd["counts"][e] == 0:
            assert not grads["dW13"][e].any() and not grads["dW2"][e].any()


def test_routing_weight_gradient_finite_differences():
    """d loss / d w[t,j] against a perturbation of the combine weight itself."""
    inp = _tiny_inputs(8)
    fwd = O.layer_forward(inp)
    grads = O.layer_backward(inp, fwd)
    W_up = inp["W_up"]
    g = inp["g"]
    for (t, j) in [(0, 0), (3, 1), (5, 0)]:
        slot = fwd["slot_of"][t, j]
        o = fwd["y_perm"][slot] / fwd["row_w"][slot]
        # out[t] is linear in w[t,j] with slope o W_up
        np.testing.assert_allclose(grads["d_w"][t, j], np.dot(o @ W_up, g[t]), rtol=1e-12)


def test_zipf_workload_statistics():
    """The skewed workload has the stated shape: top 5% of experts hold >30% of
    the assignments and roughly 200 experts get 0-2 tokens."""
    cfg = I.CONFIGS[2]
    inp = I.make_layer_inputs(cfg)
    L = O.router_logits(inp["x"], inp["Wr"], inp["bias"])
    counts = O.expert_counts(O.topk_select(L, cfg.k), cfg.E)
    top = np.sort(counts)[::-1]
    assert top[:45].sum() / counts.sum() > 0.30
    assert 150 <= int((counts <= 2).sum()) <= 260


# ---------------------------------------------------------------- auxiliary balance loss

def test_aux_loss_balanced_closed_form():
    """Equal logits: every token spreads evenly, pbar = 1/E, loss = -log E and
    the gradient vanishes (the balanced point is the loss's minimum)."""
    L = np.full((7, 12), 0.3)
    pbar, loss = O.aux_balance_loss(L)
    np.testing.assert_allclose(pbar, 1.0 / 12, rtol=1e-15)
    assert abs(loss + math.log(12.0)) < 1e-14
    np.testing.assert_allclose(O.aux_balance_loss_backward(L), 0.0, atol=1e-17)


def test_aux_loss_two_experts_by_hand():
    """Two tokens, two experts, logits (ln3, 0) and (0, 0): s = (3/4, 1/2) and
    (1/2, 1/2), P = (3/5, 2/5) and (1/2, 1/2), pbar = (11/20, 9/20)."""
    L = np.array([[math.log(3.0), 0.0], [0.0, 0.0]])
    pbar, loss = O.aux_balance_loss(L)
    np.testing.assert_allclose(pbar, [0.55, 0.45], rtol=1e-14)
    assert abs(loss - (0.55 * math.log(0.55) + 0.45 * math.log(0.45))) < 1e-14
    # skewed experts: raising expert 0's logit on any token makes it worse
    g = O.aux_balance_loss_backward(L)
    assert g[0, 0] > 0 and g[1, 0] > 0 and g[0, 1] < 0 and g[1, 1] < 0


def test_aux_loss_gradient_finite_differences():
    rng = np.random.default_rng(12)
    L = rng.standard_normal((9, 7)) * 1.3
    b = rng.standard_normal(7) * 0.2
    g = O.aux_balance_loss_backward(L, b, scale=0.7)
    h = 1e-6
    for (t, e) in [(0, 0), (3, 5), (8, 2), (4, 6)]:
        Lp, Lm = L.copy(), L.copy()
        Lp[t, e] += h
        Lm[t, e] -= h
        fd = 0.7 * (O.aux_balance_loss(Lp, b)[1] - O.aux_balance_loss(Lm, b)[1]) / (2 * h)
        assert abs(fd - g[t, e]) < 1e-8 * max(1.0, abs(fd)), (t, e, fd, g[t, e])


# ---------------------------------------------------------------- replica planner

def _check_plan(counts, P, pieces, load):
    E = len(counts)
    C = -(-sum(counts) // P)
    assert sum(load) == sum(counts) and max(load) <= C
    # every expert's rows are covered exactly once, in contiguous pieces
    for e in range(E):
        mine = sorted((p for p in pieces if p[0] == e), key=lambda p: p[2])
        pos = 0
        for (_, _, first, n) in mine:
            assert first == pos and n > 0
            pos += n
        assert pos == counts[e]
    per = E // P
    # an expert's first piece stays on its owning rank whenever that rank had room
    for (e, r, first, n) in pieces:
        if first == 0 and n > 0 and r != e // per:
            owner = e // per
            assert load[owner] == C
    for r in range(P):
        assert load[r] == sum(p[3] for p in pieces if p[1] == r)


def test_replica_plan_page_illustration():
    """32 tasks spread unevenly over 8 ranks (one expert per rank) end as 4 per rank."""
    counts = [12, 1, 2, 9, 0, 3, 4, 1]
    pieces, load = O.replica_plan(counts, 8)
    assert load == [4] * 8
    _check_plan(counts, 8, pieces, load)
    # the hot experts 0 and 3 get replicas, expert identity is kept
    assert {p[0] for p in pieces if p[1] != p[0]} == {0, 3}


@pytest.mark.parametrize("seed", range(6))
def test_replica_plan_invariants(seed):
    rng = np.random.default_rng(seed)
    P = int(rng.choice([1, 2, 4, 8]))
    E = P * int(rng.integers(1, 6))
    counts = rng.multinomial(int(rng.integers(0, 400)), rng.dirichlet(np.full(E, 0.3))).tolist()
    pieces, load = O.replica_plan(counts, P)
    _check_plan(counts, P, pieces, load)


# ---------------------------------------------------------------- bucket order

def test_bucket_classes_by_hand():
    assert [O.expert_bucket_class(c) for c in (0, 1, 128, 129, 256, 257, 512, 1024, 1025)] == \
        [0, 1, 1, 2, 2, 2, 3, 4, 4]


@pytest.mark.parametrize("seed", range(4))
def test_bucket_order_invariants(seed):
    rng = np.random.default_rng(seed)
    E = int(rng.integers(1, 200))
    counts = rng.multinomial(int(rng.integers(0, 30000)), rng.dirichlet(np.full(E, 0.3)))
    order, sched = O.bucket_order(counts)
    assert sorted(order.tolist()) == list(range(E))
    cls = [O.expert_bucket_class(counts[e]) for e in order]
    assert all(a >= b for a, b in zip(cls, cls[1:]))
    for c in set(cls):
        ids = [e for e in order if O.expert_bucket_class(counts[e]) == c]
        assert ids == sorted(ids)
    tiles = [(int(counts[e]) + 127) // 128 for e in order]
    assert sched.tolist() == [0] + np.cumsum(tiles).tolist()
    assert sched[-1] == O.m_tiles_schedule(counts)[-1]


def test_empty_batch_closed_form():
    """No tokens: empty outputs and input gradient, zero counts and offsets, and
    every weight gradient exactly zero (each is a sum over no tokens)."""
    inp = I.make_layer_inputs(0, T=0)
    cfg = inp["cfg"]
    fwd = O.layer_forward(inp)
    bwd = O.layer_backward(inp, fwd)
    assert fwd["out"].shape == (0, cfg.d) and bwd["dx"].shape == (0, cfg.d)
    assert not np.any(fwd["counts"]) and not np.any(fwd["offsets"])
    for name in ("dWr", "dW_dn", "dW13", "dW2", "dW13_sh", "dW2_sh", "dW_up"):
        assert bwd[name].shape and not np.any(bwd[name]), name
