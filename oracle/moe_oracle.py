"""fp64 CPU oracle of the LatentMoE layer: routing, permute, grouped SwiGLU
experts, weighted combine, latent projections, and their backward.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this module:
only the tests, the smoke check of ``__graft_entry__`` and the CPU-baseline leg
of ``bench.py`` use it. It shares no code with the CUDA library.

All arithmetic is float64 with no intermediate rounding; inputs are the bf16
(or fp32) values widened exactly. numpy's matmul and sort serve as library
steps; there is no blocking, fusion or reordering beyond the definitions.

Sources (the pages give the structure, not the formulas):
  [MOE-A] "昇腾实现Kimi K3.1 Pro模型LoRA训练适配" page, section
          "Kimi K3.1 Pro——面向长程智能体的开源旗舰大模型": 896 routed experts,
          16 activated per token.
  [MOE-B] "TorchTitan Ascend开源" page, section "Kimi K3.1 Pro 模型结构",
          LatentMoE paragraph: 896 routed + 2 shared experts, 16 active, expert
          compute in a low-dimensional latent space.
  [MOE-C] "昇腾实现Kimi K3.1 Pro模型LoRA训练适配" page, section
          "MoE(Mixture of Experts):算子融合与通信协同": dynamic routing, token
          dispatch, Permute / Unpermute / Grouped GEMM as the core operators.
  [MOE-D] "TorchTitan Ascend开源" page, section "在线负载规划": per-expert load
          counted from the current routing result.
  [PLAN]  "TorchTitan Ascend开源" page, sections "在线负载规划" and
          "MoonEP动态负载均衡与专家并行优化": online replica planning.
  [BUCKET] "大模型落地昇腾:从适配挑战到高效训练实践" page, section "二、算力侧":
          multi-bucket batching of experts with similar token counts.
  [AUX]   "大模型落地昇腾:从适配挑战到高效训练实践" page, section "三、通信侧":
          an auxiliary load-balance loss that constrains the entropy of the
          routing distribution.
  [SWAP]  "昇腾实现Kimi K3.1 Pro模型LoRA训练适配" page, section "Swap Core:算子级
          精准缓存与异步 Offload 协同,训练性能提升 15%": the outputs of selected
          MatMul/GMM operators are cached for the backward, optionally compressed
          by FP8 activation quantization and dequantization.
Readings where the pages are silent (router = sigmoid(x@Wr) with renormalised
top-k weights, lower expert id wins ties, tokens of an expert in ascending
token order, shared experts in latent space with weight 1, routing weight
applied to the expert output) are the plainest ones the workload statements
support; each function below states the one it uses.

Parity pins: every function here is pinned by tests/test_oracle_*.py against
brute force, closed forms, invariants or finite differences; none is
"parity unpinned".
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "router_logits", "topk_select", "sigmoid", "routing_weights", "expert_counts",
    "expert_offsets", "permutation_maps", "permute_rows", "swiglu_expert",
    "grouped_swiglu", "combine", "layer_forward", "layer_backward",
    "ep_rank_forward", "m_tiles_schedule", "router_backward", "swiglu_expert_backward",
    "aux_balance_loss", "aux_balance_loss_backward", "replica_plan", "bucket_order",
    "expert_bucket_class", "e4m3_round", "fp8_block_scale", "fp8_block_quantize",
    "fp8_block_dequantize", "FP8_BLOCK",
]


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        import torch  # only to widen torch inputs exactly
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# Routing  [MOE-A], [MOE-C]
# --------------------------------------------------------------------------

def router_logits(x, Wr, bias=None) -> np.ndarray:
    """L[t,e] = sum_i x[t,i] Wr[i,e] (+ b[e]).  The router reads the model-width
    activations x (not the latent z); the optional per-expert bias is part of
    the logit and so moves both the selection and the weights."""
    L = _f64(x) @ _f64(Wr)
    if bias is not None:
        L = L + _f64(bias)[None, :]
    return L


def topk_select(L, k: int) -> np.ndarray:
    """Ids of the k largest logits per token, ordered by (logit desc, id asc).

    Selecting on the logit equals selecting on sigmoid(logit) (strictly
    increasing) without the saturation ties of the sigmoid. A stable sort of
    the negated logits keeps equal values in ascending id order, so the lower
    id wins a tie. Returns int64 [T,k]."""
    L = _f64(L)
    order = np.argsort(-L, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def sigmoid(v) -> np.ndarray:
    v = _f64(v)
    return 1.0 / (1.0 + np.exp(-v))


def routing_weights(L, idx):
    """s_j = sigmoid(L[t, idx_j]); w_j = s_j / sum_j' s_j' (no scale, no eps:
    sigmoid > 0 so the sum is positive). Returns (w, s), both [T,k]."""
    s = sigmoid(np.take_along_axis(_f64(L), np.asarray(idx), axis=1))
    return s / s.sum(axis=1, keepdims=True), s


# --------------------------------------------------------------------------
# Permute bookkeeping  [MOE-C], [MOE-D]
# --------------------------------------------------------------------------

def expert_counts(idx, E: int) -> np.ndarray:
    """counts[e] = number of (token, slot) pairs routed to expert e."""
    counts = np.zeros(E, dtype=np.int64)
    np.add.at(counts, np.asarray(idx).reshape(-1), 1)
    return counts


def expert_offsets(counts) -> np.ndarray:
    """Exclusive prefix sum, E+1 entries; offsets[E] = T*k."""
    c = np.asarray(counts, dtype=np.int64)
    out = np.zeros(c.size + 1, dtype=np.int64)
    out[1:] = np.cumsum(c)
    return out


def permutation_maps(idx, E: int):
    """Stable counting sort of the (token, slot) pairs by expert.

    Rows of expert e occupy [offsets[e], offsets[e+1]) of the permuted buffer,
    tokens in ascending order (a token routes to an expert at most once, so
    (e, t) is a unique key). Returns (slot_of [T,k], token_of [T*k], offsets)."""
    idx = np.asarray(idx)
    T, k = idx.shape
    offsets = expert_offsets(expert_counts(idx, E))
    flat_e = idx.reshape(-1)                      # pair p = t*k + j, ascending t
    order = np.argsort(flat_e, kind="stable")     # by expert, then by p
    slot_of = np.empty(T * k, dtype=np.int64)
    slot_of[order] = np.arange(T * k)
    token_of = order // k
    return slot_of.reshape(T, k), token_of.astype(np.int64), offsets


def m_tiles_schedule(counts, tile_m: int = 128) -> np.ndarray:
    """Exclusive prefix sum of ceil(counts[e] / tile_m), E+1 entries: the row-tile
    index range of each expert in a grouped GEMM with tile_m-row tiles."""
    c = np.asarray(counts, dtype=np.int64)
    tiles = (c + tile_m - 1) // tile_m
    out = np.zeros(c.size + 1, dtype=np.int64)
    out[1:] = np.cumsum(tiles)
    return out


def permute_rows(z, token_of) -> np.ndarray:
    """z_perm[r] = z[token_of[r]]."""
    return _f64(z)[np.asarray(token_of)]


# --------------------------------------------------------------------------
# Experts  [MOE-B], [MOE-C]
# --------------------------------------------------------------------------

def _silu(g):
    return g / (1.0 + np.exp(-g))


def swiglu_expert(zrows, W13e, W2e, return_parts: bool = False):
    """o = (silu(z W_gate) * (z W_up)) W2 with W13e = [W_gate | W_up] ([l, 2f])."""
    zrows, W13e, W2e = _f64(zrows), _f64(W13e), _f64(W2e)
    f = W2e.shape[0]
    gu = zrows @ W13e
    g, u = gu[:, :f], gu[:, f:]
    h = _silu(g) * u
    o = h @ W2e
    if return_parts:
        return o, g, u, h
    return o


def grouped_swiglu(z_perm, W13, W2, offsets, row_w=None):
    """y_perm[r] = row_w[r] * swiglu_expert(z_perm[r], W13[e], W2[e]) for the
    expert e whose segment [offsets[e], offsets[e+1]) holds r. Empty segments
    contribute nothing. row_w=None means weight 1."""
    z_perm = _f64(z_perm)
    y = np.zeros((z_perm.shape[0], _f64(W2[0]).shape[1]))
    E = len(offsets) - 1
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            y[a:b] = swiglu_expert(z_perm[a:b], W13[e], W2[e])
    if row_w is not None:
        y *= _f64(row_w)[:, None]
    return y


def combine(y_perm, slot_of, y_shared=None):
    """y[t] = sum_j y_perm[slot_of[t,j]] (+ y_shared[t])."""
    y_perm = _f64(y_perm)
    y = y_perm[np.asarray(slot_of)].sum(axis=1)
    if y_shared is not None:
        y = y + _f64(y_shared)
    return y


# --------------------------------------------------------------------------
# FP8 cache of the GMM outputs  [SWAP]
# --------------------------------------------------------------------------
# Reading (the page names FP8 activation quantization, not its format): OCP
# FP8 E4M3 (4 exponent bits with bias 7, 3 mantissa bits, subnormals, largest
# finite value 448, no infinities), round to nearest with ties to the even
# mantissa, saturating at +-448; one power-of-two scale per row and block of
# FP8_BLOCK = 64 consecutive columns of g (and of u), the smallest that brings
# the block's largest magnitude to at most 448 (power of two: scaling is exact,
# so the rounding decisions depend on the values alone).

FP8_BLOCK = 64
E4M3_MAX = 448.0


def e4m3_round(y) -> np.ndarray:
    """The E4M3 value nearest to y (ties to even mantissa), clamped to +-448."""
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    _, ex = np.frexp(a)                       # a = m 2^ex, 0.5 <= m < 1
    E = np.maximum(ex - 1, -6)                # binade exponent; subnormals share 2^-6's
    spacing = np.ldexp(1.0, E - 3)            # 3 mantissa bits
    q = np.minimum(np.round(a / spacing) * spacing, E4M3_MAX)   # np.round: half to even
    return np.where(y < 0, -q, q)


def fp8_block_scale(amax: float) -> float:
    """Smallest power of two s with amax <= 448 s (1 for amax < 2^-100)."""
    amax = float(amax)
    if not amax >= 2.0 ** -100:
        return 1.0
    m, ex = np.frexp(amax)                    # amax = m 2^ex; 448 = 0.875 2^9
    return float(np.ldexp(1.0, int(ex) - 9 + (1 if m > 0.875 else 0)))


def fp8_block_quantize(x, block: int = FP8_BLOCK):
    """x [rows, cols] (cols a multiple of block) -> (q, scales): q the E4M3
    values of x / scale, scales [rows, cols / block]."""
    x = _f64(x)
    rows, cols = x.shape
    nb = cols // block
    scales = np.ones((rows, nb))
    q = np.zeros_like(x)
    for r in range(rows):
        for b in range(nb):
            blk = x[r, b * block:(b + 1) * block]
            sc = fp8_block_scale(np.max(np.abs(blk)))
            scales[r, b] = sc
            q[r, b * block:(b + 1) * block] = e4m3_round(blk / sc)
    return q, scales


def fp8_block_dequantize(q, scales, block: int = FP8_BLOCK) -> np.ndarray:
    """q * scale, the scale repeated over its block."""
    return _f64(q) * np.repeat(_f64(scales), block, axis=1)


# --------------------------------------------------------------------------
# Whole layer
# --------------------------------------------------------------------------

def layer_forward(inp: dict, k: int | None = None, idx=None) -> dict:
    """Forward of the latent MoE layer on the bf16 inputs of `inp`.

    out = (y_sh + sum_j w_j o_j) W_up with z = x W_dn, o_j = expert_j(z),
    y_sh = sum_s SwiGLU_s(z) (shared experts in latent space, weight 1),
    routing on x as above. Returns every intermediate (fp64).

    Staged parity: `idx` [T,k], when given, replaces the selection step (a
    selection decided on logits of another precision, where a token whose
    k-th and (k+1)-th logits are closer than that precision's rounding may
    pick another last expert); the weights still follow from the fp64 logits
    of the selected experts, and every later step is unchanged."""
    cfg = inp["cfg"]
    k = cfg.k if k is None else k
    x = _f64(inp["x"])
    E = cfg.E
    L = router_logits(x, inp["Wr"], inp.get("bias"))
    idx = topk_select(L, k) if idx is None else np.asarray(idx, dtype=np.int64)
    w, s = routing_weights(L, idx)
    z = x @ _f64(inp["W_dn"])
    slot_of, token_of, offsets = permutation_maps(idx, E)
    z_perm = permute_rows(z, token_of)
    row_w = w.reshape(-1)[np.argsort(slot_of.reshape(-1))]    # row_w[slot_of[t,j]] = w[t,j]
    y_perm = grouped_swiglu(z_perm, inp["W13"], inp["W2"], offsets, row_w)
    y_sh = np.zeros_like(z)
    for sidx in range(inp["W13_sh"].shape[0]):
        y_sh += swiglu_expert(z, inp["W13_sh"][sidx], inp["W2_sh"][sidx])
    y_lat = combine(y_perm, slot_of, y_sh)
    out = y_lat @ _f64(inp["W_up"])
    return dict(L=L, idx=idx, w=w, s=s, z=z, slot_of=slot_of, token_of=token_of,
                offsets=offsets, counts=np.diff(offsets), z_perm=z_perm, row_w=row_w,
                y_perm=y_perm, y_sh=y_sh, y_lat=y_lat, out=out)


def swiglu_expert_backward(zrows, W13e, W2e, d_o, gu_cache=None):
    """Chain rule through o = (silu(g) * u) W2, [g|u] = z W13.
    Returns dz, dW13e, dW2e.

    gu_cache = (g~, u~): the backward's g and u come from a cache of the
    forward's values (the FP8 cache of [SWAP], see fp8_block_quantize) in the
    SwiGLU derivative; h, the down projection's input, is the forward's own
    (reading: the cache holds the GMM output [g|u]; h is kept as it is)."""
    zrows, W13e, W2e = _f64(zrows), _f64(W13e), _f64(W2e)
    f = W2e.shape[0]
    gu = zrows @ W13e
    g, u = gu[:, :f], gu[:, f:]
    h = _silu(g) * u
    dW2e = h.T @ d_o
    dh = d_o @ W2e.T
    if gu_cache is not None:
        g, u = _f64(gu_cache[0]), _f64(gu_cache[1])
    sg = 1.0 / (1.0 + np.exp(-g))
    silu = g * sg
    dg = dh * u * sg * (1.0 + g * (1.0 - sg))     # d silu / dg = s (1 + g (1 - s))
    du = dh * silu
    dgu = np.concatenate([dg, du], axis=1)
    return dgu @ W13e.T, zrows.T @ dgu, dW2e


def layer_backward(inp: dict, fwd: dict, dout=None, fp8_cache: bool = False) -> dict:
    """Gradients of loss = sum(out * dout) (dout defaults to inp["g"]) with
    respect to x and every weight, routing held at its forward choice (the
    selection is piecewise constant; the router bias is a constant).
    fp8_cache: the routed experts' backward takes g and u from their FP8 block
    cache (fp8_block_quantize of each expert's g and u, [SWAP]); the shared
    experts keep theirs exact.

    Returns dx, dWr, dW_dn, dW13, dW2, dW13_sh, dW2_sh, dW_up and the routing
    weight gradient d_w [T,k] (fp64)."""
    cfg = inp["cfg"]
    E = cfg.E
    g = _f64(inp["g"] if dout is None else dout)
    x = _f64(inp["x"])
    W_up, W_dn, Wr = _f64(inp["W_up"]), _f64(inp["W_dn"]), _f64(inp["Wr"])
    # out = y_lat W_up
    dy_lat = g @ W_up.T
    dW_up = fwd["y_lat"].T @ g
    z, z_perm, offsets = fwd["z"], fwd["z_perm"], fwd["offsets"]
    token_of, slot_of, row_w = fwd["token_of"], fwd["slot_of"], fwd["row_w"]
    # y_lat[t] = y_sh[t] + sum_j y_perm[slot_of[t,j]];  y_perm[r] = w_r o_r
    dy_perm = dy_lat[token_of]
    R = z_perm.shape[0]
    dz_perm = np.zeros_like(z_perm)
    d_row_w = np.zeros(R)
    dW13 = np.zeros((E,) + tuple(inp["W13"].shape[1:]))
    dW2 = np.zeros((E,) + tuple(inp["W2"].shape[1:]))
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b == a:
            continue                                   # empty expert: zero gradient
        o, ge, ue, _ = swiglu_expert(z_perm[a:b], inp["W13"][e], inp["W2"][e], True)
        d_row_w[a:b] = np.einsum("rc,rc->r", dy_perm[a:b], o)
        d_o = dy_perm[a:b] * row_w[a:b, None]
        cache = None
        if fp8_cache:
            cache = tuple(fp8_block_dequantize(*fp8_block_quantize(v)) for v in (ge, ue))
        dz_perm[a:b], dW13[e], dW2[e] = swiglu_expert_backward(z_perm[a:b], inp["W13"][e],
                                                         inp["W2"][e], d_o, cache)
    S = inp["W13_sh"].shape[0]
    dz = np.zeros_like(z)
    dW13_sh = np.zeros((S,) + tuple(inp["W13_sh"].shape[1:]))
    dW2_sh = np.zeros((S,) + tuple(inp["W2_sh"].shape[1:]))
    for sidx in range(S):
        dzs, dW13_sh[sidx], dW2_sh[sidx] = swiglu_expert_backward(z, inp["W13_sh"][sidx],
                                                             inp["W2_sh"][sidx], dy_lat)
        dz += dzs
    dz += dz_perm[slot_of].sum(axis=1)
    d_w = d_row_w[slot_of]                              # [T,k]
    dL = router_backward(d_w, fwd["w"], fwd["s"], fwd["idx"], E)
    dWr = x.T @ dL
    dW_dn = x.T @ dz
    dx = dz @ W_dn.T + dL @ Wr.T
    return dict(dy_lat=dy_lat, dy_perm=dy_perm, d_row_w=d_row_w, d_w=d_w, dL=dL,
                dz_perm=dz_perm, dz=dz, dx=dx, dWr=dWr, dW_dn=dW_dn, dW13=dW13,
                dW2=dW2, dW13_sh=dW13_sh, dW2_sh=dW2_sh, dW_up=dW_up)


def router_backward(d_w, w, s, idx, E: int) -> np.ndarray:
    """Gradient of the router logits from the routing-weight gradient d_w [T,k].

    w_j = s_j / sum_i s_i gives dL/ds_j = (d_w_j - sum_i w_i d_w_i) / sum_i s_i;
    s_j = sigmoid(L_j) gives ds_j/dL_j = s_j (1 - s_j). Unselected experts get
    zero (the top-k choice is piecewise constant). Returns dense dL [T,E]."""
    d_w, w, s = _f64(d_w), _f64(w), _f64(s)
    ssum = s.sum(axis=1, keepdims=True)
    ds = (d_w - (w * d_w).sum(axis=1, keepdims=True)) / ssum
    dL = np.zeros((d_w.shape[0], E))
    np.put_along_axis(dL, np.asarray(idx), ds * s * (1.0 - s), axis=1)
    return dL


# --------------------------------------------------------------------------
# Auxiliary load balance  [AUX]: "大模型落地昇腾" page, section "三、通信侧",
# routing-aware token dispatch: an auxiliary loss at the routing stage that
# constrains the entropy of the routing distribution.
# --------------------------------------------------------------------------

def aux_balance_loss(L, bias=None):
    """Negative entropy of the batch's mean routing distribution.

    P(e|t) = s[t,e] / sum_e' s[t,e'] with s = sigmoid(L + b) over all E experts
    (the router's scores normalised per token); pbar_e = mean_t P(e|t);
    loss = sum_e pbar_e log pbar_e = -H(pbar), smallest (-log E) when the
    batch's routing mass is spread evenly. Returns (pbar [E], loss)."""
    L = _f64(L)
    if bias is not None:
        L = L + _f64(bias)[None, :]
    s = sigmoid(L)
    P = s / s.sum(axis=1, keepdims=True)
    pbar = P.mean(axis=0)
    return pbar, float(np.sum(pbar * np.log(pbar)))


def aux_balance_loss_backward(L, bias=None, scale: float = 1.0):
    """d(scale * aux_balance_loss)/dL, dense [T,E]:
    d/dP(e|t) = (log pbar_e + 1) / T; P = s / S gives
    d/ds_j = (c_j - sum_e c_e P_e) / (T S) with c = log pbar (the +1 cancels
    because sum_e P_e = 1); ds_j/dL_j = s_j (1 - s_j)."""
    L = _f64(L)
    if bias is not None:
        L = L + _f64(bias)[None, :]
    T = L.shape[0]
    s = sigmoid(L)
    S = s.sum(axis=1, keepdims=True)
    P = s / S
    c = np.log(P.mean(axis=0))[None, :]
    inner = (c * P).sum(axis=1, keepdims=True)
    return scale * s * (1.0 - s) * (c - inner) / (T * S)


# --------------------------------------------------------------------------
# Online load planning with dynamic replicas  [PLAN]: "TorchTitan Ascend开源" page,
# sections "在线负载规划" and "MoonEP动态负载均衡与专家并行优化": per-expert
# loads of the current batch plus each device's remaining capacity decide where
# hot experts get replicas; tokens keep their expert; in the page's figure 32
# unevenly spread tasks end as 4 on each of 8 ranks.
# --------------------------------------------------------------------------

def replica_plan(counts, P: int):
    """Greedy plan of an expert-parallel layout: rank r owns experts
    [r*E/P, (r+1)*E/P) (E divisible by P); every rank may process at most
    C = ceil(sum(counts) / P) rows.

    1. Each rank takes the rows of its own experts, in expert order, while it
       has capacity.
    2. The rows left over, expert by expert, go to ranks in rank order, each
       taking as many as its spare capacity allows (a replica of the expert).
    Returns (pieces, load): pieces = list of (expert, rank, first_row, n_rows)
    with rows counted within the expert's segment, in the order they were
    made; load[r] = rows rank r processes (max(load) = C)."""
    counts = [int(c) for c in counts]
    E = len(counts)
    assert E % P == 0
    per = E // P
    R = sum(counts)
    C = -(-R // P)
    load = [0] * P
    done = [0] * E
    pieces = []
    for r in range(P):
        for e in range(r * per, (r + 1) * per):
            take = min(counts[e], C - load[r])
            if take > 0:
                pieces.append((e, r, 0, take))
                load[r] += take
                done[e] = take
    for e in range(E):
        r = 0
        while done[e] < counts[e]:
            while load[r] >= C:
                r += 1
            take = min(counts[e] - done[e], C - load[r])
            pieces.append((e, r, done[e], take))
            load[r] += take
            done[e] += take
    return pieces, load


# --------------------------------------------------------------------------
# Multi-bucket batching  [BUCKET]: "大模型落地昇腾" page, section "二、算力侧":
# experts with similar token counts are grouped into buckets, each run with one
# batch shape.
# --------------------------------------------------------------------------

def expert_bucket_class(count, tile_m: int = 128) -> int:
    """0 for an empty expert, else 1 + floor(log2(ceil(count / tile_m))): experts
    in one class need the same number of tile_m-row tiles up to a factor < 2."""
    nt = -(-int(count) // tile_m)
    return 0 if nt == 0 else 1 + int(nt).bit_length() - 1


def bucket_order(counts, tile_m: int = 128):
    """Experts ordered by bucket class, largest class first, ascending expert id
    within a class, empty experts last; and the exclusive scan of their row
    tiles in that order. Returns (order [E], tile_sched_ordered [E+1])."""
    counts = [int(c) for c in counts]
    cls = [expert_bucket_class(c, tile_m) for c in counts]
    order = sorted(range(len(counts)), key=lambda e: (-cls[e], e))
    sched = [0]
    for e in order:
        sched.append(sched[-1] + -(-counts[e] // tile_m))
    return np.asarray(order, dtype=np.int64), np.asarray(sched, dtype=np.int64)


def ep_rank_forward(z_perm, counts, W13, W2, w, perm):
    """Expert compute of one expert-parallel rank on pre-permuted rows, then the
    weighted return to arrival order: out[perm[r]] = w[r] * o[r], where o[r] is
    the SwiGLU output of the expert owning row r. No cross-row reduction (the
    per-token sum happens on the token's home rank)."""
    offsets = expert_offsets(counts)
    y = grouped_swiglu(z_perm, W13, W2, offsets, w)
    out = np.empty_like(y)
    out[np.asarray(perm)] = y
    return out
