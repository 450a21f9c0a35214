"""Seeded synthetic inputs for the LatentMoE layer (configurations 0-4).

This module only draws random numbers and rounds them to bf16. It holds none
of the layer's arithmetic, so both the CUDA path and the fp64 oracle can take
their inputs from it without sharing any computation.

Every tensor is drawn from its own child of ``numpy.random.SeedSequence(seed)``
(numpy's PCG64 + ziggurat normals are bit-reproducible across platforms), so a
tensor does not depend on which other tensors were drawn, and the per-expert
weight slabs can be drawn in parallel threads.

Shapes follow the model description on the "TorchTitan Ascend开源" page,
section "Kimi K3.1 Pro 模型结构" (896 routed experts, 16 active, 2 shared,
experts in a low-dimensional latent space), at the sizes of the five
workloads below.
"""
from __future__ import annotations

import dataclasses
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

__all__ = ["LayerConfig", "CONFIGS", "EPRankConfig", "EP_RANK", "make_layer_inputs",
           "make_ep_rank_inputs", "make_logits", "make_topk_ids", "ZIPF_ALPHA", "to_f64"]


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    name: str
    seed: int
    T: int      # tokens
    d: int      # model width
    l: int      # latent width
    E: int      # routed experts
    k: int      # experts per token
    S: int      # shared experts
    f: int      # expert FFN width
    skew: bool = False      # Zipf(1.1) per-expert router bias
    backward: bool = False  # draw the upstream gradient g as well


CONFIGS = {
    0: LayerConfig("tiny_T256_E64_top4", 0, 256, 256, 128, 64, 4, 1, 64),
    1: LayerConfig("latentmoe_T4096_E896_top16", 1, 4096, 4096, 1024, 896, 16, 2, 512),
    2: LayerConfig("latentmoe_zipf_T4096_E896_top16", 2, 4096, 4096, 1024, 896, 16, 2, 512,
                   skew=True),
    4: LayerConfig("latentmoe_fwd_bwd_T16384_E896_top16", 4, 16384, 4096, 1024, 896, 16, 2, 512,
                   backward=True),
}


@dataclasses.dataclass(frozen=True)
class EPRankConfig:
    name: str = "ep64_rank_14experts_R65536"
    seed: int = 3
    E: int = 14
    R: int = 65536
    l: int = 1024
    f: int = 512
    dirichlet_alpha: float = 0.5
    w_lo: float = 0.01
    w_hi: float = 0.2


EP_RANK = EPRankConfig()

# Scale of the Zipf router bias b_e = ZIPF_ALPHA * ln(p_pi(e)), p_r ~ r^-1.1.
# Chosen once (bisection over alpha with the oracle's routing, script
# tests/golden/calibrate_zipf_alpha.py) so that at T=4096 the top 5% of experts
# hold >30% of the assignments and about 200 experts receive 0-2 tokens.
ZIPF_ALPHA = 0.78

_N_THREADS = max(1, min(16, os.cpu_count() or 1))


def _normal_f32(seq: np.random.SeedSequence, shape, std: float) -> np.ndarray:
    a = np.random.default_rng(seq).standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        a *= np.float32(std)
    return a


def _bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)


def _normal_bf16(seq, shape, std) -> torch.Tensor:
    return _bf16(_normal_f32(seq, shape, std))


def _stacked_normal_bf16(seq, n: int, shape, std) -> torch.Tensor:
    """n independent slabs of `shape`, slab i drawn from child i of `seq`."""
    out = torch.empty((n,) + tuple(shape), dtype=torch.bfloat16)
    kids = seq.spawn(n)

    def fill(i):
        out[i].copy_(_normal_bf16(kids[i], shape, std))

    with ThreadPoolExecutor(_N_THREADS) as ex:
        list(ex.map(fill, range(n)))
    return out


def make_layer_inputs(cfg: LayerConfig | int, T: int | None = None,
                      std_w: float = 0.02) -> dict:
    """Inputs of one layer call: activations, weights, optional bias and dout.

    Layouts (row-major, bf16 unless noted):
      x [T,d]; Wr [d,E]; bias [E] fp32 or None; W_dn [d,l];
      W13 [E,l,2f] (gate columns 0..f-1, up columns f..2f-1); W2 [E,f,l];
      W13_sh [S,l,2f]; W2_sh [S,f,l]; W_up [l,d]; g [T,d] (upstream gradient).
    `T` overrides the token count (the weights do not depend on it).
    """
    if isinstance(cfg, int):
        cfg = CONFIGS[cfg]
    T = cfg.T if T is None else T
    root = np.random.SeedSequence(cfg.seed)
    (s_x, s_wr, s_dn, s_13, s_2, s_13sh, s_2sh, s_up, s_g, s_bias) = root.spawn(10)
    d, l, E, S, f = cfg.d, cfg.l, cfg.E, cfg.S, cfg.f
    inp = {
        "cfg": cfg,
        "x": _normal_bf16(s_x, (T, d), 1.0),
        "Wr": _normal_bf16(s_wr, (d, E), std_w),
        "W_dn": _normal_bf16(s_dn, (d, l), std_w),
        "W13": _stacked_normal_bf16(s_13, E, (l, 2 * f), std_w),
        "W2": _stacked_normal_bf16(s_2, E, (f, l), std_w),
        "W13_sh": _stacked_normal_bf16(s_13sh, S, (l, 2 * f), std_w),
        "W2_sh": _stacked_normal_bf16(s_2sh, S, (f, l), std_w),
        "W_up": _normal_bf16(s_up, (l, d), std_w),
        "bias": None,
        "g": _normal_bf16(s_g, (T, d), 1.0),
    }
    if cfg.skew:
        rng = np.random.default_rng(s_bias)
        perm = rng.permutation(E)
        ranks = np.arange(1, E + 1, dtype=np.float64)
        p = ranks ** -1.1
        p /= p.sum()
        inp["bias"] = torch.from_numpy((ZIPF_ALPHA * np.log(p[perm])).astype(np.float32))
    return inp


def make_ep_rank_inputs(cfg: EPRankConfig = EP_RANK) -> dict:
    """Pre-permuted rows of one expert-parallel rank (14 local experts).

    counts ~ Multinomial(R, Dirichlet(alpha)); z_perm [R,l] ~ N(0,1) bf16 (rows of
    expert e are contiguous, experts in order); w [R] ~ U(w_lo, w_hi) fp32;
    perm [R] int64 is the arrival permutation pi (slot r returns to row perm[r]);
    W13 [E,l,2f], W2 [E,f,l] ~ N(0, 0.02) bf16.
    """
    root = np.random.SeedSequence(cfg.seed)
    s_cnt, s_z, s_w, s_pi, s_13, s_2 = root.spawn(6)
    rng = np.random.default_rng(s_cnt)
    probs = rng.dirichlet(np.full(cfg.E, cfg.dirichlet_alpha))
    counts = rng.multinomial(cfg.R, probs).astype(np.int32)
    w = np.random.default_rng(s_w).uniform(cfg.w_lo, cfg.w_hi, cfg.R).astype(np.float32)
    perm = np.random.default_rng(s_pi).permutation(cfg.R)
    return {
        "cfg": cfg,
        "counts": torch.from_numpy(counts),
        "z_perm": _normal_bf16(s_z, (cfg.R, cfg.l), 1.0),
        "w": torch.from_numpy(w),
        "perm": torch.from_numpy(perm.astype(np.int64)),
        "W13": _stacked_normal_bf16(s_13, cfg.E, (cfg.l, 2 * cfg.f), 0.02),
        "W2": _stacked_normal_bf16(s_2, cfg.E, (cfg.f, cfg.l), 0.02),
    }


def make_logits(seed: int, T: int, E: int, ties: bool = False) -> torch.Tensor:
    """fp32 router logits [T,E] ~ N(0, 1.28^2) (the spread x@Wr has at d=4096).

    With ties=True the values are quantised to multiples of 1/8 in [-4, 4], so
    that most tokens hold exactly equal logits around their top-k boundary.
    """
    a = _normal_f32(np.random.SeedSequence(seed), (T, E), 1.28)
    if ties:
        a = np.clip(np.round(a * 8.0) / 8.0, -4.0, 4.0).astype(np.float32)
    return torch.from_numpy(a)


def make_topk_ids(seed: int, T: int, E: int, k: int, skew: float = 0.0) -> torch.Tensor:
    """Distinct expert ids [T,k] int32 per token, uniform or Zipf-skewed choice."""
    rng = np.random.default_rng(np.random.SeedSequence(seed))
    if skew > 0:
        p = np.arange(1, E + 1, dtype=np.float64) ** -skew
        p /= p.sum()
        p = p[rng.permutation(E)]
    else:
        p = None
    out = np.empty((T, k), dtype=np.int32)
    for t in range(T):
        out[t] = rng.choice(E, size=k, replace=False, p=p)
    return torch.from_numpy(out)


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact widening of a bf16/fp32 tensor to a float64 numpy array."""
    return t.detach().to("cpu", torch.float64).numpy()
