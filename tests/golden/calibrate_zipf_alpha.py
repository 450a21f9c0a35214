"""Choose the scale alpha of the Zipf(1.1) router bias of the skewed workload
(T=4096, d=4096, E=896, top-16): b_e = alpha * ln(p_pi(e)), p_r ~ r^-1.1.

Target statistics of the skewed workload: the top 5% of experts hold more than
30% of the assignments and about 200 experts receive 0-2 tokens. Routing is
computed with the fp64 oracle only. Prints one line per candidate alpha and
the bisection result for "experts with 0-2 tokens" = 200.

Run:  python tests/golden/calibrate_zipf_alpha.py
"""
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle as O  # noqa: E402
from sparse_moe_layer_topk_gb300 import inputs as I  # noqa: E402


def stats(L0, bias_unit, alpha, k, E):
    idx = O.topk_select(L0 + alpha * bias_unit[None, :], k)
    counts = O.expert_counts(idx, E)
    top = np.sort(counts)[::-1]
    n5 = int(round(0.05 * E))
    return top[:n5].sum() / counts.sum(), int((counts <= 2).sum())


def main():
    cfg = I.CONFIGS[2]
    inp = I.make_layer_inputs(cfg)
    L0 = O.router_logits(inp["x"], inp["Wr"])
    unit = I.to_f64(inp["bias"]) / I.ZIPF_ALPHA        # ln(p_pi(e))
    for a in (0.25, 0.5, 0.75, 1.0, 1.25, 1.5, 2.0):
        share, low = stats(L0, unit, a, cfg.k, cfg.E)
        print(f"alpha={a:.3f} top5%share={share:.3f} experts_with_0..2={low}")
    lo, hi = 0.0, 4.0
    for _ in range(30):
        mid = 0.5 * (lo + hi)
        if stats(L0, unit, mid, cfg.k, cfg.E)[1] < 200:
            lo = mid
        else:
            hi = mid
    share, low = stats(L0, unit, hi, cfg.k, cfg.E)
    print(f"bisection: alpha={hi:.4f} top5%share={share:.3f} experts_with_0..2={low}")


if __name__ == "__main__":
    main()
