"""Run one libmoe entry point on a synthetic case of the layer's shapes.

For profiling single kernels (e.g. under ncu) without holding the whole layer:
each case allocates only what its entry point touches, calls it `--reps` times
after one warm-up call, and prints its average CUDA-event time.

    python -m sparse_moe_layer_topk_gb300.kernel_cases topk --reps 5
    python -m sparse_moe_layer_topk_gb300.kernel_cases gather --reps 5

Cases (T=16384 tokens, E=896 experts, k=16, l=1024 unless overridden):
  topk     moe_topk_from_logits on fp32 logits [T][E]
  permute  moe_permute (maps + row gather of z [T][l])
  gather   moe_unpermute_combine_bwd (row gather [T][l] -> [T*k][l])
  combine  moe_unpermute_combine ([T*k][l] + [T][l] -> [T][l])
"""
from __future__ import annotations

import argparse

import torch

from . import _lib as M
from . import build as B
from . import inputs as I


def _case(name, T, E, k, l):
    dev = "cuda"
    if name == "topk":
        L = I.make_logits(1, T, E).to(dev)
        idx = torch.empty(T, k, dtype=torch.int32, device=dev)
        w = torch.empty(T, k, dtype=torch.float32, device=dev)
        s = torch.empty(T, k, dtype=torch.float32, device=dev)
        return lambda: M.moe_topk_from_logits(L, None, T, E, k, idx, w, s)
    ids = I.make_topk_ids(2, T, E, k).to(dev)
    R = T * k
    if name == "permute":
        z = torch.randn(T, l, device=dev).to(torch.bfloat16)
        zp = torch.empty(R, l, dtype=torch.bfloat16, device=dev)
        bufs = [torch.empty(n, dtype=torch.int32, device=dev) for n in (E, E + 1, R, R, E + 1)]
        wsb = M.moe_workspace_size(M.MOE_OP_PERMUTE, T=T, E=E)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        return lambda: M.moe_permute(z, ids, None, T, l, E, k, zp, bufs[0], bufs[1], bufs[2],
                                     bufs[3], bufs[4], None, ws, wsb)
    perm = torch.randperm(R, generator=torch.Generator().manual_seed(3))
    token_of = (perm // k).to(torch.int32).to(dev)
    slot_of = torch.empty(R, dtype=torch.int32)
    slot_of[perm] = torch.arange(R, dtype=torch.int32)
    slot_of = slot_of.to(dev)
    if name == "gather":
        src = torch.randn(T, l, device=dev).to(torch.bfloat16)
        dst = torch.empty(R, l, dtype=torch.bfloat16, device=dev)
        return lambda: M.moe_unpermute_combine_bwd(src, token_of, T, k, l, dst)
    if name == "combine":
        yp = torch.randn(R, l, device=dev).to(torch.bfloat16)
        ysh = torch.randn(T, l, device=dev).to(torch.bfloat16)
        out = torch.empty(T, l, dtype=torch.bfloat16, device=dev)
        return lambda: M.moe_unpermute_combine(yp, slot_of, ysh, T, k, l, out)
    raise SystemExit(f"unknown case {name}")


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["topk", "permute", "gather", "combine"])
    ap.add_argument("--reps", type=int, default=5)
    ap.add_argument("--tokens", type=int, default=16384)
    ap.add_argument("--experts", type=int, default=896)
    ap.add_argument("--k", type=int, default=16)
    ap.add_argument("--latent", type=int, default=1024)
    a = ap.parse_args()
    B.build_library()
    fn = _case(a.case, a.tokens, a.experts, a.k, a.latent)
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(a.reps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    print(f"{a.case}: {e0.elapsed_time(e1) / a.reps * 1000:.1f} us per call")


if __name__ == "__main__":
    main()
