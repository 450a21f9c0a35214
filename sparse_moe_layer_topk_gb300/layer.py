"""The LatentMoE layer as a sequence of libmoe calls (forward and backward).

PyTorch only provides the device buffers and the stream; every step runs in a
libmoe CUDA kernel. One instance holds all activations, workspaces and weight
gradients for a fixed token count T, so a step allocates nothing.

Forward  (loss-free):  route_topk -> latent_proj(down) -> permute ->
         grouped_swiglu -> shared_swiglu -> unpermute_combine -> latent_proj(up)
Backward (dout given): latent_proj_bwd(up) -> unpermute_combine_bwd ->
         grouped_swiglu_bwd -> shared_swiglu_bwd -> permute_bwd ->
         latent_proj_bwd(down) -> route_topk_bwd (adds the router's dx)

With fused_gather the permute only builds the maps and the grouped GEMMs
gather their permuted rows from z and dy_lat themselves
(moe_grouped_swiglu[_bwd]_gather): z_perm and dy_perm are never written. It
saves ~1 GB of activations and ~2 GB of DRAM traffic at T=16384 but is slower
on GB300 (the row copies keep fewer bytes in flight per SM than the tiled TMA
loads of the permuted tensors), so the default is the explicit permute.

With fp8_cache the routed experts' GMM output [g|u] is kept for the backward
as E4M3 with one scale per row and 64 features (moe_grouped_swiglu[_bwd]_fp8cache)
instead of bf16: 1 + 1/16 bytes per value instead of 2, and the backward's
SwiGLU derivative reads the dequantized values.
"""
from __future__ import annotations

import torch

from . import _lib as M

BF16 = torch.bfloat16


class LatentMoELayer:
    def __init__(self, weights: dict, T: int, k: int, wgrad_dtype: int = M.MOE_DTYPE_F32,
                 device="cuda", fused_gather: bool = False, aux_scale: float = 0.0,
                 fp8_cache: bool = False):
        if fp8_cache and fused_gather:
            raise ValueError("fp8_cache runs with the explicit permute")
        self.w = weights
        self.fused_gather = fused_gather
        self.fp8_cache = fp8_cache
        self.aux_scale = aux_scale  # > 0: add aux_scale * the auxiliary balance loss
        self.T = T
        self.k = k
        self.d, self.E = weights["Wr"].shape
        self.l = weights["W_dn"].shape[1]
        self.f = weights["W2"].shape[1]
        self.S = weights["W13_sh"].shape[0]
        self.R = T * k
        self.wgrad_dtype = wgrad_dtype
        dev = torch.device(device)
        T_, k_, d, l, f, E, S, R = T, k, self.d, self.l, self.f, self.E, self.S, self.R
        e = lambda *shape, dt=BF16: torch.empty(shape, dtype=dt, device=dev)  # noqa: E731
        wdt = torch.float32 if wgrad_dtype == M.MOE_DTYPE_F32 else BF16
        # forward activations
        self.topk_idx = e(T_, k_, dt=torch.int32)
        self.topk_w = e(T_, k_, dt=torch.float32)
        self.topk_s = e(T_, k_, dt=torch.float32)
        self.z = e(T_, l)
        self.counts = e(E, dt=torch.int32)
        self.offsets = e(E + 1, dt=torch.int32)
        self.tile_sched = e(E + 1, dt=torch.int32)
        self.slot_of = e(T_, k_, dt=torch.int32)
        self.token_of = e(R, dt=torch.int32)
        self.row_w = e(R, dt=torch.float32)
        self.z_perm = None if fused_gather else e(R, l)
        self.gu = None if fp8_cache else e(R, 2 * f)
        self.gu8 = e(R, 2 * f, dt=torch.uint8) if fp8_cache else None
        self.gu_scale = e(R, 2 * f // 64, dt=torch.float32) if fp8_cache else None
        self.h = e(R, f)
        self.y_perm = e(R, l)
        self.gu_sh = e(T_, S * 2 * f)
        self.h_sh = e(T_, S * f)
        self.y_sh = e(T_, l)
        self.y_lat = e(T_, l)
        self.out = e(T_, d)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        # backward
        self.dy_lat = e(T_, l)
        self.dy_perm = None if fused_gather else e(R, l)
        self.dz_perm = e(R, l)
        self.d_row_w = e(R, dt=torch.float32)
        self.d_topk_w = e(T_, k_, dt=torch.float32)
        self.dz_sh = e(T_, l)
        self.dz = e(T_, l)
        self.dx = e(T_, d)
        self.grads = {
            "W_up": e(l, d, dt=wdt), "W_dn": e(d, l, dt=wdt), "Wr": e(d, E, dt=wdt),
            "W13": e(E, l, 2 * f, dt=wdt), "W2": e(E, f, l, dt=wdt),
            "W13_sh": e(S, l, 2 * f, dt=wdt), "W2_sh": e(S, f, l, dt=wdt),
        }
        # workspaces
        ws = lambda op, **kw: M.moe_workspace_size(op, **kw)  # noqa: E731
        self.ws_sizes = {
            "route": ws(M.MOE_OP_ROUTE_TOPK, T=T_, E=E),
            "permute": ws(M.MOE_OP_PERMUTE, T=T_, E=E),
            "gbwd": ws(M.MOE_OP_GROUPED_SWIGLU_BWD, T=R, k=1, f=f),
            "sbwd": ws(M.MOE_OP_SHARED_SWIGLU_BWD, T=T_, l=l, f=f, S=S),
            "rbwd": ws(M.MOE_OP_ROUTE_TOPK_BWD, T=T_, E=E),
            "aux": ws(M.MOE_OP_ROUTER_AUX, T=T_, E=E),
        }
        self.p_mean = e(E, dt=torch.float32)
        self.aux_loss = e(1, dt=torch.float32)
        self.ws = {n: torch.empty(max(b, 256), dtype=torch.uint8, device=dev)
                   for n, b in self.ws_sizes.items()}

    # ------------------------------------------------------------------ forward
    def forward(self, x, stream=None):
        w, T, k, d, l, f, E, S, R = (self.w, self.T, self.k, self.d, self.l, self.f, self.E,
                                     self.S, self.R)
        self.x = x
        # router logits, top-k and the latent z = x W_dn (one GEMM over [Wr | W_dn])
        M.moe_route_topk_latent(x, w["Wr"], w.get("bias"), w["W_dn"], T, d, E, k, l,
                                self.topk_idx, self.topk_w, self.topk_s, self.z, self.ws["route"],
                                self.ws_sizes["route"], self.err, stream)
        if self.aux_scale > 0:
            # the router logits stay in the route workspace until the backward
            M.moe_router_aux_loss(self.ws["route"], w.get("bias"), T, E, self.p_mean, self.aux_loss,
                                  self.ws["aux"], self.ws_sizes["aux"], stream)
        fused = self.fused_gather
        M.moe_permute(None if fused else self.z, self.topk_idx, self.topk_w, T, l, E, k,
                      self.z_perm, self.counts, self.offsets, self.slot_of, self.token_of,
                      self.tile_sched, self.row_w, self.ws["permute"], self.ws_sizes["permute"],
                      self.err, stream)
        if fused:
            M.moe_grouped_swiglu_gather(self.z, self.token_of, T, w["W13"], w["W2"], self.offsets,
                                        self.tile_sched, self.row_w, E, R, l, f, self.gu, self.h,
                                        self.y_perm, stream)
        elif self.fp8_cache:
            M.moe_grouped_swiglu_fp8cache(self.z_perm, w["W13"], w["W2"], self.offsets,
                                          self.tile_sched, self.row_w, E, R, l, f, self.gu8,
                                          self.gu_scale, self.h, self.y_perm, stream)
        else:
            M.moe_grouped_swiglu(self.z_perm, w["W13"], w["W2"], self.offsets, self.tile_sched,
                                 self.row_w, E, R, l, f, self.gu, self.h, self.y_perm, stream)
        M.moe_shared_swiglu(self.z, w["W13_sh"], w["W2_sh"], T, l, f, S, self.gu_sh, self.h_sh,
                            self.y_sh, stream)
        M.moe_unpermute_combine(self.y_perm, self.slot_of, self.y_sh, T, k, l, self.y_lat, stream)
        M.moe_latent_proj(self.y_lat, w["W_up"], T, l, d, self.out, stream)
        return self.out

    # ------------------------------------------------------------------ backward
    def backward(self, dout, stream=None):
        w, T, k, d, l, f, E, S, R = (self.w, self.T, self.k, self.d, self.l, self.f, self.E,
                                     self.S, self.R)
        g = self.grads
        wd = self.wgrad_dtype
        M.moe_latent_proj_bwd(dout, self.y_lat, w["W_up"], T, l, d, self.dy_lat, g["W_up"], wd,
                              stream)
        if self.fused_gather:
            M.moe_grouped_swiglu_bwd_gather(self.dy_lat, self.z, self.token_of, T, w["W13"],
                                            w["W2"], self.gu, self.h, self.row_w, self.offsets,
                                            self.tile_sched, E, R, l, f, self.dz_perm,
                                            self.d_row_w, g["W13"], g["W2"], wd, self.ws["gbwd"],
                                            self.ws_sizes["gbwd"], stream)
        elif self.fp8_cache:
            M.moe_unpermute_combine_bwd(self.dy_lat, self.token_of, T, k, l, self.dy_perm, stream)
            M.moe_grouped_swiglu_bwd_fp8cache(self.dy_perm, self.z_perm, w["W13"], w["W2"],
                                              self.gu8, self.gu_scale, self.h, self.row_w,
                                              self.offsets, self.tile_sched, E, R, l, f,
                                              self.dz_perm, self.d_row_w, g["W13"], g["W2"], wd,
                                              self.ws["gbwd"], self.ws_sizes["gbwd"], stream)
        else:
            M.moe_unpermute_combine_bwd(self.dy_lat, self.token_of, T, k, l, self.dy_perm, stream)
            M.moe_grouped_swiglu_bwd(self.dy_perm, self.z_perm, w["W13"], w["W2"], self.gu,
                                     self.h, self.row_w, self.offsets, self.tile_sched, E, R, l,
                                     f, self.dz_perm, self.d_row_w, g["W13"], g["W2"], wd,
                                     self.ws["gbwd"], self.ws_sizes["gbwd"], stream)
        M.moe_shared_swiglu_bwd(self.dy_lat, self.z, w["W13_sh"], w["W2_sh"], self.gu_sh,
                                self.h_sh, T, l, f, S, self.dz_sh, g["W13_sh"], g["W2_sh"], wd,
                                self.ws["sbwd"], self.ws_sizes["sbwd"], stream)
        M.moe_permute_bwd(self.dz_perm, self.slot_of, self.dz_sh, T, k, l, self.dz, stream)
        # dW_dn here; dx = dz W_dn^T + dL Wr^T in the router backward's fused GEMM
        M.moe_latent_proj_bwd(self.dz, self.x, w["W_dn"], T, d, l, None, g["W_dn"], wd, stream)
        aux = self.aux_scale > 0
        M.moe_route_topk_bwd(self.d_row_w, self.slot_of, self.topk_idx, self.topk_w, self.topk_s,
                             self.x, w["Wr"], T, d, E, k, self.d_topk_w, self.dx, g["Wr"], wd,
                             self.ws["route"] if aux else None, w.get("bias") if aux else None,
                             self.p_mean if aux else None, self.aux_scale, self.dz, w["W_dn"], l,
                             self.ws["rbwd"], self.ws_sizes["rbwd"], self.err, stream)
        return self.dx

    def step(self, x, dout, stream=None):
        self.forward(x, stream)
        return self.backward(dout, stream)

    def capture_step(self, x, dout):
        """Records one forward + backward on the fixed buffers x and dout as a
        CUDA graph; graph.replay() reruns it on the current stream. A step
        allocates nothing and never waits on the host, so it captures whole (run
        one eager step first: the library sets its kernels' attributes then)."""
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.step(x, dout)
        return g

    def capture_halves(self, x, dout):
        """The forward on x and the backward on dout as two CUDA graphs, so that
        a step may start before its dout has arrived."""
        gf = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gf):
            self.forward(x)
        gb = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gb):
            self.backward(dout)
        return gf, gb

    def steps_from_host(self, x_host, g_host, dx_host, graphs: bool = True):
        """Forward + backward for each (x, dout) pair of pinned host tensors,
        writing each step's input gradient back to the pinned dx_host[i].

        The host->device copy of step i+1 and the device->host copy of step i-1
        run on their own streams (separate copy engines) while step i computes;
        device inputs and input gradients are double-buffered and ordered with
        events, so every step still copies its own inputs in and its gradient
        out. A step's forward waits for its x alone and its backward for its
        dout, which is copied in after x. With graphs, each slot's forward and
        backward are CUDA graphs captured on first use. Returns after the last copy has been enqueued; synchronise the
        current stream's device to wait for the results."""
        n = len(x_host)
        assert len(g_host) == n and len(dx_host) == n
        dev = self.dx.device
        comp = torch.cuda.current_stream()
        h2d = torch.cuda.Stream(device=dev)
        d2h = torch.cuda.Stream(device=dev)
        if not hasattr(self, "_pipe"):
            self._pipe = {
                "x": [torch.empty_like(self.dx) for _ in range(2)],
                "g": [torch.empty_like(self.dx) for _ in range(2)],
                "dx": [torch.empty_like(self.dx) for _ in range(2)],
            }
        P = self._pipe
        if graphs and not hasattr(self, "_pipe_graphs"):
            keep = self.dx
            self._pipe_graphs = []
            for s in range(2):
                self.dx = P["dx"][s]
                self._pipe_graphs.append(self.capture_halves(P["x"][s], P["g"][s]))
            self.dx = keep
        ev = lambda: torch.cuda.Event()  # noqa: E731
        loaded_x = [None] * n
        loaded_g = [None] * n
        computed = [None] * n
        drained = [None] * n

        def load(i):
            s = i & 1
            with torch.cuda.stream(h2d):
                if i >= 2:
                    h2d.wait_event(computed[i - 2])  # slot s no longer read by step i-2
                P["x"][s].copy_(x_host[i], non_blocking=True)
                loaded_x[i] = ev()
                loaded_x[i].record(h2d)
                P["g"][s].copy_(g_host[i], non_blocking=True)
                loaded_g[i] = ev()
                loaded_g[i].record(h2d)

        keep = self.dx  # the eager steps write their input gradient into the slots
        load(0)
        try:
            for i in range(n):
                s = i & 1
                if i + 1 < n:
                    load(i + 1)
                comp.wait_event(loaded_x[i])
                if graphs:
                    self._pipe_graphs[s][0].replay()
                else:
                    self.forward(P["x"][s])
                comp.wait_event(loaded_g[i])
                if i >= 2:
                    comp.wait_event(drained[i - 2])  # dx slot s copied out by step i-2
                if graphs:
                    self._pipe_graphs[s][1].replay()
                else:
                    self.dx = P["dx"][s]
                    self.backward(P["g"][s])
                computed[i] = ev()
                computed[i].record(comp)
                with torch.cuda.stream(d2h):
                    d2h.wait_event(computed[i])
                    dx_host[i].copy_(P["dx"][s], non_blocking=True)
                    drained[i] = ev()
                    drained[i].record(d2h)
        finally:
            self.dx = keep
        comp.wait_event(drained[n - 1])


def weights_to_device(inp: dict, device="cuda") -> dict:
    names = ("Wr", "W_dn", "W13", "W2", "W13_sh", "W2_sh", "W_up")
    out = {n: inp[n].to(device) for n in names}
    out["bias"] = inp["bias"].to(device) if inp.get("bias") is not None else None
    return out
