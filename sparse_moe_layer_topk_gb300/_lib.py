"""ctypes binding of libmoe: one Python function per C entry point, same name
and argument order (include/moe.h). Only argument marshalling happens here:
tensors become device pointers, `stream=None` becomes torch's current CUDA
stream, and a non-zero status raises MoEError. Every computation runs in the
library's CUDA kernels; there is no fallback when the library is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_ARG = -1
MOE_ERR_ALIGN = -2
MOE_ERR_WORKSPACE = -3
MOE_ERR_UNSUPPORTED = -4
MOE_ERR_CUDA = -5
MOE_FLAG_BAD_EXPERT = 1
MOE_FLAG_NONFINITE = 2
MOE_FLAG_TIMEOUT = 4
MOE_DTYPE_F32 = 0
MOE_DTYPE_BF16 = 1
MOE_OP_ROUTE_TOPK = 1
MOE_OP_PERMUTE = 2
MOE_OP_GROUPED_SWIGLU_BWD = 3
MOE_OP_SHARED_SWIGLU_BWD = 4
MOE_OP_ROUTE_TOPK_BWD = 5
MOE_OP_ROUTER_AUX = 6

_P = ctypes.c_void_p
_I = ctypes.c_int
_Z = ctypes.c_size_t
_F = ctypes.c_float

# name -> argument types (pointer args are _P; the last one is always the stream)
SIGNATURES = {
    "moe_version": ([], _I),
    "moe_status_string": ([_I], ctypes.c_char_p),
    "moe_last_cuda_error": ([], _I),
    "moe_workspace_size": ([_I, _I, _I, _I, _I, _I, _I, _I], _Z),
    "moe_router_logits": ([_P, _P, _I, _I, _I, _P, _P], _I),
    "moe_topk_from_logits": ([_P, _P, _I, _I, _I, _P, _P, _P, _P, _P], _I),
    "moe_route_topk": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _Z, _P, _P], _I),
    "moe_route_topk_latent": ([_P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _Z, _P, _P],
                              _I),
    "moe_permute": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _P, _P], _I),
    "moe_permute_noalloc": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "moe_latent_proj": ([_P, _P, _I, _I, _I, _P, _P], _I),
    "moe_latent_proj_bwd": ([_P, _P, _P, _I, _I, _I, _P, _P, _I, _P], _I),
    "moe_grouped_swiglu": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_grouped_swiglu_fp8cache": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P],
                                    _I),
    "moe_grouped_swiglu_gather": ([_P, _P, _I, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P],
                                  _I),
    "moe_grouped_swiglu_bwd_gather": ([_P, _P, _P, _I, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                       _P, _P, _P, _P, _I, _P, _Z, _P], _I),
    "moe_shared_swiglu": ([_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P], _I),
    "moe_unpermute_combine": ([_P, _P, _P, _I, _I, _I, _P, _P], _I),
    "moe_unpermute_combine_bwd": ([_P, _P, _I, _I, _I, _P, _P], _I),
    "moe_grouped_swiglu_bwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P,
                                _I, _P, _Z, _P], _I),
    "moe_grouped_swiglu_bwd_fp8cache": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I,
                                         _P, _P, _P, _P, _I, _P, _Z, _P], _I),
    "moe_shared_swiglu_bwd": ([_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _I, _P, _Z, _P],
                              _I),
    "moe_permute_bwd": ([_P, _P, _P, _I, _I, _I, _P, _P], _I),
    "moe_route_topk_bwd": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _I, _P, _P, _P,
                            _F, _P, _P, _I, _P, _Z, _P, _P], _I),
    "moe_router_aux_loss": ([_P, _P, _I, _I, _P, _P, _P, _Z, _P], _I),
    "moe_replica_plan": ([_P, _I, _I, _P, _P, _P, _P], _I),
    "moe_expert_buckets": ([_P, _I, _P, _P, _P], _I),
    "moe_grouped_swiglu_ordered": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _P],
                                   _I),
    "moe_diag_wait_timeout": ([ctypes.c_longlong, _P, _P, _P], _I),
    "moe_timing_enable": ([_I], _I),
    "moe_timing_report": ([ctypes.c_char_p, _Z], _I),
}


class MoEError(RuntimeError):
    pass


_lib = None


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmoe.so (built by build.build_library); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(path):
            raise MoEError(f"{path} is missing: build it with "
                           "sparse_moe_layer_topk_gb300.build.build_library()")
        lib = ctypes.CDLL(path)
        for name, (args, res) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = res
        _lib = lib
    return _lib


_EMPTY = {}


def _empty_ptr(device):
    """A valid, aligned device address standing for an array of zero elements:
    the library refuses null pointers and never touches a zero-length array."""
    t = _EMPTY.get(device)
    if t is None:
        t = _EMPTY[device] = torch.empty(256, dtype=torch.uint8, device=device)
    return t.data_ptr()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        if not x.is_cuda:
            if x.numel():
                raise MoEError("libmoe takes device tensors")
            return None
        return x.data_ptr() if x.numel() else _empty_ptr(x.device)
    return int(x)


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, torch.cuda.Stream):
        return s.cuda_stream
    return int(s)


def _check(status: int, name: str):
    if status != MOE_OK:
        msg = load().moe_status_string(status).decode()
        extra = ""
        if status == MOE_ERR_CUDA:
            extra = f" (cudaError {load().moe_last_cuda_error()})"
        raise MoEError(f"{name} failed: {msg}{extra}")


def _call(name, *args):
    lib = load()
    argtypes = SIGNATURES[name][0]
    conv = []
    for a, t in zip(args[:-1], argtypes[:-1]):
        conv.append(_ptr(a) if t is _P else a)
    conv.append(_stream(args[-1]))
    _check(getattr(lib, name)(*conv), name)


def moe_version() -> int:
    return load().moe_version()


def moe_workspace_size(op, T=0, d=0, l=0, E=0, k=0, f=0, S=0) -> int:
    return load().moe_workspace_size(op, T, d, l, E, k, f, S)


def moe_router_logits(x, Wr, T, d, E, logits, stream=None):
    _call("moe_router_logits", x, Wr, T, d, E, logits, stream)


def moe_topk_from_logits(logits, bias, T, E, k, topk_idx, topk_w, topk_s, err_flag=None,
                         stream=None):
    _call("moe_topk_from_logits", logits, bias, T, E, k, topk_idx, topk_w, topk_s, err_flag,
          stream)


def moe_route_topk(x, Wr, bias, T, d, E, k, topk_idx, topk_w, topk_s, ws, ws_bytes,
                   err_flag=None, stream=None):
    _call("moe_route_topk", x, Wr, bias, T, d, E, k, topk_idx, topk_w, topk_s, ws, ws_bytes,
          err_flag, stream)


def moe_route_topk_latent(x, Wr, bias, W_dn, T, d, E, k, l, topk_idx, topk_w, topk_s, z, ws,
                          ws_bytes, err_flag=None, stream=None):
    _call("moe_route_topk_latent", x, Wr, bias, W_dn, T, d, E, k, l, topk_idx, topk_w, topk_s, z,
          ws, ws_bytes, err_flag, stream)


def moe_permute(z, topk_idx, topk_w, T, l, E, k, z_perm, counts, offsets, slot_of, token_of,
                tile_sched, row_w, ws, ws_bytes, err_flag=None, stream=None):
    _call("moe_permute", z, topk_idx, topk_w, T, l, E, k, z_perm, counts, offsets, slot_of,
          token_of, tile_sched, row_w, ws, ws_bytes, err_flag, stream)


def moe_permute_noalloc(z, topk_idx, topk_w, T, l, E, k, z_perm, counts, offsets, slot_of,
                        token_of, tile_sched, row_w, err_flag=None, stream=None):
    """moe_permute without a workspace argument, for callers that cannot allocate
    device memory; the scratch is a fixed array inside the library (see moe.h)."""
    _call("moe_permute_noalloc", z, topk_idx, topk_w, T, l, E, k, z_perm, counts, offsets,
          slot_of, token_of, tile_sched, row_w, err_flag, stream)


def moe_latent_proj(inp, W, M, K, N, out, stream=None):
    _call("moe_latent_proj", inp, W, M, K, N, out, stream)


def moe_latent_proj_bwd(dout, inp, W, M, K, N, din, dW, wgrad_dtype, stream=None):
    _call("moe_latent_proj_bwd", dout, inp, W, M, K, N, din, dW, wgrad_dtype, stream)


def moe_grouped_swiglu(z_perm, W13, W2, offsets, tile_sched, row_w, E, R, l, f, gu_save, h,
                       y_perm, stream=None):
    _call("moe_grouped_swiglu", z_perm, W13, W2, offsets, tile_sched, row_w, E, R, l, f, gu_save,
          h, y_perm, stream)


def moe_grouped_swiglu_fp8cache(z_perm, W13, W2, offsets, tile_sched, row_w, E, R, l, f, gu8,
                                gu_scale, h, y_perm, stream=None):
    _call("moe_grouped_swiglu_fp8cache", z_perm, W13, W2, offsets, tile_sched, row_w, E, R, l, f,
          gu8, gu_scale, h, y_perm, stream)


def moe_grouped_swiglu_gather(z, token_of, T, W13, W2, offsets, tile_sched, row_w, E, R, l, f,
                              gu_save, h, y_perm, stream=None):
    _call("moe_grouped_swiglu_gather", z, token_of, T, W13, W2, offsets, tile_sched, row_w, E, R,
          l, f, gu_save, h, y_perm, stream)


def moe_grouped_swiglu_bwd_gather(dy_lat, z, token_of, T, W13, W2, gu_save, h, row_w, offsets,
                                  tile_sched, E, R, l, f, dz_perm, d_row_w, dW13, dW2, wgrad_dtype,
                                  ws, ws_bytes, stream=None):
    _call("moe_grouped_swiglu_bwd_gather", dy_lat, z, token_of, T, W13, W2, gu_save, h, row_w,
          offsets, tile_sched, E, R, l, f, dz_perm, d_row_w, dW13, dW2, wgrad_dtype, ws, ws_bytes,
          stream)


def moe_shared_swiglu(z, W13_sh, W2_sh, T, l, f, S, gu_save, h, y_sh, stream=None):
    _call("moe_shared_swiglu", z, W13_sh, W2_sh, T, l, f, S, gu_save, h, y_sh, stream)


def moe_unpermute_combine(y_perm, slot_of, y_shared, T, k, l, y_lat, stream=None):
    _call("moe_unpermute_combine", y_perm, slot_of, y_shared, T, k, l, y_lat, stream)


def moe_unpermute_combine_bwd(dy_lat, token_of, T, k, l, dy_perm, stream=None):
    _call("moe_unpermute_combine_bwd", dy_lat, token_of, T, k, l, dy_perm, stream)


def moe_grouped_swiglu_bwd(dy_perm, z_perm, W13, W2, gu_save, h, row_w, offsets, tile_sched, E,
                           R, l, f, dz_perm, d_row_w, dW13, dW2, wgrad_dtype, ws, ws_bytes,
                           stream=None):
    _call("moe_grouped_swiglu_bwd", dy_perm, z_perm, W13, W2, gu_save, h, row_w, offsets,
          tile_sched, E, R, l, f, dz_perm, d_row_w, dW13, dW2, wgrad_dtype, ws, ws_bytes, stream)


def moe_grouped_swiglu_bwd_fp8cache(dy_perm, z_perm, W13, W2, gu8, gu_scale, h, row_w, offsets,
                                    tile_sched, E, R, l, f, dz_perm, d_row_w, dW13, dW2,
                                    wgrad_dtype, ws, ws_bytes, stream=None):
    _call("moe_grouped_swiglu_bwd_fp8cache", dy_perm, z_perm, W13, W2, gu8, gu_scale, h, row_w,
          offsets, tile_sched, E, R, l, f, dz_perm, d_row_w, dW13, dW2, wgrad_dtype, ws, ws_bytes,
          stream)


def moe_shared_swiglu_bwd(dy, z, W13_sh, W2_sh, gu_save, h, T, l, f, S, dz_sh, dW13_sh, dW2_sh,
                          wgrad_dtype, ws, ws_bytes, stream=None):
    _call("moe_shared_swiglu_bwd", dy, z, W13_sh, W2_sh, gu_save, h, T, l, f, S, dz_sh, dW13_sh,
          dW2_sh, wgrad_dtype, ws, ws_bytes, stream)


def moe_permute_bwd(dz_perm, slot_of, dz_shared, T, k, l, dz, stream=None):
    _call("moe_permute_bwd", dz_perm, slot_of, dz_shared, T, k, l, dz, stream)


def moe_route_topk_bwd(d_row_w, slot_of, topk_idx, topk_w, topk_s, x, Wr, T, d, E, k, d_topk_w,
                       dx_accum, dWr, wgrad_dtype, aux_logits, aux_bias, aux_p_mean, aux_scale, dz,
                       W_dn, l, ws, ws_bytes, err_flag=None, stream=None):
    _call("moe_route_topk_bwd", d_row_w, slot_of, topk_idx, topk_w, topk_s, x, Wr, T, d, E, k,
          d_topk_w, dx_accum, dWr, wgrad_dtype, aux_logits, aux_bias, aux_p_mean, float(aux_scale),
          dz, W_dn, l, ws, ws_bytes, err_flag, stream)


def moe_router_aux_loss(logits, bias, T, E, p_mean, loss, ws, ws_bytes, stream=None):
    _call("moe_router_aux_loss", logits, bias, T, E, p_mean, loss, ws, ws_bytes, stream)


def moe_diag_wait_timeout(limit_ns, err_flag, waited_ns, stream=None):
    _call("moe_diag_wait_timeout", int(limit_ns), err_flag, waited_ns, stream)


def moe_timing_enable(on: bool):
    load().moe_timing_enable(1 if on else 0)


def moe_timing_report() -> dict:
    """{label: (launches, total_ms)} of the launches timed since the last report."""
    lib = load()
    n = lib.moe_timing_report(None, 0)
    buf = ctypes.create_string_buffer(n + 1)
    lib.moe_timing_report(buf, n + 1)
    out = {}
    for line in buf.value.decode().splitlines():
        name, cnt, ms = line.split()
        out[name] = (int(cnt), float(ms))
    return out


def moe_replica_plan(counts, E, P, pieces, n_pieces, rank_load, stream=None):
    _call("moe_replica_plan", counts, E, P, pieces, n_pieces, rank_load, stream)


def moe_expert_buckets(counts, E, expert_order, tile_sched_ordered, stream=None):
    _call("moe_expert_buckets", counts, E, expert_order, tile_sched_ordered, stream)


def moe_grouped_swiglu_ordered(z_perm, W13, W2, offsets, tile_sched_ordered, expert_order, row_w,
                               E, R, l, f, gu_save, h, y_perm, stream=None):
    _call("moe_grouped_swiglu_ordered", z_perm, W13, W2, offsets, tile_sched_ordered,
          expert_order, row_w, E, R, l, f, gu_save, h, y_perm, stream)
