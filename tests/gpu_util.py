"""Helpers of the GPU parity tests: library loading, tolerance checks."""
import numpy as np
import pytest
import torch

from sparse_moe_layer_topk_gb300 import _lib as M
from sparse_moe_layer_topk_gb300 import build as B

# Stated tolerances of the layer for bf16 I/O with fp32 accumulation (max-abs,
# relative Frobenius)
MAX_ABS = 2e-2
REL_FRO = 1e-2


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    B.build_library()
    M.load()


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def check_close(name, got, ref, max_abs=MAX_ABS, rel_fro=REL_FRO, scale_by_max=False):
    """max|got-ref| <= max_abs (after dividing by max|ref| when scale_by_max)
    and ||got-ref||_F <= rel_fro * ||ref||_F."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref)
    mx = err.max() if err.size else 0.0
    if scale_by_max:
        mref = np.abs(ref).max() if ref.size else 0.0
        mx = mx / mref if mref > 0 else mx
    fro_ref = np.linalg.norm(ref)
    fro = np.linalg.norm(got - ref) / fro_ref if fro_ref > 0 else np.linalg.norm(got - ref)
    assert mx <= max_abs and fro <= rel_fro, f"{name}: max_err={mx:.3e} rel_fro={fro:.3e}"
    return mx, fro


def check_close_chunked(name, got, ref, chunk=32, max_abs=MAX_ABS, rel_fro=REL_FRO,
                        scale_by_max=False):
    """check_close of a large tensor `got` (torch, any device) against `ref`
    (numpy fp64): the same two criteria, accumulated over slices of axis 0 so
    that no full-size fp64 temporary is made."""
    ref = np.asarray(ref)
    assert tuple(got.shape) == ref.shape, (name, tuple(got.shape), ref.shape)
    mx = se = sr = mref = 0.0
    for i in range(0, ref.shape[0], chunk):
        g = f64(got[i:i + chunk])
        r = np.asarray(ref[i:i + chunk], dtype=np.float64)
        assert np.all(np.isfinite(g)), f"{name}: non-finite values"
        d = np.abs(g - r)
        if d.size:
            mx = max(mx, float(d.max()))
            mref = max(mref, float(np.abs(r).max()))
        se += float(np.sum(d * d))
        sr += float(np.sum(r * r))
    if scale_by_max and mref > 0:
        mx /= mref
    fro = np.sqrt(se / sr) if sr > 0 else np.sqrt(se)
    assert mx <= max_abs and fro <= rel_fro, f"{name}: max_err={mx:.3e} rel_fro={fro:.3e}"
    return mx, fro


def dev(t, dtype=None):
    t = t if dtype is None else t.to(dtype)
    return t.contiguous().cuda()
