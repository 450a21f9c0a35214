"""Pins of the oracle's FP8 cache of the GMM outputs (e4m3_round,
fp8_block_scale, fp8_block_quantize / dequantize and the cached backward)
against the E4M3 format's own definition, brute force over its 256 codes, a
library conversion where one exists, and invariants. CPU only."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from sparse_moe_layer_topk_gb300 import inputs as I


def _e4m3_grid():
    """Every finite E4M3 value from the bit fields: sign, 4 exponent bits (bias
    7), 3 mantissa bits; exponent 0 is subnormal (m 2^-9), exponent 15 with
    mantissa 7 is NaN. Returns the sorted non-negative values and, for each,
    the parity of its 7-bit magnitude code (exponent << 3 | mantissa)."""
    vals, codes = [], []
    for e in range(16):
        for m in range(8):
            if e == 15 and m == 7:
                continue
            v = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
            vals.append(v)
            codes.append((e << 3) | m)
    order = np.argsort(vals)
    return np.asarray(vals)[order], np.asarray(codes)[order]


def test_e4m3_grid_from_the_format():
    vals, _ = _e4m3_grid()
    assert len(vals) == 127 and vals[0] == 0.0
    assert vals[-1] == 448.0 and vals[1] == 2.0 ** -9
    assert np.all(np.diff(vals) > 0)
    np.testing.assert_array_equal(O.e4m3_round(vals), vals)
    np.testing.assert_array_equal(O.e4m3_round(-vals), -vals)


def test_e4m3_ties_to_even_and_saturation():
    vals, codes = _e4m3_grid()
    for i in range(len(vals) - 1):
        a, b = vals[i], vals[i + 1]
        mid = (a + b) / 2
        even = a if codes[i] % 2 == 0 else b
        assert O.e4m3_round(mid) == even, (a, b)
        assert O.e4m3_round(-mid) == -even
        assert O.e4m3_round(np.nextafter(mid, b)) == b
        assert O.e4m3_round(np.nextafter(mid, a)) == a
    for v in (448.5, 463.9, 464.0, 500.0, 1e30):
        assert O.e4m3_round(v) == 448.0 and O.e4m3_round(-v) == -448.0


def test_e4m3_matches_torch_float8_within_range():
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("no float8_e4m3fn in this PyTorch")
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.normal(0, s, 4000) for s in (1e-3, 0.05, 1.0, 30.0, 150.0)])
    x = np.clip(x, -448.0, 448.0).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.e4m3_round(x.astype(np.float64)), ref)


def test_block_scale_is_the_smallest_power_of_two():
    rng = np.random.default_rng(5)
    amaxes = np.concatenate([np.exp(rng.uniform(-60, 60, 2000)),
                             448.0 * 2.0 ** np.arange(-40, 41)])
    for a in amaxes:
        s = O.fp8_block_scale(a)
        m, _ = np.frexp(s)
        assert m == 0.5                        # a power of two
        assert a <= 448.0 * s and a > 224.0 * s, (a, s)
    assert O.fp8_block_scale(448.0) == 1.0 and O.fp8_block_scale(448.0 * 8) == 8.0
    assert O.fp8_block_scale(np.nextafter(448.0, 1e9)) == 2.0
    assert O.fp8_block_scale(0.0) == 1.0 and O.fp8_block_scale(2.0 ** -101) == 1.0


def test_block_quantize_round_trip():
    rng = np.random.default_rng(6)
    rows, cols = 40, 2 * O.FP8_BLOCK
    x = rng.normal(0, 1, (rows, cols)) * np.exp(rng.uniform(-8, 8, (rows, 1)))
    x[3, :O.FP8_BLOCK] = 0.0                   # an all-zero block
    q, sc = O.fp8_block_quantize(x)
    assert sc.shape == (rows, 2)
    assert np.all(np.abs(q) <= 448.0)
    np.testing.assert_array_equal(O.e4m3_round(q), q)   # q are E4M3 values
    for r in range(rows):
        for b in range(2):
            blk = q[r, b * O.FP8_BLOCK:(b + 1) * O.FP8_BLOCK]
            if r == 3 and b == 0:
                assert sc[r, b] == 1.0 and not blk.any()
            else:
                assert 224.0 <= np.max(np.abs(blk)) <= 448.0
    xd = O.fp8_block_dequantize(q, sc)
    scaled = np.abs(x) / np.repeat(sc, O.FP8_BLOCK, axis=1)
    err = np.abs(xd - x) / np.repeat(sc, O.FP8_BLOCK, axis=1)
    normal = scaled >= 2.0 ** -6
    # half a unit in the last place: 2^-4 relative (normals), 2^-10 absolute (subnormals)
    assert np.all(err[normal] <= scaled[normal] * 2.0 ** -4)
    assert np.all(err[~normal] <= 2.0 ** -10)


def test_backward_with_the_exact_cache_is_the_plain_backward():
    rng = np.random.default_rng(7)
    z = rng.normal(0, 1, (9, 32))
    W13 = rng.normal(0, 0.2, (32, 2 * 16))
    W2 = rng.normal(0, 0.2, (16, 32))
    d_o = rng.normal(0, 1, (9, 32))
    g, u = (z @ W13)[:, :16], (z @ W13)[:, 16:]
    plain = O.swiglu_expert_backward(z, W13, W2, d_o)
    cached = O.swiglu_expert_backward(z, W13, W2, d_o, (g, u))
    for a, b in zip(plain, cached):
        np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-13)


def test_layer_backward_fp8_cache_enters_only_the_swiglu_derivative():
    """The FP8 cache changes the routed experts' dz and dW13 by about the E4M3
    rounding (2^-4 at most, ~2 % rms per element) and leaves dW2, the routing
    weight gradient and the shared experts' gradients exactly as they are."""
    cfg = dataclasses.replace(I.CONFIGS[0], name="tiny_T256_E64_top4_f128", f=128)
    inp = I.make_layer_inputs(cfg)
    fwd = O.layer_forward(inp)
    exact = O.layer_backward(inp, fwd)
    fp8 = O.layer_backward(inp, fwd, fp8_cache=True)
    for name in ("dW2", "d_row_w", "dW13_sh", "dW2_sh", "dW_up", "dL"):
        np.testing.assert_array_equal(fp8[name], exact[name], err_msg=name)
    for name in ("dW13", "dz_perm"):
        rel = np.linalg.norm(fp8[name] - exact[name]) / np.linalg.norm(exact[name])
        assert 1e-3 < rel < 4e-2, (name, rel)
