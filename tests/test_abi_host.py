"""Host-side checks of the C ABI (no GPU needed): the library builds, loads
and exports every entry point include/moe.h declares; the binding covers them
with the right arity; argument errors are reported before any CUDA call."""
import os
import re

import pytest

from sparse_moe_layer_topk_gb300 import _lib as M
from sparse_moe_layer_topk_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declarations():
    """name -> (return type text, [argument texts]) of every moe_* prototype."""
    txt = open(os.path.join(ROOT, "include", "moe.h")).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    txt = re.sub(r"//[^\n]*", "", txt)
    decls = {}
    for m in re.finditer(r"^\s*((?:const\s+)?[\w\s\*]+?)\b(moe_\w+)\s*\(([^)]*)\)\s*;", txt, re.M):
        args = [a.strip() for a in m.group(3).split(",") if a.strip() and a.strip() != "void"]
        decls[m.group(2)] = (m.group(1).strip(), args)
    return decls


def _declared():
    return {name: len(args) for name, (_, args) in _declarations().items()}


def _ctype_of(c_text):
    """The ctypes type the binding must use for one C type (or argument) text."""
    if "*" in c_text:
        return M.ctypes.c_char_p if re.search(r"\bchar\s*\*", c_text) else M._P
    if "size_t" in c_text:
        return M._Z
    if re.search(r"\blong\s+long\b", c_text):
        return M.ctypes.c_longlong
    if re.search(r"\bfloat\b", c_text):
        return M._F
    if re.search(r"\bint\b", c_text):
        return M._I
    raise AssertionError(f"unmapped C type: {c_text}")


@pytest.fixture(scope="module")
def lib():
    B.build_library()
    return M.load()


def test_every_declared_symbol_is_exported_and_bound(lib):
    decls = _declared()
    assert len(decls) >= 18
    for name, nargs in decls.items():
        assert hasattr(lib, name), name
        assert name in M.SIGNATURES, name
        assert len(M.SIGNATURES[name][0]) == nargs, (name, nargs)


def test_binding_types_match_the_header():
    """Every argument and return type of the ctypes binding is the one the header
    declares (a pointer passed as an int, or a float as a pointer, would be
    marshalled wrongly without any error)."""
    for name, (ret, args) in _declarations().items():
        argtypes, restype = M.SIGNATURES[name]
        want = [_ctype_of(a) for a in args]
        assert list(argtypes) == want, (name, [t.__name__ for t in argtypes],
                                        [t.__name__ for t in want])
        assert restype == _ctype_of(ret), (name, ret)


def test_wrapper_parameters_follow_the_header_order():
    """Each Python wrapper names its parameters as the header does, in the same
    order, so two arguments of one C type cannot be swapped unnoticed (`in` is a
    Python keyword and becomes `inp`)."""
    import inspect
    # entry points the binding calls directly, or wraps with another interface
    unwrapped = {"moe_status_string", "moe_last_cuda_error", "moe_timing_report"}
    for name, (_, args) in _declarations().items():
        if name in unwrapped:
            continue
        header = [re.findall(r"(\w+)\s*$", a.replace("*", " "))[0] for a in args]
        header = ["inp" if h == "in" else h for h in header]
        params = list(inspect.signature(getattr(M, name)).parameters)
        assert params == header, (name, params, header)
        # and hands them to the library in that order
        passed = _call_args(getattr(M, name))
        if passed is not None:
            assert passed == [name] + params, (name, passed)


def _call_args(fn):
    """The arguments of the wrapper's `_call(...)` as names (the entry point's
    name as its string), or None when the wrapper does not use _call."""
    import ast
    import inspect
    import textwrap
    tree = ast.parse(textwrap.dedent(inspect.getsource(fn)))
    for node in ast.walk(tree):
        if isinstance(node, ast.Call) and getattr(node.func, "id", None) == "_call":
            out = []
            for a in node.args:
                if isinstance(a, ast.Call) and getattr(a.func, "id", None) in ("int", "float"):
                    a = a.args[0]  # a plain conversion of the argument
                out.append(a.value if isinstance(a, ast.Constant) else getattr(a, "id", None))
            return out
    return None


def test_status_strings_and_version(lib):
    assert lib.moe_version() >= 1
    for code in (M.MOE_OK, M.MOE_ERR_ARG, M.MOE_ERR_ALIGN, M.MOE_ERR_WORKSPACE,
                 M.MOE_ERR_UNSUPPORTED, M.MOE_ERR_CUDA):
        assert lib.moe_status_string(code)


def test_workspace_sizes(lib):
    assert M.moe_workspace_size(M.MOE_OP_ROUTE_TOPK, T=4096, E=896) >= 4096 * 896 * 4
    assert M.moe_workspace_size(M.MOE_OP_PERMUTE, T=4096, E=896) >= 16 * 896 * 4
    # the SwiGLU-backward row partials need at least one slot per row even for f < 128
    assert M.moe_workspace_size(M.MOE_OP_GROUPED_SWIGLU_BWD, T=100, k=1, f=64) >= \
        100 * (2 * 64 * 2 + 64 * 2 + 4)
    assert M.moe_workspace_size(M.MOE_OP_ROUTE_TOPK_BWD, T=10, E=64) >= 10 * 64 * 2
    assert M.moe_workspace_size(M.MOE_OP_ROUTER_AUX, T=4096, E=896) >= 256 * 896 * 4


def test_argument_errors_before_any_cuda_call(lib):
    P = 0x1000
    # null pointers
    assert lib.moe_latent_proj(None, None, 4, 64, 64, None, None) == M.MOE_ERR_ARG
    # dimension not a multiple of 64
    assert lib.moe_latent_proj(P, P, 4, 64, 96, P, None) == M.MOE_ERR_ALIGN
    # misaligned pointer
    assert lib.moe_latent_proj(P + 2, P, 4, 64, 64, P, None) == M.MOE_ERR_ALIGN
    # k out of range, E too large
    assert lib.moe_topk_from_logits(P, None, 4, 64, 33, P, P, P, None, None) == M.MOE_ERR_ARG
    assert lib.moe_topk_from_logits(P, None, 4, 2048, 4, P, P, P, None, None) == M.MOE_ERR_ARG
    # workspace too small
    assert lib.moe_route_topk(P, P, None, 64, 64, 64, 4, P, P, P, P, 16, None, None) == \
        M.MOE_ERR_WORKSPACE
    assert lib.moe_permute(None, P, None, 64, 64, 64, 4, None, P, P, P, P, P, None, P, 8, None,
                           None) == M.MOE_ERR_WORKSPACE
    # backward without the saved gate/up activations is not supported
    assert lib.moe_grouped_swiglu_bwd(P, P, P, P, None, P, P, P, P, 8, 64, 64, 64, P, P, P, P, 0,
                                      P, 1 << 30, None) == M.MOE_ERR_UNSUPPORTED
    # bad wgrad dtype
    assert lib.moe_latent_proj_bwd(P, P, P, 4, 64, 64, None, P, 7, None) == M.MOE_ERR_ARG
    # the fused input gradient of the router backward: latent width not a
    # multiple of 64, or no W_dn, is refused before anything is enqueued
    assert lib.moe_route_topk_bwd(P, P, P, P, P, P, P, 64, 64, 64, 4, None, P, None, 0, None, None,
                                  None, 0.0, P, P, 96, P, 1 << 30, None, None) == M.MOE_ERR_ALIGN
    assert lib.moe_route_topk_bwd(P, P, P, P, P, P, P, 64, 64, 64, 4, None, P, None, 0, None, None,
                                  None, 0.0, P, None, 128, P, 1 << 30, None, None) == M.MOE_ERR_ARG
    # the weight-gradient half of the projection backward is checked before the
    # input-gradient GEMM is enqueued
    assert lib.moe_latent_proj_bwd(P, None, P, 4, 64, 64, P, P, 0, None) == M.MOE_ERR_ARG
    # an auxiliary-loss gradient needs the batch's mean routing distribution
    assert lib.moe_route_topk_bwd(P, P, P, P, P, P, P, 64, 64, 64, 4, None, None, None, 0, P, None,
                                  None, 1.0, None, None, 0, P, 1 << 30, None, None) == M.MOE_ERR_ARG


def test_zero_tokens_enqueue_nothing(lib):
    """With T = 0 the forward calls and the row-movement backward calls return
    MOE_OK before any CUDA call (this host has no GPU, so any call would fail)."""
    P = 0x1000
    assert lib.moe_router_logits(P, P, 0, 64, 64, P, None) == M.MOE_OK
    assert lib.moe_topk_from_logits(P, None, 0, 64, 4, P, P, P, None, None) == M.MOE_OK
    assert lib.moe_route_topk(P, P, None, 0, 64, 64, 4, P, P, P, P, 256, None, None) == M.MOE_OK
    assert lib.moe_latent_proj(P, P, 0, 64, 64, P, None) == M.MOE_OK
    assert lib.moe_latent_proj_bwd(P, P, P, 0, 64, 64, P, None, 0, None) == M.MOE_OK
    assert lib.moe_grouped_swiglu(P, P, P, P, P, P, 4, 0, 64, 64, P, P, P, None) == M.MOE_OK
    assert lib.moe_shared_swiglu(P, P, P, 0, 64, 64, 1, P, P, P, None) == M.MOE_OK
    assert lib.moe_unpermute_combine(P, P, None, 0, 4, 64, P, None) == M.MOE_OK
    assert lib.moe_unpermute_combine_bwd(P, P, 0, 4, 64, P, None) == M.MOE_OK
    assert lib.moe_permute_bwd(P, P, None, 0, 4, 64, P, None) == M.MOE_OK


@pytest.mark.parametrize("T", [256, 1024, 2048, 4096, 16384, 65536])
@pytest.mark.parametrize("l,f,S", [(1024, 512, 2), (256, 64, 1), (512, 256, 3)])
def test_bench_split_k_rule_matches_the_library(lib, T, l, f, S):
    """bench.py restates the library's K-slice rule for the shared experts' weight
    gradients (to count the split-K reduction's bytes); the library's workspace size
    for the shared-expert backward (dgu plus the larger of the two gradients' fp32
    slices) must agree with it."""
    import bench

    cfg = type("Cfg", (), {"S": S, "f": f, "l": l})
    up256 = lambda b: (b + 255) // 256 * 256  # noqa: E731
    slices = max((m * n * 4 * s if s > 1 else 0) for m, n, s in bench.splitk_shapes(cfg, T))
    want = up256(T * S * f * 2 * 2) + up256(slices)
    assert M.moe_workspace_size(M.MOE_OP_SHARED_SWIGLU_BWD, T=T, l=l, f=f, S=S) == want
