"""The allocation-free permute (moe_permute_noalloc) against the regular one.

moe_permute_noalloc serves callers that cannot allocate device memory: it
keeps its scratch in a fixed array inside the library instead of a workspace
the caller passes. Its outputs must equal moe_permute's bit for bit (all of
them are integers or copied values), on consecutive calls that reuse the same
array with different sizes; and the maps of one call equal the oracle's
counting sort outright. This file sorts after every other test file, so a run
that stops at the first failure has run every other test first; it also
passes on its own in a fresh process, where its first call sets the array up."""
import numpy as np
import pytest
import torch

import oracle as O
from sparse_moe_layer_topk_gb300 import _lib as M
from sparse_moe_layer_topk_gb300 import inputs as I

from gpu_util import need_gpu

pytestmark = pytest.mark.gpu

NAMES = ("counts", "offsets", "slot_of", "token_of", "tile_sched", "row_w", "z_perm", "err")


def _buffers(T, E, k, l):
    R = T * k
    dev = "cuda"
    return dict(
        counts=torch.full((E,), -7, dtype=torch.int32, device=dev),
        offsets=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        slot_of=torch.full((T, k), -7, dtype=torch.int32, device=dev),
        token_of=torch.full((R,), -7, dtype=torch.int32, device=dev),
        tile_sched=torch.full((E + 1,), -7, dtype=torch.int32, device=dev),
        row_w=torch.full((R,), -7.0, dtype=torch.float32, device=dev),
        z_perm=torch.zeros(R, l, dtype=torch.bfloat16, device=dev),
        err=torch.zeros(1, dtype=torch.int32, device=dev),
    )


def _run_both(seed, T, E, k, l, skew, with_z=True):
    idx = I.make_topk_ids(seed, T, E, k, skew=skew).cuda()
    g = torch.Generator().manual_seed(seed)
    z = torch.randn(T, l, generator=g).to(torch.bfloat16).cuda() if with_z else None
    tw = torch.rand(T, k, generator=g).cuda()
    ref = _buffers(T, E, k, l)
    wsb = M.moe_workspace_size(M.MOE_OP_PERMUTE, T=T, E=E)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    M.moe_permute(z, idx, tw, T, l, E, k, ref["z_perm"], ref["counts"], ref["offsets"],
                  ref["slot_of"], ref["token_of"], ref["tile_sched"], ref["row_w"], ws, wsb,
                  ref["err"])
    got = _buffers(T, E, k, l)
    M.moe_permute_noalloc(z, idx, tw, T, l, E, k, got["z_perm"], got["counts"], got["offsets"],
                          got["slot_of"], got["token_of"], got["tile_sched"], got["row_w"],
                          got["err"])
    torch.cuda.synchronize()
    for n in NAMES:
        a, b = got[n].cpu(), ref[n].cpu()
        if a.dtype == torch.bfloat16:
            a, b = a.view(torch.int16), b.view(torch.int16)
        assert torch.equal(a, b), n
    assert int(got["err"].item()) == 0
    return idx.cpu().numpy(), got


def test_noalloc_permute_matches_workspace_permute_on_consecutive_calls():
    need_gpu()
    # two calls in a row on the shared array: the big case leaves stale
    # contents that the smaller, differently skewed case must not see
    _run_both(101, 4096, 896, 16, 256, 0.0)
    _run_both(102, 1000, 896, 16, 128, 1.1)
    idx, got = _run_both(103, 300, 64, 4, 64, 0.0)
    slot_of, token_of, offsets = O.permutation_maps(idx, 64)
    assert np.array_equal(got["slot_of"].cpu().numpy(), slot_of)
    assert np.array_equal(got["token_of"].cpu().numpy(), token_of)
    assert np.array_equal(got["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(got["tile_sched"].cpu().numpy(), O.m_tiles_schedule(np.diff(offsets)))


def test_noalloc_permute_at_its_largest_size_and_with_no_tokens():
    """The largest problem the fixed scratch holds (ceil(T / 256) * E equal to
    its 262144 ints: T = 65536, E = 1024), then an empty batch, whose counts,
    offsets and tile schedule must be all zero."""
    need_gpu()
    _run_both(104, 65536, 1024, 1, 64, 0.0, with_z=False)
    E = 64
    b = _buffers(0, E, 4, 64)
    M.moe_permute_noalloc(None, b["slot_of"], None, 0, 64, E, 4, None, b["counts"],
                          b["offsets"], b["slot_of"], b["token_of"], b["tile_sched"], None,
                          b["err"])
    torch.cuda.synchronize()
    for n in ("counts", "offsets", "tile_sched"):
        assert not b[n].cpu().any(), n
    assert int(b["err"].item()) == 0


def test_noalloc_permute_rejects_problems_beyond_its_scratch():
    need_gpu()
    # one chunk past the capacity (257 * 1024 > 262144), and far past it
    for T, E, k in ((65537, 1024, 1), (80000, 896, 1)):
        with pytest.raises(M.MoEError, match="workspace"):
            M.moe_permute_noalloc(None, 0x1000, None, T, 0, E, k, None, 0x1000, 0x1000, 0x1000,
                                  0x1000, 0x1000, None, None)
