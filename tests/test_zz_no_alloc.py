"""moe_dispatch_noalloc: the dispatch for callers that cannot allocate.

Some callers cannot give this library device memory: a layer plugin inside an
inference engine only receives the layer's own tensors, and a serving loop
that fixed its memory plan at start-up must not call cudaMalloc later.  For
them moe_dispatch_noalloc keeps its scratch in a fixed device array inside the
library.  This test calls it through the C ABI and checks that it gives the
same offsets, row_experts, perm and gathered rows as moe_dispatch (which takes
a workspace), bit for bit as the dispatch tests require, on calls in a row
of different shapes (one of them at the array's size limit, where the chunk
scan runs as its own kernel), with slots holding indices >= E, and that
problems too large for the array are refused.

The file is named so that pytest collects it last."""
import ctypes

import numpy as np
import pytest
import torch

from top_routing_grouped_fp32_gb300.inputs import make_routing_logits

pytestmark = pytest.mark.gpu

BF16 = 2


def _noalloc(lib, idx, E, x):
    T, k = idx.shape
    N = T * k
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    rows = torch.empty(N, dtype=torch.int32, device="cuda")
    perm = torch.empty(N, dtype=torch.int32, device="cuda")
    x_disp = torch.empty((N, x.shape[1]), dtype=x.dtype, device="cuda")
    st = lib.moe_dispatch_noalloc(
        ctypes.c_void_p(idx.data_ptr()), T, E, k, ctypes.c_void_p(x.data_ptr()), BF16, x.shape[1],
        ctypes.c_void_p(offsets.data_ptr()), ctypes.c_void_p(rows.data_ptr()),
        ctypes.c_void_p(perm.data_ptr()), ctypes.c_void_p(x_disp.data_ptr()),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.moe_last_error().decode()
    return offsets, rows, perm, x_disp


def _case(moe, T, E, k, H, seed):
    logits = make_routing_logits(T, E, "bf16", seed=seed, device="cuda")
    idx, _ = moe.moe_route(logits, k, True)
    x = torch.randn((T, H), generator=torch.Generator(device="cuda").manual_seed(seed),
                    device="cuda").to(torch.bfloat16)
    return idx, x


def _check_equal(got, ref):
    assert torch.equal(got[0], ref.offsets)
    assert torch.equal(got[1], ref.row_experts)
    assert torch.equal(got[2], ref.perm)
    # rows past offsets[E] (slots holding an index >= E) are not written
    nv = int(ref.offsets[-1].item())
    assert torch.equal(got[3][:nv].view(torch.int16), ref.x_disp[:nv].view(torch.int16))


def test_noalloc_dispatch_matches_workspace_dispatch(cuda_lib):
    lib = cuda_lib.load()
    # calls in a row with different shapes, so that the scratch still holds an
    # earlier call's contents.  (16384, 64, 6) and (1000, 8, 2) have small
    # chunk-histogram tables, which the scatter blocks scan themselves;
    # (65280, 1024, 2) is at the array's limit (255 chunks x 2049 words) and
    # takes the separate scan kernel, whose chunk bases fill the array's
    # second region.
    for T, E, k, H, seed in [(16384, 64, 6, 256, 1), (65280, 1024, 2, 64, 3), (1000, 8, 2, 64, 2)]:
        idx, x = _case(cuda_lib, T, E, k, H, seed)
        ref = cuda_lib.moe_dispatch(idx, E, x=x)
        got = _noalloc(lib, idx, E, x)
        torch.cuda.synchronize()
        _check_equal(got, ref)


def test_noalloc_dispatch_invalid_indices(cuda_lib):
    """Indices >= E are not dispatched: offsets[E] counts only the valid
    slots, and perm and row_experts end in 0xFFFFFFFF (-1 as int32)."""
    lib = cuda_lib.load()
    T, E, k, H = 700, 16, 3, 64
    g = np.random.default_rng(7)
    idx_h = np.stack([g.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    bad = g.choice(T * k, size=41, replace=False)
    idx_h.reshape(-1)[bad] = E + g.integers(0, 1000, size=bad.size)
    idx = torch.from_numpy(idx_h).cuda()
    x = torch.randn((T, H), generator=torch.Generator(device="cuda").manual_seed(5),
                    device="cuda").to(torch.bfloat16)
    for _ in range(2):
        ref = cuda_lib.moe_dispatch(idx, E, x=x)
        got = _noalloc(lib, idx, E, x)
        torch.cuda.synchronize()
        _check_equal(got, ref)
    flat = idx_h.reshape(-1)
    valid = np.flatnonzero(flat < E)
    nv = valid.size
    assert nv == T * k - bad.size
    offsets, rows, perm = (t.cpu().numpy() for t in got[:3])
    assert offsets[E] == nv
    # the valid slots as a stable sort by expert (the dispatch order)
    order = valid[np.argsort(flat[valid], kind="stable")]
    assert np.array_equal(perm[:nv], order)
    assert np.array_equal(rows[:nv], flat[order])
    assert np.all(perm[nv:] == -1) and np.all(rows[nv:] == -1)


def test_noalloc_dispatch_rejects_oversized_problems(cuda_lib):
    lib = cuda_lib.load()
    fake = ctypes.c_void_p(0x10000)  # never touched: the size check comes first
    st = lib.moe_dispatch_noalloc(fake, 70000, 1024, 2, None, BF16, 0, fake, fake, fake, None, None)
    assert st == 4  # MOE_ERR_UNSUPPORTED
    assert "use moe_dispatch with a workspace" in lib.moe_last_error().decode()
