"""moe_dispatch_noalloc: the dispatch for callers that cannot allocate.

Some callers cannot give this library device memory: a layer plugin inside an
inference engine only receives the layer's own tensors, and a serving loop
that fixed its memory plan at start-up must not call cudaMalloc later.  For
them moe_dispatch_noalloc keeps its scratch in a fixed device array inside the
library.  This test calls it through the C ABI and checks that it gives the
same offsets, row_experts, perm and gathered rows as moe_dispatch (which takes
a workspace), bit for bit as the dispatch tests require, on two calls in a
row, and that problems too large for the array are refused.

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


def test_noalloc_dispatch_matches_workspace_dispatch(cuda_lib):
    lib = cuda_lib.load()
    # two calls in a row, the second smaller than the first, so that the
    # scratch still holds the first call's larger contents
    for T, E, k, H, seed in [(16384, 64, 6, 256, 1), (1000, 8, 2, 64, 2)]:
        idx, x = _case(cuda_lib, T, E, k, H, seed)
        ref = cuda_lib.moe_dispatch(idx, E, x=x)
        got = _noalloc(lib, idx, E, x)
        torch.cuda.synchronize()
        assert torch.equal(got[0], ref.offsets)
        assert torch.equal(got[1], ref.row_experts)
        assert torch.equal(got[2], ref.perm)
        assert torch.equal(got[3].view(torch.int16), ref.x_disp.view(torch.int16))


def test_noalloc_dispatch_rejects_oversized_problems(cuda_lib):
    lib = cuda_lib.load()
    fake = ctypes.c_void_p(0x10000)  # never touched: the size check comes first
    st = lib.moe_dispatch_noalloc(fake, 70000, 1024, 2, None, BF16, 0, fake, fake, fake, None, None)
    assert st == 4  # MOE_ERR_UNSUPPORTED
    assert "use moe_dispatch with a workspace" in lib.moe_last_error().decode()
