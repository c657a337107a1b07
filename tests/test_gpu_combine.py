"""Combine parity: moe_combine against the oracle's weighted combine."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_y_close, oracle_dispatch_of, u32, values
from top_routing_grouped_fp32_gb300.inputs import TORCH_DTYPES

pytestmark = pytest.mark.gpu


def _case(moe, T, E, k, H, dtype, wdtype, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    logits = torch.randn((T, E), generator=g, device="cuda").to(TORCH_DTYPES[wdtype])
    idx, w = moe.moe_route(logits, k, True)
    d = moe.moe_dispatch(idx, E)
    eo = torch.randn((T * k, H), generator=g, device="cuda").to(TORCH_DTYPES[dtype])
    y = moe.moe_combine(eo, d.perm, w, k)
    torch.cuda.synchronize()
    _, o_perm, _ = oracle_dispatch_of(idx, E)
    assert np.array_equal(u32(d.perm), o_perm), "perm differs"
    ref = oracle.combine(values(eo), o_perm, values(w))
    return y, ref


@pytest.mark.parametrize("T,E,k,H,dtype,wdtype", [
    (300, 8, 2, 256, "bf16", "bf16"), (129, 16, 6, 2048, "bf16", "f32"), (50, 4, 4, 64, "f32", "f32"),
    (77, 5, 3, 60, "f16", "bf16"), (1, 1, 1, 8, "bf16", "f16"), (64, 64, 64, 24, "f32", "bf16"),
])
def test_combine_shapes(cuda_lib, T, E, k, H, dtype, wdtype):
    y, ref = _case(cuda_lib, T, E, k, H, dtype, wdtype, seed=T + H)
    # one rounding of an FP32 sum (relative 2^-9 for bf16, 2^-12 for f16, with a
    # factor 2 margin) plus the FP32 accumulation error, bounded in absolute
    # terms by 1e-5 of the largest output
    tol = {"bf16": 2 ** -8, "f16": 2 ** -11, "f32": 0.0}[dtype]
    got = values(y)
    assert np.all(np.abs(got - ref) <= tol * np.abs(ref) + 1e-5 * np.abs(ref).max())


def test_combine_nan_rows(cuda_lib):
    T, E, k, H = 20, 4, 2, 16
    logits = torch.randn((T, E), device="cuda").to(torch.bfloat16)
    logits[3, 1] = float("nan")
    logits[7] = float("-inf")
    idx, w = cuda_lib.moe_route(logits, k, True)
    d = cuda_lib.moe_dispatch(idx, E)
    eo = torch.randn((T * k, H), device="cuda").to(torch.bfloat16)
    y = cuda_lib.moe_combine(eo, d.perm, w, k)
    torch.cuda.synchronize()
    _, o_perm, _ = oracle_dispatch_of(idx, E)
    assert np.array_equal(u32(d.perm), o_perm), "perm differs"
    ref = oracle.combine(values(eo), o_perm, values(w))
    assert_y_close(y, ref, "bf16")
    assert torch.isnan(y[3]).all() and torch.isnan(y[7]).all()
    assert torch.isfinite(y[0]).all()


def test_combine_undispatched_slot_is_nan(cuda_lib):
    """A slot that no dispatched row holds (invalid index) makes its token NaN."""
    T, E, k, H = 10, 4, 2, 8
    idx_np = np.array([[0, 1]] * T, np.uint32)
    idx_np[4, 1] = 9
    d = cuda_lib.moe_dispatch(torch.from_numpy(idx_np.view(np.int32)).cuda(), E)
    w = torch.full((T, k), 0.5, dtype=torch.bfloat16, device="cuda")
    eo = torch.ones((T * k, H), dtype=torch.bfloat16, device="cuda")
    y = cuda_lib.moe_combine(eo, d.perm, w, k)
    torch.cuda.synchronize()
    assert torch.isnan(y[4]).all()
    assert torch.all(y[torch.arange(T, device="cuda") != 4] == 1.0)
