"""Sigmoid group-limited routing (user guide section 10) against the oracle.

Indices bit-exact (the FP32 selection uses the correctly rounded FP32
sigmoid on both sides), FP32 weights within 1e-6 relative of the oracle's
FP64 weights, stored weights = RNE(FP32 weights), NaN rows; and the fused
forward with this router against the oracle's staged chain."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DT, assert_cast_is_rne, assert_weights_match, assert_y_close, stored, u32, values
from top_routing_grouped_fp32_gb300.inputs import make_inputs, make_routing_logits, small_workload

pytestmark = pytest.mark.gpu


def _check(moe, logits, k, groups, sel, top_two, renorm, scale, bias=None):
    idx, w, w32 = moe.moe_route_sigmoid_grouped(logits, k, groups, sel, top_two, renorm, scale,
                                                bias=bias, weights_f32=True)
    torch.cuda.synchronize()
    o_idx, o_pre, _ = oracle.route_sigmoid_grouped(
        stored(logits), DT[logits.dtype], k, groups, sel, top_two, renorm, scale,
        None if bias is None else bias.cpu().numpy())
    got = u32(idx)
    if not np.array_equal(got, o_idx):
        bad = np.argwhere((got != o_idx).any(1)).ravel()[:5]
        raise AssertionError(f"rows {bad.tolist()}: gpu {got[bad].tolist()} oracle {o_idx[bad].tolist()}")
    assert_weights_match(w32, o_pre)
    assert_cast_is_rne(w, w32)
    return got


@pytest.mark.parametrize("dtype", ["bf16", "f32", "f16"])
@pytest.mark.parametrize("T,E,k,groups,sel,top_two,renorm,scale,with_bias", [
    (2048, 256, 8, 8, 4, True, True, 2.5, True),      # group-limited, top-two, bias, scale
    (1000, 64, 6, 1, 1, False, False, 1.0, False),    # one group: plain sigmoid top-k
    (777, 128, 8, 16, 3, False, True, 1.0, True),     # max group score
    (300, 1024, 64, 128, 32, True, True, 0.5, True),  # limits: 128 groups, k=64
    (50, 12, 3, 3, 3, True, False, 1.0, True),       # all groups kept
    (33, 2, 1, 1, 1, False, True, 1.0, False),
])
def test_sigmoid_routing_matches_oracle(cuda_lib, dtype, T, E, k, groups, sel, top_two, renorm,
                                        scale, with_bias):
    logits = make_routing_logits(T, E, dtype, seed=T + E, device="cuda")
    bias = None
    if with_bias:
        g = torch.Generator(device="cuda").manual_seed(E)
        bias = (torch.randn(E, generator=g, device="cuda") * 0.1).float()
    _check(cuda_lib, logits, k, groups, sel, top_two, renorm, scale, bias)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_sigmoid_routing_every_16bit_logit(cuda_lib, dtype):
    """Every non-NaN 16-bit logit pattern once, 64 to a row and all 64 selected: the
    scores are ranked exactly as the oracle ranks its FP64 sigmoid rounded to FP32
    (saturated values near 0 and 1 tie in FP32 and fall back to the lower id)."""
    bits = torch.from_numpy(np.random.default_rng(7).permutation(65536).astype(np.int16))
    logits = bits.view(torch.bfloat16 if dtype == "bf16" else torch.float16).clone()
    logits[torch.isnan(logits)] = 0.0
    _check(cuda_lib, logits.view(1024, 64).cuda(), 64, 1, 1, False, False, 1.0)


def test_sigmoid_routing_ties_and_nan(cuda_lib):
    vals = torch.tensor([-1.0, 0.0, 0.0, 0.5, 2.0], device="cuda")
    g = torch.Generator(device="cuda").manual_seed(3)
    logits = vals[torch.randint(0, 5, (400, 64), generator=g, device="cuda")].to(torch.bfloat16)
    logits[5, 7] = float("nan")
    logits[9, :] = float("-inf")   # sigmoid 0: a finite row
    logits[11, 3] = float("inf")   # sigmoid 1: a finite row
    bias = torch.zeros(64, dtype=torch.float32, device="cuda")
    bias[::9] = 0.25
    got = _check(cuda_lib, logits, 4, 8, 2, True, True, 1.0, bias)
    assert got[5].tolist() == [0, 1, 2, 3]


@pytest.mark.parametrize("dtype,renorm", [("bf16", True), ("f32", False)])
def test_fused_forward_sigmoid_grouped(cuda_lib, dtype, renorm):
    wl = small_workload(600, 16, 4, 256, 384 if dtype == "bf16" else 40, dtype=dtype,
                        renormalize=renorm, seed=31)
    if dtype == "f32":
        wl = small_workload(200, 16, 4, 64, 40, dtype="f32", renormalize=renorm, seed=31)
    inp = make_inputs(wl, device="cuda")
    bias = (torch.randn(wl.E, generator=torch.Generator(device="cuda").manual_seed(2), device="cuda")
            * 0.2).float()
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    y = experts.forward_sigmoid_grouped(inp["x"], inp["logits"], wl.top_k, 4, 2, True, renorm, 1.5,
                                        bias=bias)
    torch.cuda.synchronize()
    # oracle: staged chain on the oracle's own routing
    idx, _, w_cast = oracle.route_sigmoid_grouped(stored(inp["logits"]), dtype, wl.top_k, 4, 2, True,
                                                  renorm, 1.5, bias.cpu().numpy())
    off, _, perm, _ = oracle.dispatch(idx, wl.E)
    xd = values(inp["x"])[perm // wl.top_k]
    eo = oracle.experts(xd, off, stored(inp["gate"]), stored(inp["up"]), stored(inp["down"]), dtype)
    ref = oracle.combine(eo, perm, w_cast)
    assert_y_close(y, ref, dtype)
