"""Routing parity: moe_route against the FP64 oracle.

Indices bit-exact; FP32 weights within 1e-6 relative of the oracle's pre-cast
weights; stored weights equal to the FP32 weights rounded to nearest-even in
the logits dtype; NaN rows where the contract puts them."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_cast_is_rne, assert_weights_match, oracle_route, u32
from top_routing_grouped_fp32_gb300.inputs import (TORCH_DTYPES, WORKLOADS, make_inputs,
                                                   make_routing_logits)

pytestmark = pytest.mark.gpu


def _check(moe, logits, k, renorm):
    idx, w, w32 = moe.moe_route(logits, k, renorm, weights_f32=True)
    torch.cuda.synchronize()
    o_idx, o_pre, _ = oracle_route(logits, k, renorm)
    got = u32(idx)
    if not np.array_equal(got, o_idx):
        bad = np.argwhere((got != o_idx).any(1)).ravel()[:5]
        raise AssertionError(f"indices differ in rows {bad.tolist()}: gpu {got[bad].tolist()} "
                             f"oracle {o_idx[bad].tolist()}")
    assert_weights_match(w32, o_pre)
    assert_cast_is_rne(w, w32)
    return got, w32


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_route_workloads(cuda_lib, name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, device="cuda", weights=False)
    got, w32 = _check(cuda_lib, inp["logits"], wl.top_k, wl.renormalize)
    if wl.forced_ties:
        # the eight tied rows of the tiny workload, by the tie rule
        assert got[:8].tolist() == [[0, 1], [1, 2], [0, 1], [0, 1], [0, 2], [3, 1], [0, 1], [0, 3]]
    if wl.poison_frac:
        rows = inp["meta"]["poison"]["rows"]
        assert np.all(got[rows] == np.arange(wl.top_k))
        assert torch.isnan(w32[rows]).all()
        ctrl = inp["meta"]["poison"]["control"]
        assert torch.isfinite(w32[ctrl]).all()


@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("T,E,k", [(1, 1, 1), (33, 37, 5), (257, 100, 33), (64, 1024, 64),
                                   (16, 64, 64), (500, 256, 8), (7, 2, 2), (130, 160, 3),
                                   # every lanes-per-row / values-per-lane form, T not a
                                   # multiple of the rows per block
                                   (77, 8, 8), (99, 16, 16), (101, 30, 7), (45, 512, 20),
                                   (33, 128, 64)])
@pytest.mark.parametrize("renorm", [False, True])
def test_route_shapes_and_dtypes(cuda_lib, dtype, T, E, k, renorm):
    logits = make_routing_logits(T, E, dtype, seed=T * 7 + E, device="cuda")
    _check(cuda_lib, logits, k, renorm)


def test_route_ties_at_scale(cuda_lib):
    """Logits from a tiny value set: most rows have many exact ties."""
    g = torch.Generator(device="cuda").manual_seed(5)
    vals = torch.tensor([-1.0, 0.0, 0.0, 0.5, 2.0], device="cuda")
    for E, k in [(64, 6), (256, 8), (37, 4)]:
        pick = torch.randint(0, 5, (300, E), generator=g, device="cuda")
        logits = vals[pick].to(torch.bfloat16).contiguous()
        logits[::7, ::3] = -0.0
        _check(cuda_lib, logits, k, True)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_route_every_16bit_logit(cuda_lib, dtype):
    """Every 16-bit pattern except NaN and +inf once, 64 to a row and all 64 selected:
    the indices give the full selection order (subnormals, -0 against +0, -inf,
    saturated weights) against the oracle's."""
    bits = torch.from_numpy(np.random.default_rng(11).permutation(65536).astype(np.int16))
    logits = bits.view(TORCH_DTYPES[dtype]).clone()
    logits[torch.isnan(logits) | (logits == float("inf"))] = 0.0
    _check(cuda_lib, logits.view(1024, 64).cuda(), 64, False)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_route_minus_inf_picks_and_padding(cuda_lib, dtype):
    """E = 37 leaves padding entries in the last lane of a row; rows with fewer finite
    logits than k must pick real -inf experts, lowest id first, never padding."""
    g = torch.Generator(device="cuda").manual_seed(13)
    logits = torch.full((64, 37), float("-inf"), device="cuda")
    for r in range(64):
        n = r % 5  # 0..4 finite logits, k = 8
        cols = torch.randperm(37, generator=g, device="cuda")[:n]
        logits[r, cols] = torch.randn(n, generator=g, device="cuda")
    logits[0, 36] = 1.0  # keep row 0 from being all -inf (that row is poisoned)
    got, _ = _check(cuda_lib, logits.to(TORCH_DTYPES[dtype]), 8, True)
    assert (got < 37).all()


def test_route_nan_rule(cuda_lib):
    rows = [
        [0.0, float("nan"), 1.0, 2.0, -1.0],
        [0.0, float("inf"), 1.0, 2.0, -1.0],
        [float("-inf")] * 5,
        [float("-inf"), 1.0, float("-inf"), 0.0, float("-inf")],
        [0.1, 0.2, 0.3, 0.4, 0.5],
    ]
    for dt in ("f32", "bf16", "f16"):
        logits = torch.tensor(rows, dtype=TORCH_DTYPES[dt], device="cuda")
        got, w32 = _check(cuda_lib, logits, 3, True)
        assert np.all(got[:3] == [0, 1, 2]) and torch.isnan(w32[:3]).all()
        assert got[3].tolist() == [1, 3, 0]
        assert w32[3, 2].item() == 0.0


def test_route_misaligned_logits(cuda_lib):
    """Rows that do not start on a vector boundary take the scalar load path."""
    base = make_routing_logits(300 * 64 + 1, 1, "bf16", seed=9, device="cuda").view(-1)
    logits = base[1:].view(300, 64)
    assert logits.data_ptr() % 4 != 0
    _check(cuda_lib, logits, 6, False)


def test_route_empty_batch(cuda_lib):
    logits = torch.empty((0, 8), dtype=torch.bfloat16, device="cuda")
    idx, w = cuda_lib.moe_route(logits, 2, True)
    assert idx.shape == (0, 2) and w.shape == (0, 2)


def test_route_k1_renorm_is_one(cuda_lib):
    logits = make_routing_logits(100, 16, "f32", seed=3, device="cuda")
    idx, w, w32 = cuda_lib.moe_route(logits, 1, True, weights_f32=True)
    assert torch.all(w32 == 1.0)


def test_route_invalid_arguments_raise(cuda_lib):
    logits = make_routing_logits(4, 8, "bf16", seed=1, device="cuda")
    with pytest.raises(cuda_lib.MoeError, match="INVALID_ARG"):
        cuda_lib.moe_route(logits, 9, True)
    with pytest.raises(cuda_lib.MoeError, match="DTYPE"):
        cuda_lib.moe_route(logits.double(), 2, True)
