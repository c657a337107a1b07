"""Dispatch parity: moe_dispatch against the oracle's stable counting sort.

offsets, row_experts and perm bit-exact; x_disp rows byte-identical to the
token rows they copy; indices >= E reported through the device status."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import u32
from top_routing_grouped_fp32_gb300.inputs import TORCH_DTYPES, WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _check(moe, idx_np, E, x=None):
    idx = torch.from_numpy(idx_np.astype(np.uint32).view(np.int32)).cuda()
    d = moe.moe_dispatch(idx, E, x=x)
    status = moe.moe_get_device_status(d.workspace)
    o_off, o_rows, o_perm, bad = oracle.dispatch(idx_np, E)
    assert np.array_equal(u32(d.offsets), o_off), "offsets differ"
    assert np.array_equal(u32(d.perm), o_perm), "perm differs"
    assert np.array_equal(u32(d.row_experts), o_rows), "row_experts differ"
    assert status == (6 if bad else 0)
    if x is not None:
        n = int(o_off[-1])
        k = idx_np.shape[1]
        want = x[torch.from_numpy((o_perm[:n] // k).astype(np.int64)).cuda()]
        assert torch.equal(d.x_disp[:n].view(torch.int16) if x.dtype != torch.float32
                           else d.x_disp[:n].view(torch.int32),
                           want.view(torch.int16) if x.dtype != torch.float32 else want.view(torch.int32))
    return d


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_dispatch_workloads(cuda_lib, name):
    wl = WORKLOADS[name]
    inp = make_inputs(wl, device="cuda", weights=False)
    idx, _ = cuda_lib.moe_route(inp["logits"], wl.top_k, wl.renormalize)
    d = _check(cuda_lib, u32(idx).reshape(wl.T, wl.top_k), wl.E, x=inp["x"])
    # every token appears exactly k times
    cnt = np.bincount(u32(d.perm) // wl.top_k, minlength=wl.T)
    assert np.all(cnt == wl.top_k)


@pytest.mark.parametrize("T,E,k,H,dtype", [
    (1, 1, 1, 8, "bf16"), (255, 7, 3, 64, "bf16"), (257, 7, 3, 64, "f16"), (1000, 64, 6, 136, "bf16"),
    (300, 1024, 64, 16, "bf16"), (40, 50, 33, 24, "f32"), (513, 9, 2, 30, "bf16"), (100, 3, 3, 12, "f32"),
    # 15 chunks x 1025 histogram words: the scatter blocks scan the table themselves;
    # 16 chunks x 1025 words: over the limit, the one-block scan kernel runs
    (3840, 1024, 8, 16, "bf16"), (4000, 1024, 8, 16, "bf16"), (70000, 64, 2, 8, "bf16"),
])
def test_dispatch_shapes(cuda_lib, T, E, k, H, dtype):
    rng = np.random.default_rng(T + E + k)
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.uint32)
    x = torch.randn((T, H), generator=torch.Generator(device="cuda").manual_seed(T), device="cuda")
    _check(cuda_lib, idx, E, x=x.to(TORCH_DTYPES[dtype]))


def test_dispatch_repeated_experts_in_a_row(cuda_lib):
    """Indices from outside moe_route may repeat inside a row: order stays by slot."""
    rng = np.random.default_rng(1)
    for T, E, k in [(300, 5, 4), (70, 40, 40), (64, 64, 64)]:
        idx = rng.integers(0, E, size=(T, k)).astype(np.uint32)
        _check(cuda_lib, idx, E)


def test_dispatch_invalid_indices(cuda_lib):
    rng = np.random.default_rng(2)
    idx = rng.integers(0, 8, size=(600, 4)).astype(np.uint32)
    idx[5, 1] = 8
    idx[599, 3] = 0xFFFFFFFF
    idx[300, 0] = 1000
    x = torch.randn((600, 32), device="cuda").to(torch.bfloat16)
    d = _check(cuda_lib, idx, 8, x=x)
    perm = u32(d.perm)
    assert np.all(perm[-3:] == 0xFFFFFFFF)


def test_dispatch_empty_batch(cuda_lib):
    idx = torch.empty((0, 2), dtype=torch.int32, device="cuda")
    d = cuda_lib.moe_dispatch(idx, 4)
    assert u32(d.offsets).tolist() == [0, 0, 0, 0, 0]


def test_dispatch_is_deterministic(cuda_lib):
    wl = WORKLOADS["finegrained_bf16"]
    inp = make_inputs(wl, device="cuda", weights=False)
    idx, _ = cuda_lib.moe_route(inp["logits"], wl.top_k, wl.renormalize)
    a = cuda_lib.moe_dispatch(idx, wl.E, x=inp["x"])
    b = cuda_lib.moe_dispatch(idx, wl.E, x=inp["x"])
    torch.cuda.synchronize()
    for f in ("offsets", "perm", "row_experts"):
        assert torch.equal(getattr(a, f), getattr(b, f))
    assert torch.equal(a.x_disp.view(torch.int16), b.x_disp.view(torch.int16))
