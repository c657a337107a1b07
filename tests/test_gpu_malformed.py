"""Malformed inputs to the staged calls: the kernels' own checks turn them
into a status code or a defined result, never into an access outside the
buffers.

* moe_experts_forward / moe_experts_backward with offsets that run backwards
  or past N: the call clamps them on the device and reports
  MOE_ERR_INVALID_INDEX in the workspace status word; the context stays
  usable and a following call with good offsets gives the oracle's result.
* moe_combine_backward with perm entries at or past T*k: those rows hold no
  slot (dexpert = 0) and the slots they would have held stay NaN."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_y_close, stored, values
from top_routing_grouped_fp32_gb300.inputs import make_inputs, small_workload

pytestmark = pytest.mark.gpu

INVALID_INDEX = 6


def _experts(cuda_lib, E, H, I, seed):
    wl = small_workload(64, E, 1, H, I, dtype="bf16", seed=seed)
    inp = make_inputs(wl, device="cuda")
    return cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"]), inp


BAD_OFFSETS = [
    [0, 50, 30, 120, 200],     # runs backwards
    [0, 60, 120, 180, 900],    # past N
    [10, 5, 900, 3, 1],        # both
]


@pytest.mark.parametrize("bad", BAD_OFFSETS)
def test_experts_forward_malformed_offsets(cuda_lib, bad):
    E, H, I, N = 4, 256, 384, 240
    ex, inp = _experts(cuda_lib, E, H, I, seed=71)
    g = torch.Generator(device="cuda").manual_seed(72)
    x_disp = torch.randn((N, H), generator=g, device="cuda").to(torch.bfloat16)
    ws = torch.empty(ex._lib.moe_experts_workspace_size(ex.handle, N), dtype=torch.uint8, device="cuda")
    off_bad = torch.tensor(bad, dtype=torch.int32, device="cuda")
    ex.forward_dispatched(x_disp, off_bad, workspace=ws)
    assert cuda_lib.moe_get_device_status(ws) == INVALID_INDEX
    # the same workspace and context, good offsets: status clears, result matches the oracle
    off = np.array([0, 60, 120, 180, 240], dtype=np.uint32)
    out = ex.forward_dispatched(x_disp, torch.from_numpy(off.view(np.int32)).cuda(), workspace=ws)
    assert cuda_lib.moe_get_device_status(ws) == 0
    ref = oracle.experts(values(x_disp), off, stored(inp["gate"]), stored(inp["up"]), stored(inp["down"]),
                         "bf16")
    assert_y_close(out, ref, "bf16")


@pytest.mark.parametrize("strategy", ["scalar", "tensor_core"])
@pytest.mark.parametrize("bad", BAD_OFFSETS)
def test_experts_backward_malformed_offsets(cuda_lib, bad, strategy):
    E, H, I, N = 4, 256, 384, 240
    ex, inp = _experts(cuda_lib, E, H, I, seed=73)
    g = torch.Generator(device="cuda").manual_seed(74)
    x_disp = torch.randn((N, H), generator=g, device="cuda").to(torch.bfloat16)
    dout = torch.randn((N, H), generator=g, device="cuda").to(torch.bfloat16)
    ws = torch.empty(ex._lib.moe_experts_backward_workspace_size(ex.handle, N), dtype=torch.uint8,
                     device="cuda")
    off_bad = torch.tensor(bad, dtype=torch.int32, device="cuda")
    ex.backward(x_disp, off_bad, dout, workspace=ws, strategy=strategy)
    assert cuda_lib.moe_get_device_status(ws) == INVALID_INDEX
    off = np.array([0, 60, 120, 180, 240], dtype=np.uint32)
    dinput, dgate, _, _ = ex.backward(x_disp, torch.from_numpy(off.view(np.int32)).cuda(), dout,
                                      workspace=ws, strategy=strategy)
    assert cuda_lib.moe_get_device_status(ws) == 0
    ref = oracle.experts_backward(values(x_disp), off, stored(inp["gate"]), stored(inp["up"]),
                                  stored(inp["down"]), "bf16", values(dout))
    assert_y_close(dinput, ref[0], "bf16", "dinput")
    got, r = values(dgate), ref[1]
    assert np.max(np.abs(got - r)) <= 2e-2 * np.max(np.abs(r))


def test_combine_backward_perm_past_the_slots(cuda_lib):
    T, k, H = 50, 2, 64
    g = torch.Generator(device="cuda").manual_seed(75)
    eo = torch.randn((T * k, H), generator=g, device="cuda").to(torch.bfloat16)
    dy = torch.randn((T, H), generator=g, device="cuda").to(torch.bfloat16)
    w = torch.rand((T, k), generator=g, device="cuda").to(torch.bfloat16)
    perm = np.arange(T * k, dtype=np.uint32)
    bad_rows = [3, 40, 99]
    perm[bad_rows] = [T * k, T * k + 7, 0xFFFFFFF0]  # past the T*k slots
    dex, dw = cuda_lib.moe_combine_backward(eo, torch.from_numpy(perm.view(np.int32)).cuda(), w, dy, k)
    torch.cuda.synchronize()
    r_dex, r_dw = oracle.combine_backward(values(eo), np.where(perm < T * k, perm, 0xFFFFFFFF).astype(np.uint32),
                                          values(w), values(dy))
    assert torch.all(dex[bad_rows] == 0)
    assert_y_close(dex, r_dex, "bf16", "dexpert")
    got = values(dw)
    assert np.array_equal(np.isnan(got), np.isnan(r_dw))
    assert np.isnan(got.ravel()[bad_rows]).all()  # slots 3, 40 and 99 are held by no row
    ok = ~np.isnan(r_dw)
    assert np.max(np.abs(got[ok] - r_dw[ok])) <= 1e-5 * np.max(np.abs(r_dw[ok]))
