"""Failure detection on the GPU without a fault.

Every wait on an mbarrier inside this library's kernels is bounded: when the
limit passes, the kernel records MOE_ERR_DEVICE_TIMEOUT in the workspace
status word and returns.  moe_selftest_bounded_wait runs that path on purpose
(a barrier nothing completes, a 50 ms limit); the host then reads the status
and the context keeps working.  Invalid expert indices reaching dispatch are
the other device-side condition; they are covered in test_gpu_dispatch.py."""
import ctypes

import pytest
import torch

from top_routing_grouped_fp32_gb300.inputs import make_inputs, small_workload

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_context_survives(cuda_lib):
    lib = cuda_lib.load()
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.moe_selftest_bounded_wait(ctypes.c_void_p(ws.data_ptr()), 50, stream)
    assert st == 0, lib.moe_last_error().decode()
    assert cuda_lib.moe_get_device_status(ws) == 7  # MOE_ERR_DEVICE_TIMEOUT
    assert "bounded wait" in lib.moe_last_error().decode()

    # the context is still usable: a full forward runs and reports OK
    wl = small_workload(256, 8, 2, 256, 256, dtype="bf16", seed=2)
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    fws = experts.forward_workspace(wl.T, wl.top_k, inp["logits"].dtype)
    y = experts.forward(inp["x"], inp["logits"], wl.top_k, wl.renormalize, workspace=fws)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all()
    assert cuda_lib.moe_get_device_status(fws) == 0


def test_selftest_argument_checks(cuda_lib):
    lib = cuda_lib.load()
    ws = torch.zeros(512, dtype=torch.uint8, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.moe_selftest_bounded_wait(None, 50, stream) == 1
    assert lib.moe_selftest_bounded_wait(ctypes.c_void_p(ws.data_ptr() + 16), 50, stream) == 1
    assert lib.moe_selftest_bounded_wait(ctypes.c_void_p(ws.data_ptr()), 0, stream) == 1
    assert lib.moe_selftest_bounded_wait(ctypes.c_void_p(ws.data_ptr()), 5000, stream) == 1
