"""The pipelined host-buffer forward (moe_host_pipeline_*) gives, batch by
batch, bitwise the results of moe_forward on the same inputs, whatever the
batch sizes, the pipeline depth and the order in which slots are reused."""
import pytest
import torch

from top_routing_grouped_fp32_gb300.inputs import make_inputs, small_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("depth", [2, 3])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_pipeline_matches_device_forward(cuda_lib, depth, dtype):
    T_max, E, k, H, I = 600, 8, 2, 128, 192
    batches = [600, 577, 1, 600, 320, 599, 64]
    wl = small_workload(T_max, E, k, H, I, dtype=dtype, seed=41)
    base = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(base["gate"], base["up"], base["down"])
    pipe = experts.host_pipeline(T_max, k, True, logits_dtype=base["logits"].dtype, depth=depth)
    ins, outs, refs = [], [], []
    for i, T in enumerate(batches):
        b = make_inputs(small_workload(T, E, k, H, I, dtype=dtype, seed=100 + i), device="cuda")
        xh, lh = b["x"].cpu().pin_memory(), b["logits"].cpu().pin_memory()
        yh = torch.full((T, H), float("nan"), dtype=b["x"].dtype).pin_memory()
        ins.append((xh, lh))
        outs.append(yh)
        refs.append(experts.forward(b["x"], b["logits"], k, True))
        pipe.submit(xh, lh, yh)
    pipe.sync()
    torch.cuda.synchronize()
    for T, yh, ref in zip(batches, outs, refs):
        assert torch.equal(yh.view(torch.int16 if yh.dtype != torch.float32 else torch.int32),
                           ref.cpu().view(torch.int16 if ref.dtype != torch.float32 else torch.int32)), T
    pipe.close()


def test_pipeline_rejects_oversize_batches(cuda_lib):
    wl = small_workload(64, 4, 2, 64, 64, dtype="bf16", seed=2)
    b = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(b["gate"], b["up"], b["down"])
    pipe = experts.host_pipeline(32, 2, True, logits_dtype=b["logits"].dtype)
    xh, lh = b["x"].cpu().pin_memory(), b["logits"].cpu().pin_memory()
    yh = torch.empty((64, 64), dtype=torch.bfloat16).pin_memory()
    with pytest.raises(RuntimeError, match="SHAPE"):
        pipe.submit(xh, lh, yh)
    with pytest.raises(RuntimeError, match="INVALID_ARG"):
        experts.host_pipeline(32, 2, True, logits_dtype=b["logits"].dtype, depth=5)
    pipe.close()
