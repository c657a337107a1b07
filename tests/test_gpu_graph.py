"""Stream capture: the fused forward and the expert backward (both
strategies) recorded into a CUDA graph and replayed give bitwise the results
of the same calls made eagerly (the header's capturability claim)."""
import pytest
import torch

from top_routing_grouped_fp32_gb300.inputs import TORCH_DTYPES, make_inputs, small_workload

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


@pytest.mark.parametrize("T,E,k,H,I", [(600, 8, 2, 256, 384), (2000, 4, 2, 128, 192)])
def test_forward_graph_replay(cuda_lib, T, E, k, H, I):
    wl = small_workload(T, E, k, H, I, dtype="bf16", seed=T)
    inp = make_inputs(wl, device="cuda")
    ex = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    ws = ex.forward_workspace(T, k, inp["logits"].dtype)
    y_eager = ex.forward(inp["x"], inp["logits"], k, True, workspace=ws).clone()
    y = torch.empty_like(y_eager)
    ex.forward(inp["x"], inp["logits"], k, True, y=y, workspace=ws)  # warm-up before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ex.forward(inp["x"], inp["logits"], k, True, y=y, workspace=ws)
    y.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(y), _bits(y_eager))
    # new inputs copied into the captured buffers: the replay follows them
    x2 = torch.randn_like(inp["x"], dtype=torch.float32).to(inp["x"].dtype)
    ref = ex.forward(x2, inp["logits"], k, True)
    inp["x"].copy_(x2)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(_bits(y), _bits(ref))


@pytest.mark.parametrize("strategy", ["scalar", "tensor_core"])
def test_expert_backward_graph_replay(cuda_lib, strategy):
    T, E, k, H, I = 1500, 4, 2, 320, 704
    wl = small_workload(T, E, k, H, I, dtype="bf16", seed=3)
    inp = make_inputs(wl, device="cuda")
    ex = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    idx, _ = cuda_lib.moe_route(inp["logits"], k, True)
    d = cuda_lib.moe_dispatch(idx, E, x=inp["x"])
    dout = torch.randn((T * k, H), device="cuda").to(TORCH_DTYPES["bf16"])
    N = T * k
    ws = cuda_lib._workspace(ex._lib.moe_experts_backward_workspace_size(ex.handle, N), "cuda")
    eager = [t.clone() for t in ex.backward(d.x_disp, d.offsets, dout, workspace=ws, strategy=strategy)]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = ex.backward(d.x_disp, d.offsets, dout, workspace=ws, strategy=strategy)
    for o in outs:
        o.fill_(0)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(outs, eager):
        assert torch.equal(_bits(a), _bits(b))
