"""Expert parity: moe_experts_forward (grouped gate/up + SwiGLU + down) against
the oracle on the same dispatched rows.  Sizes span several 128-row tiles,
ragged segment ends, empty experts, K and N not multiples of the tile, both
16-bit dtypes on the tcgen05 path and FP32 / odd shapes on the SIMT path."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DT, assert_y_close, oracle_dispatch_of, stored, u32, values
from top_routing_grouped_fp32_gb300.inputs import make_inputs, small_workload

pytestmark = pytest.mark.gpu


def _run(moe, T, E, k, H, I, dtype, seed=0, skew=0.0):
    wl = small_workload(T, E, k, H, I, dtype=dtype, seed=seed, skew=skew)
    inp = make_inputs(wl, device="cuda")
    experts = moe.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    idx, _ = moe.moe_route(inp["logits"], k, True)
    d = moe.moe_dispatch(idx, E, x=inp["x"])
    out = experts.forward_dispatched(d.x_disp, d.offsets)
    torch.cuda.synchronize()
    # the oracle's inputs come from its own dispatch of the routing result
    off, _, xd = oracle_dispatch_of(idx, E, inp["x"])
    assert np.array_equal(u32(d.offsets), off), "offsets differ"
    ref = oracle.experts(xd, off, stored(inp["gate"]), stored(inp["up"]), stored(inp["down"]), dtype)
    n = int(off[-1])
    assert_y_close(out[:n], ref[:n], dtype, "expert_out")
    return experts, d, out


@pytest.mark.parametrize("T,E,k,H,I,dtype", [
    (200, 4, 2, 512, 384, "bf16"),     # 400 rows, 3 gate/up n-blocks, 2 down n-blocks
    (200, 4, 2, 512, 384, "f16"),
    (333, 6, 3, 264, 200, "bf16"),     # ragged K (264, 200) and ragged n (I=200, H=264)
    (97, 16, 2, 128, 136, "bf16"),     # many experts with few rows, some empty
    (1024, 8, 2, 256, 1408, "bf16"),   # ~256 rows/expert, 11 n-blocks
    (64, 1, 1, 64, 64, "bf16"),        # one expert, k=1
    (5, 3, 2, 72, 8, "bf16"),          # a handful of rows, I=8
    # >= 128 rows per expert on average: CTA-pair (cta_group::2) tiles of 256 rows
    (2000, 8, 2, 264, 200, "bf16"),    # ragged K and n on the pair path
    (1500, 4, 2, 256, 384, "f16"),
    (700, 2, 1, 512, 256, "bf16"),     # two experts, pair tiles straddling a segment end
])
def test_experts_tcgen05(cuda_lib, T, E, k, H, I, dtype):
    _run(cuda_lib, T, E, k, H, I, dtype, seed=T + H)


@pytest.mark.parametrize("T,E", [(800, 32), (3000, 24)])
def test_experts_skewed_segments(cuda_lib, T, E):
    """The hottest expert holds several full tiles while others are empty
    (single-CTA tiles for T=800, CTA-pair tiles for T=3000)."""
    _, d, _ = _run(cuda_lib, T, E, 4, 256, 256, "bf16", seed=3, skew=2.0 if T < 1000 else 4.0)
    cnt = np.diff(u32(d.offsets).astype(np.int64))
    assert cnt.max() > 384 and (cnt == 0).sum() > 0


@pytest.mark.parametrize("T,E,k,H,I,dtype", [
    (64, 4, 2, 64, 128, "f32"),        # the tiny workload's shapes
    (150, 5, 2, 40, 70, "f32"),
    (120, 4, 2, 60, 90, "bf16"),       # H, I not multiples of 8: SIMT path
    (80, 3, 2, 20, 44, "f16"),
])
def test_experts_simt(cuda_lib, T, E, k, H, I, dtype):
    _run(cuda_lib, T, E, k, H, I, dtype, seed=T)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_experts_segment_tails(cuda_lib, dtype):
    """Chosen segment lengths on CTA-pair tiles (N >= 128 E): the last tile of
    a segment holds 1, 63, 64, 65, 127, 128 (a half tile: M = 128 over the
    pair), 129, 255 or 256 rows (a full 256-row tile), plus segments of 1, 64
    and 128 rows alone and an empty expert."""
    counts = [257, 319, 320, 321, 383, 384, 385, 511, 512, 1, 64, 128, 0]
    E, H, I = len(counts), 264, 200
    N = sum(counts)
    assert N >= 128 * E
    wl = small_workload(64, E, 1, H, I, dtype=dtype, seed=41)
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    g = torch.Generator(device="cuda").manual_seed(42)
    x_disp = torch.randn((N, H), generator=g, device="cuda").to(inp["x"].dtype)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    offsets = torch.from_numpy(off.view(np.int32)).cuda()
    out = experts.forward_dispatched(x_disp, offsets)
    torch.cuda.synchronize()
    ref = oracle.experts(values(x_disp), off, stored(inp["gate"]), stored(inp["up"]), stored(inp["down"]),
                         dtype)
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            assert_y_close(out[a:b], ref[a:b], dtype, f"expert {e} ({b - a} rows)")


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_experts_single_cta_segment_tails(cuda_lib, dtype):
    """Chosen segment lengths on single-CTA tiles (N < 128 E): segments of
    1, 31 and 32 rows (thin tiles: A through a 32-row box), 33, 64, 127 and 128
    rows (full 128-row boxes), 129 and 200 rows (two tiles, the second holding
    1 or 72 rows, thin or not) and an empty expert; K = 264 and N = 200 leave
    ragged k-blocks and columns."""
    counts = [1, 31, 32, 33, 64, 127, 128, 129, 200, 0]
    E, H, I = len(counts), 264, 200
    N = sum(counts)
    assert N < 128 * E
    wl = small_workload(64, E, 1, H, I, dtype=dtype, seed=45)
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    g = torch.Generator(device="cuda").manual_seed(46)
    x_disp = torch.randn((N, H), generator=g, device="cuda").to(inp["x"].dtype)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    offsets = torch.from_numpy(off.view(np.int32)).cuda()
    out = experts.forward_dispatched(x_disp, offsets)
    torch.cuda.synchronize()
    ref = oracle.experts(values(x_disp), off, stored(inp["gate"]), stored(inp["up"]), stored(inp["down"]),
                         dtype)
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            assert_y_close(out[a:b], ref[a:b], dtype, f"expert {e} ({b - a} rows)")


def test_experts_output_alignment_fallback(cuda_lib):
    """moe_experts_forward into an output that is 16- but not 32-byte aligned:
    the epilogues then store 16-byte vectors instead of 32-byte sectors, with
    the same bits as an aligned output."""
    wl = small_workload(1000, 4, 2, 256, 384, dtype="bf16", seed=77)
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    idx, _ = cuda_lib.moe_route(inp["logits"], 2, True)
    d = cuda_lib.moe_dispatch(idx, wl.E, x=inp["x"])
    N = d.x_disp.shape[0]
    aligned = experts.forward_dispatched(d.x_disp, d.offsets)
    buf = torch.empty(N * wl.H + 8, dtype=torch.bfloat16, device="cuda")
    off = buf[8:].view(N, wl.H)  # 16 bytes past a 512-byte-aligned allocation
    assert off.data_ptr() % 32 == 16
    experts.forward_dispatched(d.x_disp, d.offsets, out=off)
    torch.cuda.synchronize()
    n = int(d.offsets[-1].item())
    assert torch.equal(off[:n].view(torch.int16), aligned[:n].view(torch.int16))


def test_experts_deterministic(cuda_lib):
    experts, d, out = _run(cuda_lib, 500, 8, 2, 256, 384, "bf16", seed=4)
    again = experts.forward_dispatched(d.x_disp, d.offsets)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), again.view(torch.int16))


def test_experts_rejects_mismatched_weights(cuda_lib):
    g = torch.zeros((2, 8, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(cuda_lib.MoeError, match="dimensions do not match"):
        cuda_lib.SwiGluExperts(g, g, torch.zeros((2, 8, 16), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(cuda_lib.MoeError, match="matching dtype"):
        cuda_lib.SwiGluExperts(g, g.half(), torch.zeros((2, 16, 8), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(cuda_lib.MoeError, match="rank-three"):
        cuda_lib.SwiGluExperts(g[0], g[0], g[0])
