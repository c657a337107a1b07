"""Fused forward parity (moe_forward, the call the benchmark times).

Small cases: every token against the oracle.  The five workloads at full
size: routing indices, offsets and perm read back from the workspace and
compared bit-exactly with the oracle over ALL tokens; y compared on a sample
of tokens evaluated one by one by the oracle, chosen so that every GEMM tile
holds a checked row (including poisoned rows)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DT, assert_y_close, oracle_forward_sample, oracle_route, stored, u32
from top_routing_grouped_fp32_gb300.inputs import WORKLOADS, make_inputs, small_workload, with_dtype

pytestmark = pytest.mark.gpu


def _ws_views(experts, ws, T, k, ldtype):
    lay = experts.forward_layout(T, k, ldtype)
    N = T * k
    E = experts.E
    b = ws
    idx = b[lay["idx"]:lay["idx"] + 4 * N].view(torch.int32).view(T, k)
    offsets = b[lay["offsets"]:lay["offsets"] + 4 * (E + 1)].view(torch.int32)
    perm = b[lay["perm"]:lay["perm"] + 4 * N].view(torch.int32)
    return idx, offsets, perm, lay


def _forward(moe, wl, inp, **kw):
    experts = moe.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    ws = experts.forward_workspace(wl.T, wl.top_k, inp["logits"].dtype)
    y = experts.forward(inp["x"], inp["logits"], wl.top_k, wl.renormalize, workspace=ws, **kw)
    torch.cuda.synchronize()
    return experts, ws, y


def _check_routing_and_dispatch(experts, ws, wl, logits, x=None):
    idx, offsets, perm, lay = _ws_views(experts, ws, wl.T, wl.top_k, logits.dtype)
    o_idx, _, _ = oracle_route(logits, wl.top_k, wl.renormalize)
    assert np.array_equal(u32(idx), o_idx), "routing indices differ"
    o_off, _, o_perm, bad = oracle.dispatch(o_idx, wl.E)
    assert bad == 0
    assert np.array_equal(u32(offsets), o_off), "offsets differ"
    assert np.array_equal(u32(perm), o_perm), "perm differs"
    N, rows = wl.T * wl.top_k, int(o_off[-1])
    if x is not None and (wl.H * x.element_size()) % 16 == 0:
        # token-order gather: slot_row is the inverse of perm on every slot
        slot_row = ws[lay["slot_row"]:lay["slot_row"] + 4 * N].view(torch.int32)
        inv = np.full(N, 0xFFFFFFFF, dtype=np.uint32)
        inv[o_perm[:rows]] = np.arange(rows, dtype=np.uint32)
        assert np.array_equal(u32(slot_row), inv), "slot_row is not the inverse of perm"
    if x is not None:
        s = x.element_size()
        x_disp = ws[lay["x_disp"]:lay["x_disp"] + rows * wl.H * s].view(x.dtype).view(rows, wl.H)
        src = x[torch.from_numpy((o_perm[:rows] // wl.top_k).astype(np.int64)).to(x.device)]
        assert torch.equal(x_disp.view(torch.uint8), src.contiguous().view(torch.uint8)), "x_disp differs"
    return o_idx, o_off


@pytest.mark.parametrize("T,E,k,H,I,dtype,renorm", [
    (300, 8, 2, 256, 384, "bf16", True),
    (257, 6, 3, 264, 200, "bf16", False),
    (200, 16, 4, 512, 128, "f16", True),
    (150, 5, 2, 40, 70, "f32", True),
    (100, 4, 2, 60, 90, "bf16", False),
    # >= 128 rows per expert: CTA-pair tiles with k-block tails
    (1000, 4, 2, 200, 136, "bf16", True),   # H = 3*64 + 8: a one-chunk k-block tail
    (700, 3, 3, 72, 64, "f16", False),      # H = 64 + 8
    (300, 1024, 8, 64, 64, "bf16", True),   # E at its limit: 8 KiB of per-expert tables in shared memory
    (64, 256, 64, 64, 64, "bf16", True),    # top_k at its limit: two 32-slot groups per token in the scatter
    (50, 4, 2, 8, 16, "bf16", False),       # the smallest tcgen05 shapes: one k-block, 8 of 64 columns
])
def test_forward_small_all_tokens(cuda_lib, T, E, k, H, I, dtype, renorm):
    wl = small_workload(T, E, k, H, I, dtype=dtype, renormalize=renorm, seed=T + E)
    inp = make_inputs(wl, device="cuda")
    experts, ws, y = _forward(cuda_lib, wl, inp)
    _check_routing_and_dispatch(experts, ws, wl, inp["logits"], inp["x"])
    _, _, ref = oracle_forward_sample(inp, k, renorm, np.arange(T), dtype)
    assert_y_close(y, ref, dtype)
    assert cuda_lib.moe_get_device_status(ws) == 0


def test_forward_tiny_fp32_workload(cuda_lib):
    wl = WORKLOADS["tiny_fp32"]
    inp = make_inputs(wl, device="cuda")
    experts, ws, y = _forward(cuda_lib, wl, inp)
    o_idx, _ = _check_routing_and_dispatch(experts, ws, wl, inp["logits"], inp["x"])
    assert o_idx[:8].tolist() == [[0, 1], [1, 2], [0, 1], [0, 1], [0, 2], [3, 1], [0, 1], [0, 3]]
    _, _, ref = oracle_forward_sample(inp, wl.top_k, wl.renormalize, np.arange(wl.T), "f32")
    assert_y_close(y, ref, "f32")


# Rows per m-tile of the grouped GEMMs: 128 for a single-CTA tile, 256 for a
# CTA pair (two 128-row halves).  Covering every 128-row block of every
# expert's segment covers every tile and every half of every pair tile.
TILE_ROWS = 128


def _tile_cover_tokens(wl, o_off, o_perm, seed=0):
    """Tokens such that every 128-row block of every expert's segment (counted
    from the segment start, as the GEMM tiles are) holds at least one of their
    rows, plus the token of each segment's last row.  From the oracle's own
    dispatch of the full routing result."""
    rng = np.random.default_rng(seed)
    toks = set()
    for e in range(wl.E):
        a, b = int(o_off[e]), int(o_off[e + 1])
        for m0 in range(a, b, TILE_ROWS):
            toks.add(int(o_perm[rng.integers(m0, min(b, m0 + TILE_ROWS))]) // wl.top_k)
        if b > a:
            toks.add(int(o_perm[b - 1]) // wl.top_k)
    return toks


def _assert_every_tile_hit(wl, o_off, o_perm, toks):
    row_of_slot = np.empty(wl.T * wl.top_k, np.int64)
    n = int(o_off[-1])
    row_of_slot[o_perm[:n].astype(np.int64)] = np.arange(n)
    t = np.asarray(sorted(toks), np.int64)
    rows = row_of_slot[(t[:, None] * wl.top_k + np.arange(wl.top_k)).ravel()]
    hit = set()
    for r in rows.tolist():
        e = int(np.searchsorted(o_off, r, side="right")) - 1
        hit.add((e, (r - int(o_off[e])) // TILE_ROWS))
    for e in range(wl.E):
        cnt = int(o_off[e + 1] - o_off[e])
        for m in range((cnt + TILE_ROWS - 1) // TILE_ROWS):
            assert (e, m) in hit, f"expert {e} m-block {m} holds no checked row"
        if cnt:
            assert row_of_slot[int(o_perm[int(o_off[e + 1]) - 1])] in set(rows.tolist())


@pytest.mark.slow
@pytest.mark.parametrize("dtype", ["bf16", "f16"])
@pytest.mark.parametrize("name", ["mixtral_bf16", "finegrained_bf16", "skewed_bf16", "decode_bf16"])
def test_forward_full_workloads(cuda_lib, name, dtype):
    """Full size: routing and dispatch over every token; y on a token sample
    chosen (from the oracle's dispatch) so that every 128-row block of every
    expert's segment and every segment's last row is checked, on all H
    columns (every n-block), plus the first and last tokens and, for the
    skewed workload, poisoned rows and the control row."""
    wl = with_dtype(WORKLOADS[name], dtype)
    inp = make_inputs(wl, device="cuda")
    experts, ws, y = _forward(cuda_lib, wl, inp)
    o_idx, o_off = _check_routing_and_dispatch(experts, ws, wl, inp["logits"], inp["x"])
    _, _, o_perm, _ = oracle.dispatch(o_idx, wl.E)
    toks = _tile_cover_tokens(wl, o_off, o_perm) | {0, wl.T - 1}
    meta = inp["meta"].get("poison")
    if meta:
        toks |= set(meta["rows"][:6]) | {meta["control"]}
    _assert_every_tile_hit(wl, o_off, o_perm, toks)
    toks = np.array(sorted(toks))
    _, _, ref = oracle_forward_sample(inp, wl.top_k, wl.renormalize, toks, wl.dtype)
    assert_y_close(y[torch.as_tensor(toks, device="cuda")], ref, wl.dtype)
    if wl.poison_frac:
        rows = inp["meta"]["poison"]["rows"]
        assert torch.isnan(y[rows]).all()
        others = torch.ones(wl.T, dtype=torch.bool, device="cuda")
        others[rows] = False
        assert torch.isfinite(y[others]).all()
    assert cuda_lib.moe_get_device_status(ws) == 0
    del experts, ws, y, inp
    torch.cuda.empty_cache()


@pytest.mark.slow
def test_forward_beyond_2g_elements(cuda_lib):
    """More than 2^31 elements in the dispatched rows and in the slot buffer
    (N = 1.12 M rows of H = 2048: 2.29 G elements), so every element offset
    past 2^31 must be computed in 64 bits: the gather, the GEMMs' row
    addressing, the weighted slot stores and the combine.  Routing and
    dispatch over every token and x_disp in full; y bit for bit the slot sum
    on every element; y against the oracle on a token sample that reaches
    every 128-row block of every segment and the last tokens (whose slots lie
    past 2^31 elements); the staged path (expert_out [N, H], moe_combine)
    against the oracle on the same sample."""
    T, E, k, H, I = 140000, 16, 8, 2048, 128
    assert T * k * H > 2 ** 31
    wl = small_workload(T, E, k, H, I, dtype="bf16", renormalize=True, seed=31)
    inp = make_inputs(wl, device="cuda")
    experts, ws, y = _forward(cuda_lib, wl, inp)
    o_idx, o_off = _check_routing_and_dispatch(experts, ws, wl, inp["logits"], inp["x"])
    lay = experts.forward_layout(T, k, inp["logits"].dtype)
    slots = ws[lay["slots"]:lay["slots"] + T * k * H * 2].view(torch.bfloat16).view(T, k, H)
    acc = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    for j in range(k):
        acc += slots[:, j].float()
    assert torch.equal(y.view(torch.int16), acc.to(torch.bfloat16).view(torch.int16))
    assert cuda_lib.moe_get_device_status(ws) == 0
    del acc, slots, ws
    torch.cuda.empty_cache()
    _, _, o_perm, _ = oracle.dispatch(o_idx, wl.E)
    toks = _tile_cover_tokens(wl, o_off, o_perm) | set(range(T - 8, T)) | {0}
    _assert_every_tile_hit(wl, o_off, o_perm, toks)
    toks = np.array(sorted(toks))
    _, _, ref = oracle_forward_sample(inp, k, True, toks, "bf16")
    assert_y_close(y[torch.as_tensor(toks, device="cuda")], ref, "bf16")
    # the staged calls: route, dispatch, expert forward into [N, H], combine
    idx, w = cuda_lib.moe_route(inp["logits"], k, True)
    d = cuda_lib.moe_dispatch(idx, wl.E, x=inp["x"])
    out = experts.forward_dispatched(d.x_disp, d.offsets)
    assert out.shape == (T * k, H)
    y2 = cuda_lib.moe_combine(out, d.perm, w, k)
    torch.cuda.synchronize()
    assert_y_close(y2[torch.as_tensor(toks, device="cuda")], ref, "bf16")
    del experts, y, y2, out, d, inp
    torch.cuda.empty_cache()


@pytest.mark.parametrize("T,E,k,H,I,dtype", [
    (1000, 16, 4, 512, 256, "bf16"),   # CTA-pair tiles
    (700, 3, 3, 72, 64, "f16"),        # a 72-column row
    (300, 1024, 8, 264, 64, "bf16"),   # single-CTA tiles, a 264-column row
    (64, 256, 64, 64, 64, "bf16"),     # top_k at its limit
])
def test_forward_combine_is_the_slot_sum(cuda_lib, T, E, k, H, I, dtype):
    """The fused forward's combine: y is bit for bit the ascending-j FP32 sum
    of the weighted slot rows the down epilogue left in the workspace,
    rounded once to the dtype, and a second call gives the same bits."""
    wl = small_workload(T, E, k, H, I, dtype=dtype, renormalize=True, seed=T + k)
    inp = make_inputs(wl, device="cuda")
    experts, ws, y = _forward(cuda_lib, wl, inp)
    lay = experts.forward_layout(T, k, inp["logits"].dtype)
    s = y.element_size()
    slots = ws[lay["slots"]:lay["slots"] + T * k * H * s].view(y.dtype).view(T, k, H)
    acc = torch.zeros((T, H), dtype=torch.float32, device="cuda")
    for j in range(k):
        acc += slots[:, j].float()
    assert torch.equal(y.view(torch.int16), acc.to(y.dtype).view(torch.int16))
    y2 = experts.forward(inp["x"], inp["logits"], k, True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))


def test_forward_timed_partial_events(cuda_lib):
    """moe_forward_timed records only the boundaries it is given and computes the same bits."""
    wl = small_workload(1000, 16, 4, 512, 256, dtype="bf16", renormalize=True, seed=22)
    inp = make_inputs(wl, device="cuda")
    experts, ws, y1 = _forward(cuda_lib, wl, inp)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in ev:
        e.record()
    torch.cuda.synchronize()
    y2 = experts.forward(inp["x"], inp["logits"], wl.top_k, wl.renormalize, workspace=ws,
                         events=[None, None, ev[2], ev[3], None, None])
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert ev[2].elapsed_time(ev[3]) > 0.0  # the gate/up product lies between them


def test_forward_deterministic_and_host_variant(cuda_lib):
    wl = small_workload(1000, 16, 4, 512, 256, dtype="bf16", renormalize=True, seed=21)
    inp = make_inputs(wl, device="cuda")
    experts, ws, y1 = _forward(cuda_lib, wl, inp)
    y2 = experts.forward(inp["x"], inp["logits"], wl.top_k, wl.renormalize, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    # the host-buffer entry point: the same bits
    xh = inp["x"].cpu().pin_memory()
    lh = inp["logits"].cpu().pin_memory()
    yh = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
    wsh = experts.forward_host_workspace(wl.T, wl.top_k, torch.bfloat16)
    experts.forward_host(xh, lh, wl.top_k, wl.renormalize, yh, wsh)
    torch.cuda.synchronize()
    assert torch.equal(yh.view(torch.int16), y1.cpu().view(torch.int16))


def test_forward_fp32_logits_bf16_experts(cuda_lib):
    wl = small_workload(300, 8, 2, 256, 256, dtype="bf16", renormalize=True, seed=8)
    inp = make_inputs(wl, device="cuda", logits_dtype="f32")
    experts, ws, y = _forward(cuda_lib, wl, inp)
    _check_routing_and_dispatch(experts, ws, wl, inp["logits"], inp["x"])
    _, _, ref = oracle.forward_tokens(stored(inp["x"]), stored(inp["logits"]), stored(inp["gate"]),
                                      stored(inp["up"]), stored(inp["down"]), "bf16", "f32", 2, True,
                                      np.arange(wl.T))
    assert_y_close(y, ref, "bf16")


def test_forward_staged_matches_fused(cuda_lib):
    """route -> dispatch -> forward_dispatched -> combine gives the fused result
    up to the rounding of the weighted slot values."""
    wl = small_workload(400, 8, 2, 256, 384, dtype="bf16", renormalize=False, seed=5)
    inp = make_inputs(wl, device="cuda")
    experts, ws, y = _forward(cuda_lib, wl, inp)
    idx, w = cuda_lib.moe_route(inp["logits"], 2, False)
    d = cuda_lib.moe_dispatch(idx, wl.E, x=inp["x"])
    out = experts.forward_dispatched(d.x_disp, d.offsets)
    y2 = cuda_lib.moe_combine(out, d.perm, w, 2)
    torch.cuda.synchronize()
    scale = y.float().abs().max().item()
    assert (y.float() - y2.float()).abs().max().item() <= 2 ** -7 * scale


def test_forward_empty_batch(cuda_lib):
    wl = small_workload(4, 4, 2, 64, 64, dtype="bf16", seed=1)
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    y = experts.forward(inp["x"][:0], inp["logits"][:0], 2, True)
    assert y.shape == (0, 64)
