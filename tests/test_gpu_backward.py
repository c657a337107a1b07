"""First-order training backward (user guide section 12) against the oracle.

Floating outputs follow the forward's bar (max |err| <= 1e-4 * max |ref| for
FP32 outputs or FP32 weights, 2e-2 for BF16/FP16 outputs); the oracle's
backward is itself pinned by finite differences (test_oracle_backward_pins).
The tensor-core strategy holds a, dg and du in the 16-bit weight dtype, as
the pages' training cache does, and these are the operands of its weight
gradients: each operand carries a relative rounding error of at most 2^-8
(BF16), so its FP32 weight gradients are held to 2e-2 * max |ref| too."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import DT, assert_y_close, oracle_dispatch_of, stored, u32, values
from top_routing_grouped_fp32_gb300.inputs import TORCH_DTYPES, WORKLOADS, make_inputs, small_workload

pytestmark = pytest.mark.gpu


def _close(got, ref, tol, what):
    g = values(got) if isinstance(got, torch.Tensor) else got
    assert np.array_equal(np.isnan(g), np.isnan(ref)), f"{what}: NaN positions differ"
    ok = ~np.isnan(ref)
    scale = max(np.abs(ref[ok]).max() if ok.any() else 0.0, 1e-30)
    err = np.abs(g[ok] - ref[ok]).max() if ok.any() else 0.0
    assert err <= tol * scale, f"{what}: max err {err:.3e} > {tol} * {scale:.3e}"


def _wgrad_tol(dtype, strategy):
    return 1e-4 if strategy == "scalar" else 2e-2


BWD_CASES = [
    (300, 8, 2, 256, 384, "bf16"),
    (257, 6, 3, 72, 40, "f32"),
    (257, 6, 3, 72, 40, "bf16"),     # H, I not multiples of 64: ragged k-blocks and columns
    (200, 16, 4, 128, 96, "f16"),
    (64, 1, 1, 64, 64, "bf16"),
    (1500, 4, 2, 320, 704, "bf16"),  # 750 rows per expert: CTA-pair tiles, several m-tiles
    (200, 256, 8, 128, 64, "bf16"),  # decode-like: single-CTA tiles, many empty experts
]


@pytest.mark.parametrize("strategy", ["scalar", "tensor_core"])
@pytest.mark.parametrize("T,E,k,H,I,dtype", BWD_CASES)
def test_expert_backward(cuda_lib, T, E, k, H, I, dtype, strategy):
    if strategy == "tensor_core" and dtype == "f32":
        pytest.skip("the tensor-core strategy takes F16/BF16 experts (rejection tested below)")
    wl = small_workload(T, E, k, H, I, dtype=dtype, seed=T)
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    idx, _ = cuda_lib.moe_route(inp["logits"], k, True)
    d = cuda_lib.moe_dispatch(idx, E, x=inp["x"])
    g = torch.Generator(device="cuda").manual_seed(5)
    dout = torch.randn((T * k, H), generator=g, device="cuda").to(TORCH_DTYPES[dtype])
    dinput, dgate, dup, ddown = experts.backward(d.x_disp, d.offsets, dout, strategy=strategy)
    torch.cuda.synchronize()
    off, _, xd = oracle_dispatch_of(idx, E, inp["x"])
    assert np.array_equal(u32(d.offsets), off), "offsets differ"
    ref = oracle.experts_backward(xd, off, stored(inp["gate"]), stored(inp["up"]), stored(inp["down"]),
                                  dtype, values(dout[:int(off[-1])]))
    assert_y_close(dinput, ref[0], dtype, "dinput")
    for name, got, r in (("dgate", dgate, ref[1]), ("dup", dup, ref[2]), ("ddown", ddown, ref[3])):
        _close(got, r, _wgrad_tol(dtype, strategy), name)


@pytest.mark.parametrize("dtype", ["bf16", "f16"])
def test_expert_backward_segment_tails(cuda_lib, dtype):
    """Tensor-core strategy on CTA-pair tiles with chosen segment lengths: the
    last tile of a segment holds 1, 63, 64, 65, 127, 128 (half tiles, M = 128
    over the pair), 129, 255 or 256 rows, plus segments of 1, 64 and 128 rows
    alone and an empty expert."""
    counts = [257, 319, 320, 321, 383, 384, 385, 511, 512, 1, 64, 128, 0]
    E, H, I = len(counts), 264, 200
    N = sum(counts)
    assert N >= 128 * E
    wl = small_workload(64, E, 1, H, I, dtype=dtype, seed=43)
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    g = torch.Generator(device="cuda").manual_seed(44)
    x_disp = torch.randn((N, H), generator=g, device="cuda").to(TORCH_DTYPES[dtype])
    dout = torch.randn((N, H), generator=g, device="cuda").to(TORCH_DTYPES[dtype])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    offsets = torch.from_numpy(off.view(np.int32)).cuda()
    dinput, dgate, dup, ddown = experts.backward(x_disp, offsets, dout, strategy="tensor_core")
    torch.cuda.synchronize()
    ref = oracle.experts_backward(values(x_disp), off, stored(inp["gate"]), stored(inp["up"]),
                                  stored(inp["down"]), dtype, values(dout))
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            assert_y_close(dinput[a:b], ref[0][a:b], dtype, f"dinput, expert {e} ({b - a} rows)")
    for name, got, r in (("dgate", dgate, ref[1]), ("dup", dup, ref[2]), ("ddown", ddown, ref[3])):
        _close(got, r, 2e-2, name)
    assert torch.all(dgate[E - 1] == 0) and torch.all(ddown[E - 1] == 0)


def test_expert_backward_single_cta_segment_tails(cuda_lib):
    """Tensor-core strategy on single-CTA tiles (N < 128 E) with chosen segment
    lengths: 1, 31, 32, 33, 64, 127, 128, 129 and 200 rows and an empty
    expert, K and N ragged."""
    counts = [1, 31, 32, 33, 64, 127, 128, 129, 200, 0]
    E, H, I = len(counts), 264, 200
    N = sum(counts)
    assert N < 128 * E
    wl = small_workload(64, E, 1, H, I, dtype="bf16", seed=47)
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    g = torch.Generator(device="cuda").manual_seed(48)
    x_disp = torch.randn((N, H), generator=g, device="cuda").to(torch.bfloat16)
    dout = torch.randn((N, H), generator=g, device="cuda").to(torch.bfloat16)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    offsets = torch.from_numpy(off.view(np.int32)).cuda()
    dinput, dgate, dup, ddown = experts.backward(x_disp, offsets, dout, strategy="tensor_core")
    torch.cuda.synchronize()
    ref = oracle.experts_backward(values(x_disp), off, stored(inp["gate"]), stored(inp["up"]),
                                  stored(inp["down"]), "bf16", values(dout))
    for e in range(E):
        a, b = int(off[e]), int(off[e + 1])
        if b > a:
            assert_y_close(dinput[a:b], ref[0][a:b], "bf16", f"dinput, expert {e} ({b - a} rows)")
    for name, got, r in (("dgate", dgate, ref[1]), ("dup", dup, ref[2]), ("ddown", ddown, ref[3])):
        _close(got, r, 2e-2, name)
    assert torch.all(dgate[E - 1] == 0) and torch.all(ddown[E - 1] == 0)


@pytest.mark.parametrize("strategy", ["scalar", "tensor_core"])
def test_expert_backward_empty_experts_get_zero(cuda_lib, strategy):
    wl = small_workload(100, 8, 1, 64, 64, dtype="bf16", seed=3, skew=6.0)
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    idx, _ = cuda_lib.moe_route(inp["logits"], 1, True)
    d = cuda_lib.moe_dispatch(idx, wl.E, x=inp["x"])
    dout = torch.randn((100, 64), device="cuda").to(torch.bfloat16)
    _, dgate, dup, ddown = experts.backward(d.x_disp, d.offsets, dout, strategy=strategy)
    torch.cuda.synchronize()
    cnt = np.diff(u32(d.offsets).astype(np.int64))
    assert (cnt == 0).any()
    for e in np.where(cnt == 0)[0]:
        assert torch.all(dgate[e] == 0) and torch.all(dup[e] == 0) and torch.all(ddown[e] == 0)


def test_tensor_core_backward_rejects_fp32_and_auto_falls_back(cuda_lib):
    wl = small_workload(50, 4, 2, 64, 64, dtype="f32", seed=9)
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    idx, _ = cuda_lib.moe_route(inp["logits"], 2, True)
    d = cuda_lib.moe_dispatch(idx, 4, x=inp["x"])
    dout = torch.randn((100, 64), device="cuda")
    with pytest.raises(RuntimeError, match="UNSUPPORTED|unsupported"):
        experts.backward(d.x_disp, d.offsets, dout, strategy="tensor_core")
    a = experts.backward(d.x_disp, d.offsets, dout, strategy="auto")
    s = experts.backward(d.x_disp, d.offsets, dout, strategy="scalar")
    for x, y in zip(a, s):
        assert torch.equal(x, y)


def test_tensor_core_backward_is_deterministic(cuda_lib):
    wl = small_workload(700, 8, 2, 192, 256, dtype="bf16", seed=11)
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    idx, _ = cuda_lib.moe_route(inp["logits"], 2, True)
    d = cuda_lib.moe_dispatch(idx, 8, x=inp["x"])
    dout = torch.randn((1400, 192), device="cuda").to(torch.bfloat16)
    r1 = experts.backward(d.x_disp, d.offsets, dout, strategy="tensor_core")
    r2 = experts.backward(d.x_disp, d.offsets, dout, strategy="tensor_core")
    for x, y in zip(r1, r2):
        assert torch.equal(x, y)


@pytest.mark.parametrize("dtype,wdtype", [("bf16", "bf16"), ("f32", "f32"), ("f16", "bf16")])
def test_combine_and_dispatch_backward(cuda_lib, dtype, wdtype):
    T, E, k, H = 333, 12, 3, 200
    g = torch.Generator(device="cuda").manual_seed(7)
    logits = torch.randn((T, E), generator=g, device="cuda").to(TORCH_DTYPES[wdtype])
    idx, w = cuda_lib.moe_route(logits, k, True)
    d = cuda_lib.moe_dispatch(idx, E)
    eo = torch.randn((T * k, H), generator=g, device="cuda").to(TORCH_DTYPES[dtype])
    dy = torch.randn((T, H), generator=g, device="cuda").to(TORCH_DTYPES[dtype])
    dexpert, dweights = cuda_lib.moe_combine_backward(eo, d.perm, w, dy, k)
    dx = cuda_lib.moe_dispatch_backward(eo, d.perm, T, k)
    torch.cuda.synchronize()
    _, o_perm, _ = oracle_dispatch_of(idx, E)
    assert np.array_equal(u32(d.perm), o_perm), "perm differs"
    r_dex, r_dw = oracle.combine_backward(values(eo), o_perm, values(w), values(dy))
    assert_y_close(dexpert, r_dex, dtype, "dexpert")
    _close(dweights, r_dw, 1e-5, "dweights")
    assert_y_close(dx, oracle.dispatch_backward(values(eo), o_perm, T, k), dtype, "dx")


@pytest.mark.parametrize("scoring", ["softmax", "sigmoid"])
@pytest.mark.parametrize("renorm,scale", [(True, 1.0), (False, 2.5)])
@pytest.mark.parametrize("dtype,E,k", [("f32", 64, 6), ("bf16", 256, 8), ("f16", 37, 5), ("f32", 1024, 64)])
def test_router_weights_and_backward(cuda_lib, scoring, renorm, scale, dtype, E, k):
    T = 300
    g = torch.Generator(device="cuda").manual_seed(E + k)
    logits = torch.randn((T, E), generator=g, device="cuda").to(TORCH_DTYPES[dtype])
    idx = torch.stack([torch.randperm(E, generator=g, device="cuda")[:k] for _ in range(T)]).to(torch.int32)
    idx[3, 1] = idx[3, 0]            # repeated index: gather semantics
    idx[7, 0] = E + 3                # invalid index: NaN row
    dw = torch.randn((T, k), generator=g, device="cuda")
    w = cuda_lib.moe_router_weights(logits, idx, scoring, renorm, scale)
    dl = cuda_lib.moe_router_backward(logits, idx, dw, scoring, renorm, scale)
    torch.cuda.synchronize()
    ix = u32(idx).astype(np.int64)
    ix[ix >= E] = E + 3
    lg = values(logits)
    r_w = oracle.selected_router_weights(lg, ix, scoring, renorm, scale)
    r_dl = oracle.router_backward(lg, ix, values(dw), scoring, renorm, scale)
    got_w = values(w)
    assert np.array_equal(np.isnan(got_w), np.isnan(r_w))
    ok = ~np.isnan(r_w)
    np.testing.assert_allclose(got_w[ok], r_w[ok], rtol=1e-5, atol=1e-7)
    tol = 1e-4 if dtype == "f32" else 2e-2
    _close(dl, r_dl, tol, "dlogits")
    assert torch.isnan(dl[7]).all() and torch.isnan(w[7]).all()


@pytest.mark.parametrize("name", ["finegrained_bf16", "skewed_bf16"])
def test_tensor_core_backward_full_size(cuda_lib, name):
    """Full-size workload through the tensor-core strategy; the oracle checks the
    smallest and the largest non-empty expert completely (their rows' dinput and
    their three weight gradients, each as a one-expert problem), dinput on a
    sample of rows of every other non-empty expert (first, last and random
    rows, evaluated row by row), and every empty expert is all zeros."""
    wl = WORKLOADS[name]
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    idx, _ = cuda_lib.moe_route(inp["logits"], wl.top_k, wl.renormalize)
    d = cuda_lib.moe_dispatch(idx, wl.E, x=inp["x"])
    o_off, _, xd = oracle_dispatch_of(idx, wl.E, inp["x"])
    assert np.array_equal(u32(d.offsets), o_off), "offsets differ"
    off = o_off.astype(np.int64)
    N = int(off[-1])
    g = torch.Generator(device="cuda").manual_seed(17)
    dout = torch.randn((d.x_disp.shape[0], wl.H), generator=g, device="cuda").to(TORCH_DTYPES[wl.dtype])
    dinput, dgate, dup, ddown = experts.backward(d.x_disp[:N], d.offsets, dout[:N], strategy="tensor_core")
    torch.cuda.synchronize()
    cnt = np.diff(off)
    small = int(np.argmin(np.where(cnt > 0, cnt, np.iinfo(np.int64).max)))
    large = int(np.argmax(cnt))

    def one_expert(e, rows):
        sel = torch.as_tensor([e], device="cuda")
        return oracle.experts_backward(xd[rows], np.array([0, len(rows)], np.uint32),
                                       stored(inp["gate"].index_select(0, sel)),
                                       stored(inp["up"].index_select(0, sel)),
                                       stored(inp["down"].index_select(0, sel)), wl.dtype,
                                       values(dout[torch.as_tensor(rows, device="cuda")]))

    for e in sorted({small, large}):
        rows = np.arange(int(off[e]), int(off[e + 1]))
        ref = one_expert(e, rows)
        assert_y_close(dinput[int(off[e]):int(off[e + 1])], ref[0], wl.dtype, f"dinput, expert {e}")
        for nm, got, r in (("dgate", dgate[e], ref[1][0]), ("dup", dup[e], ref[2][0]),
                           ("ddown", ddown[e], ref[3][0])):
            _close(got, r, 2e-2, f"{nm}, expert {e}")
    rng = np.random.default_rng(18)
    for e in np.where(cnt > 0)[0]:
        if e in (small, large):
            continue
        a, b = int(off[e]), int(off[e + 1])
        rows = np.unique(np.concatenate([[a, b - 1], rng.integers(a, b, size=6)]))
        ref = one_expert(int(e), rows)
        assert_y_close(dinput[torch.as_tensor(rows, device="cuda")], ref[0], wl.dtype, f"dinput rows of expert {e}")
    for z in np.where(cnt == 0)[0]:
        assert torch.all(dgate[z] == 0) and torch.all(dup[z] == 0) and torch.all(ddown[z] == 0)


@pytest.mark.slow
def test_expert_backward_beyond_2g_elements(cuda_lib):
    """Tensor-core backward over N = 1.12 M dispatched rows of H = 2048 (2.29 G
    elements in x_disp, dout, dinput and the padded row copies), so every
    element offset past 2^31 must be computed in 64 bits.  The first and the
    last expert hold a few hundred rows (the last one's rows, and its padded
    rows, lie past 2^31 elements) and are checked in full against the oracle:
    dinput on all their rows and all three weight gradients.  dinput is also
    checked on a sample of rows of every other expert (first, last and random
    rows), which the oracle evaluates row by row."""
    E, H, I = 16, 2048, 128
    rng = np.random.default_rng(61)
    mid = rng.integers(79000, 81000, size=E - 2)
    counts = np.concatenate([[200], mid, [300]]).astype(np.int64)
    N = int(counts.sum())
    assert N * H > 2 ** 31
    wl = small_workload(64, E, 1, H, I, dtype="bf16", seed=62)
    inp = make_inputs(wl, device="cuda")
    experts = cuda_lib.SwiGluExperts(inp["gate"], inp["up"], inp["down"])
    g = torch.Generator(device="cuda").manual_seed(63)
    x_disp = torch.randn((N, H), generator=g, device="cuda").to(torch.bfloat16)
    dout = torch.randn((N, H), generator=g, device="cuda").to(torch.bfloat16)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.uint32)
    offsets = torch.from_numpy(off.view(np.int32)).cuda()
    dinput, dgate, dup, ddown = experts.backward(x_disp, offsets, dout, strategy="tensor_core")
    torch.cuda.synchronize()
    gate, up, down = stored(inp["gate"]), stored(inp["up"]), stored(inp["down"])
    for e in (0, E - 1):
        a, b = int(off[e]), int(off[e + 1])
        sub = np.array([0, b - a], dtype=np.uint32)
        ref = oracle.experts_backward(values(x_disp[a:b]), sub, gate[e:e + 1], up[e:e + 1], down[e:e + 1],
                                      "bf16", values(dout[a:b]))
        assert_y_close(dinput[a:b], ref[0], "bf16", f"dinput, expert {e}")
        for name, got, r in (("dgate", dgate[e:e + 1], ref[1]), ("dup", dup[e:e + 1], ref[2]),
                             ("ddown", ddown[e:e + 1], ref[3])):
            _close(got, r, 2e-2, f"{name}, expert {e}")
    # sampled rows of the other experts, each expert's sample its own sub-problem
    for e in range(1, E - 1):
        a, b = int(off[e]), int(off[e + 1])
        rows = np.unique(np.concatenate([[a, b - 1], rng.integers(a, b, size=30)]))
        sel = torch.as_tensor(rows, device="cuda")
        sub = np.array([0, len(rows)], dtype=np.uint32)
        ref = oracle.experts_backward(values(x_disp[sel]), sub, gate[e:e + 1], up[e:e + 1], down[e:e + 1],
                                      "bf16", values(dout[sel]))
        assert_y_close(dinput[sel], ref[0], "bf16", f"dinput rows of expert {e}")
        assert torch.isfinite(dgate[e]).all() and torch.isfinite(ddown[e]).all()
    del x_disp, dout, dinput, dgate, dup, ddown, experts, inp
    torch.cuda.empty_cache()
