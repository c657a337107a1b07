"""Shared helpers of the GPU parity tests (no test functions here)."""
import numpy as np
import torch

import oracle
from top_routing_grouped_fp32_gb300.inputs import to_stored_numpy

# Output tolerances: max |y - y_oracle| <= TOL * max |y_oracle| over finite
# oracle entries (1e-4 for FP32 experts, 2e-2 for BF16/FP16), routing weights
# within 1e-6 relative of the oracle's pre-cast value.
Y_TOL = {"f32": 1e-4, "f16": 2e-2, "bf16": 2e-2}
W_RTOL = 1e-6
# below the smallest normal FP32 number a relative bound is meaningless
W_ATOL = 1e-37

DT = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}


def u32(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint32)


def stored(t: torch.Tensor) -> np.ndarray:
    return to_stored_numpy(t)


def values(t: torch.Tensor) -> np.ndarray:
    """Exact float64 values of a device tensor (decoded on the host)."""
    return t.detach().double().cpu().numpy()


def assert_weights_match(w32: torch.Tensor, w_pre: np.ndarray):
    got = values(w32)
    assert np.array_equal(np.isnan(got), np.isnan(w_pre)), "NaN weight positions differ"
    ok = ~np.isnan(w_pre)
    err = np.abs(got[ok] - w_pre[ok])
    bound = W_RTOL * np.abs(w_pre[ok]) + W_ATOL
    bad = err > bound
    assert not bad.any(), (f"{bad.sum()} weights off by more than 1e-6 relative; worst "
                           f"{(err / np.maximum(np.abs(w_pre[ok]), W_ATOL)).max():.3e}")


def assert_cast_is_rne(w: torch.Tensor, w32: torch.Tensor):
    """Stored weights are the FP32 weights rounded to nearest-even in their dtype."""
    ref = w32.to(w.dtype)
    assert torch.equal(torch.isnan(w), torch.isnan(ref))
    m = ~torch.isnan(ref)
    assert torch.equal(w[m], ref[m])


def assert_y_close(y_gpu, y_ref: np.ndarray, dtype: str, what: str = "y"):
    got = values(y_gpu) if isinstance(y_gpu, torch.Tensor) else np.asarray(y_gpu, np.float64)
    assert got.shape == y_ref.shape
    nan_ref = np.isnan(y_ref)
    assert np.array_equal(np.isnan(got), nan_ref), f"{what}: NaN positions differ"
    fin = ~nan_ref
    if not fin.any():
        return 0.0
    scale = np.max(np.abs(y_ref[fin]))
    err = np.max(np.abs(got[fin] - y_ref[fin]))
    assert err <= Y_TOL[dtype] * scale, (
        f"{what}: max abs err {err:.4e} > {Y_TOL[dtype]} * {scale:.4e}")
    return err / max(scale, 1e-300)


def oracle_route(logits: torch.Tensor, top_k: int, renorm: bool):
    return oracle.route(stored(logits), DT[logits.dtype], top_k, renorm)


def oracle_forward_sample(inp: dict, top_k: int, renorm: bool, tokens, dtype: str):
    """Oracle y for a sample of tokens, copying only the experts they touch."""
    logits = inp["logits"]
    ldt = DT[logits.dtype]
    idx, _, _ = oracle.route(stored(logits[torch.as_tensor(tokens, device=logits.device)]),
                             ldt, top_k, renorm)
    held = np.unique(idx)
    sel = torch.as_tensor(held.astype(np.int64), device=logits.device)
    g = stored(inp["gate"].index_select(0, sel))
    u = stored(inp["up"].index_select(0, sel))
    d = stored(inp["down"].index_select(0, sel))
    return oracle.forward_tokens(stored(inp["x"]), stored(logits), g, u, d, dtype, ldt, top_k,
                                 renorm, tokens, experts_held=held)


def oracle_dispatch_of(idx: torch.Tensor, E: int, x: torch.Tensor | None = None):
    """The oracle's own dispatch of a routing result: (offsets [E+1], perm [N],
    x_disp rows in dispatch order as float64, or None).  Stage tests build the
    oracle's inputs from this and never from a dispatch output of the GPU."""
    ix = u32(idx)
    k = ix.shape[1]
    off, _, perm, _ = oracle.dispatch(ix, E)
    n = int(off[-1])
    xd = None if x is None else values(x)[perm[:n].astype(np.int64) // k]
    return off, perm, xd
