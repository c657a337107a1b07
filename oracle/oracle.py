"""ctypes wrapper around ``moe_oracle.c`` (FP64 CPU oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).  Inputs are numpy
arrays holding the stored bits of F32/F16/BF16 tensors (BF16 as ``uint16``);
the C code decodes them exactly to double.  Nothing here computes any step of
the method itself: every function forwards to the C oracle.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libmoe_oracle.so")

DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, no FMA contraction) and return the path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
           "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I32 = ctypes.c_int
        lib.oracle_route.argtypes = [P, I32, I64, I64, I32, I32, P, P, P]
        lib.oracle_dispatch.argtypes = [P, I64, I64, I32, P, P, P, P]
        lib.oracle_route_sigmoid_grouped.argtypes = [P, I32, I64, I64, P, I32, I32, I32, I32, I32,
                                                     ctypes.c_double, P, P, P]
        lib.oracle_experts.argtypes = [P, P, I64, P, P, P, I32, I64, I64, P]
        lib.oracle_combine.argtypes = [P, P, P, I64, I32, I64, P]
        lib.oracle_forward_tokens.argtypes = [P, P, I32, I32, I64, I64, I32, I32, I64, I64,
                                              P, P, P, P, P, I64, P, P, P]
        lib.oracle_decode.argtypes = [P, I32, I64, P]
        lib.oracle_combine_backward.argtypes = [P, P, P, P, I64, I32, I64, P, P]
        lib.oracle_experts_backward.argtypes = [P, P, I64, P, P, P, I32, I64, I64, P, P, P, P, P]
        lib.oracle_dispatch_backward.argtypes = [P, P, I64, I32, I64, P]
        lib.oracle_selected_router_weights.argtypes = [P, P, I64, I64, I32, I32, I32, ctypes.c_double, P]
        lib.oracle_router_backward.argtypes = [P, P, P, I64, I64, I32, I32, I32, ctypes.c_double, P]
        lib.oracle_round_to_dtype.argtypes = [ctypes.c_double, I32]
        lib.oracle_round_to_dtype.restype = ctypes.c_double
        lib.oracle_num_threads.restype = I32
        lib.oracle_set_threads.argtypes = [I32]
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _stored(a: np.ndarray, dtype: str) -> np.ndarray:
    want = np.float32 if dtype == "f32" else np.uint16
    if dtype == "f16" and a.dtype == np.float16:
        a = a.view(np.uint16)
    if a.dtype != want:
        raise TypeError(f"oracle expects stored {dtype} as {want}, got {a.dtype}")
    return np.ascontiguousarray(a)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_threads(n: int) -> None:
    _load().oracle_set_threads(int(n))


def round_to_dtype(v: float, dtype: str) -> float:
    return float(_load().oracle_round_to_dtype(float(v), DTYPE_CODES[dtype]))


def decode(stored: np.ndarray, dtype: str) -> np.ndarray:
    s = _stored(stored, dtype)
    out = np.empty(s.shape, dtype=np.float64)
    _load().oracle_decode(_ptr(s), DTYPE_CODES[dtype], s.size, _ptr(out))
    return out


def route(logits: np.ndarray, dtype: str, top_k: int, renormalize: bool):
    """Routing contract for every row: returns (idx u32 [T,k], w_pre f64 [T,k], w_cast f64 [T,k])."""
    s = _stored(logits, dtype)
    T, E = s.shape
    idx = np.empty((T, top_k), np.uint32)
    w_pre = np.empty((T, top_k), np.float64)
    w_cast = np.empty((T, top_k), np.float64)
    _load().oracle_route(_ptr(s), DTYPE_CODES[dtype], T, E, top_k, int(bool(renormalize)),
                         _ptr(idx), _ptr(w_pre), _ptr(w_cast))
    return idx, w_pre, w_cast


def route_sigmoid_grouped(logits: np.ndarray, dtype: str, top_k: int, groups: int,
                          selected_groups: int, group_top_two: bool, renormalize: bool,
                          scale: float = 1.0, bias=None):
    """Sigmoid group-limited routing: (idx u32 [T,k], w_pre f64 [T,k], w_cast f64 [T,k])."""
    s = _stored(logits, dtype)
    T, E = s.shape
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    idx = np.empty((T, top_k), np.uint32)
    w_pre = np.empty((T, top_k), np.float64)
    w_cast = np.empty((T, top_k), np.float64)
    _load().oracle_route_sigmoid_grouped(_ptr(s), DTYPE_CODES[dtype], T, E,
                                         _ptr(b) if b is not None else None, top_k, groups,
                                         selected_groups, int(bool(group_top_two)),
                                         int(bool(renormalize)), float(scale),
                                         _ptr(idx), _ptr(w_pre), _ptr(w_cast))
    return idx, w_pre, w_cast


def dispatch(idx: np.ndarray, num_experts: int):
    """Stable capacity-free dispatch: returns (offsets [E+1], row_experts [N], perm [N], invalid)."""
    idx = np.ascontiguousarray(idx, dtype=np.uint32)
    T, k = idx.shape
    offsets = np.empty(num_experts + 1, np.uint32)
    n = T * k
    row_experts = np.empty(max(n, 1), np.uint32)[:n]
    perm = np.empty(max(n, 1), np.uint32)[:n]
    bad = ctypes.c_int64(0)
    _load().oracle_dispatch(_ptr(idx), T, num_experts, k, _ptr(offsets), _ptr(row_experts),
                            _ptr(perm), ctypes.byref(bad))
    return offsets, row_experts, perm, int(bad.value)


def experts(x_disp: np.ndarray, offsets: np.ndarray, gate: np.ndarray, up: np.ndarray,
            down: np.ndarray, dtype: str) -> np.ndarray:
    """SwiGLU experts on dispatched rows (x_disp given as float64 [N,H])."""
    xd = np.ascontiguousarray(x_disp, dtype=np.float64)
    g, u, d = (_stored(a, dtype) for a in (gate, up, down))
    E, I, H = g.shape
    offsets = np.ascontiguousarray(offsets, dtype=np.uint32)
    out = np.zeros((xd.shape[0], H), np.float64)
    _load().oracle_experts(_ptr(xd), _ptr(offsets), E, _ptr(g), _ptr(u), _ptr(d),
                           DTYPE_CODES[dtype], H, I, _ptr(out))
    return out


def combine(expert_out: np.ndarray, perm: np.ndarray, w_cast: np.ndarray) -> np.ndarray:
    """Weighted combine back to token order: y [T,H] float64."""
    eo = np.ascontiguousarray(expert_out, dtype=np.float64)
    T, k = w_cast.shape
    H = eo.shape[1] if eo.ndim == 2 else 0
    y = np.empty((T, H), np.float64)
    _load().oracle_combine(_ptr(eo), _ptr(np.ascontiguousarray(perm, dtype=np.uint32)),
                           _ptr(np.ascontiguousarray(w_cast, dtype=np.float64)), T, k, H, _ptr(y))
    return y


def forward_tokens(x: np.ndarray, logits: np.ndarray, gate: np.ndarray, up: np.ndarray,
                   down: np.ndarray, dtype: str, logits_dtype: str, top_k: int,
                   renormalize: bool, tokens, experts_held=None) -> tuple:
    """Per-token forward for a sample of tokens: returns (idx, w_pre, y) for those tokens.

    ``experts_held``: when given, gate/up/down hold only these expert ids, in
    this order (the sample's experts must be among them)."""
    xs = _stored(x, dtype)
    ls = _stored(logits, logits_dtype)
    g, u, d = (_stored(a, dtype) for a in (gate, up, down))
    T, H = xs.shape
    E = ls.shape[1]
    I = g.shape[1]
    slot = None
    if experts_held is not None:
        slot = np.full(E, -1, np.int64)
        slot[np.asarray(experts_held, np.int64)] = np.arange(len(experts_held))
    toks = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    n = toks.size
    idx = np.empty((n, top_k), np.uint32)
    w = np.empty((n, top_k), np.float64)
    y = np.empty((n, H), np.float64)
    _load().oracle_forward_tokens(_ptr(xs), _ptr(ls), DTYPE_CODES[logits_dtype], DTYPE_CODES[dtype],
                                  T, E, top_k, int(bool(renormalize)), H, I,
                                  _ptr(g), _ptr(u), _ptr(d),
                                  _ptr(slot) if slot is not None else None, _ptr(toks), n,
                                  _ptr(idx), _ptr(w), _ptr(y))
    return idx, w, y


# --------------------------------------------------------------------------
# first-order training backward (user guide section 12)
# --------------------------------------------------------------------------

def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def combine_backward(expert_out, perm, w, dy):
    """(dexpert [N,H], dweights [T,k]) for y = combine(expert_out, perm, w)."""
    eo, w, dy = _f64(expert_out), _f64(w), _f64(dy)
    T, k = w.shape
    H = dy.shape[1]
    dex = np.zeros_like(eo)
    dw = np.full((T, k), np.nan)
    _load().oracle_combine_backward(_ptr(eo), _ptr(np.ascontiguousarray(perm, dtype=np.uint32)),
                                    _ptr(w), _ptr(dy), T, k, H, _ptr(dex), _ptr(dw))
    return dex, dw


def experts_backward(x_disp, offsets, gate, up, down, dtype, dout):
    """(dinput [N,H], dgate [E,I,H], dup [E,I,H], ddown [E,H,I]) in float64."""
    xd, do = _f64(x_disp), _f64(dout)
    g, u, d = (_stored(a, dtype) for a in (gate, up, down))
    E, I, H = g.shape
    offsets = np.ascontiguousarray(offsets, dtype=np.uint32)
    dinput = np.zeros_like(xd)
    dg = np.zeros((E, I, H))
    du = np.zeros((E, I, H))
    dd = np.zeros((E, H, I))
    _load().oracle_experts_backward(_ptr(xd), _ptr(offsets), E, _ptr(g), _ptr(u), _ptr(d),
                                    DTYPE_CODES[dtype], H, I, _ptr(do), _ptr(dinput), _ptr(dg),
                                    _ptr(du), _ptr(dd))
    return dinput, dg, du, dd


def dispatch_backward(dinput, perm, T, k):
    """dx [T,H]: every dispatched row summed back into its token."""
    di = _f64(dinput)
    H = di.shape[1]
    dx = np.empty((T, H))
    _load().oracle_dispatch_backward(_ptr(di), _ptr(np.ascontiguousarray(perm, dtype=np.uint32)),
                                     T, k, H, _ptr(dx))
    return dx


def selected_router_weights(logits, idx, scoring: str, renormalize: bool, scale: float = 1.0):
    """Router weights of a fixed selection (scoring 'softmax' or 'sigmoid'), float64."""
    l = _f64(logits)
    ix = np.ascontiguousarray(idx, dtype=np.int64)
    T, E = l.shape
    k = ix.shape[1]
    w = np.empty((T, k))
    _load().oracle_selected_router_weights(_ptr(l), _ptr(ix), T, E, k, 0 if scoring == "softmax" else 1,
                                           int(bool(renormalize)), float(scale), _ptr(w))
    return w


def router_backward(logits, idx, dweights, scoring: str, renormalize: bool, scale: float = 1.0):
    """dL/dlogits [T,E] for the selected router weights, given dL/dweights."""
    l = _f64(logits)
    ix = np.ascontiguousarray(idx, dtype=np.int64)
    T, E = l.shape
    k = ix.shape[1]
    dl = np.empty((T, E))
    _load().oracle_router_backward(_ptr(l), _ptr(ix), _ptr(_f64(dweights)), T, E, k,
                                   0 if scoring == "softmax" else 1, int(bool(renormalize)),
                                   float(scale), _ptr(dl))
    return dl
