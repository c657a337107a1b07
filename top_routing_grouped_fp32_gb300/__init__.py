"""GB300 (sm_103a) local Mixture-of-Experts forward: Python binding.

Thin argument marshalling over the C ABI of ``include/moe.h``: every step of
routing, dispatch, the grouped SwiGLU experts and the combine runs in the CUDA
kernels of ``libmoe_gb300.so``.  PyTorch only provides device memory and the
current stream.  Index tensors are ``torch.int32`` holding the ABI's uint32
values (0xFFFFFFFF reads as -1).

Staged use, as in the ruDNN user guide, section 6 ("MoE aufrufen")::

    idx, w = moe_route(logits, top_k=2, renormalize=True)
    d = moe_dispatch(idx, num_experts=E, x=x)
    out = experts.forward_dispatched(d.x_disp, d.offsets)
    y = moe_combine(out, d.perm, w, top_k=2)

or fused: ``y = experts.forward(x, logits, top_k=2, renormalize=True)``.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import DTYPE_CODES, MoeError  # noqa: F401

_TORCH_CODES = {torch.float32: 0, torch.float16: 1, torch.bfloat16: 2}
_CODE_TORCH = {v: k for k, v in _TORCH_CODES.items()}

__all__ = ["load", "moe_route", "moe_route_sigmoid_grouped", "moe_dispatch", "moe_combine",
           "SwiGluExperts", "Dispatched", "moe_combine_backward", "moe_dispatch_backward",
           "moe_router_weights", "moe_router_backward",
           "moe_get_device_status", "MoeError", "library_path", "HostPipeline"]


def load():
    """Load the native library; raises if it has not been built."""
    return _lib.load()


def library_path() -> str:
    return _lib.LIB_PATH


def _code(t: torch.Tensor) -> int:
    try:
        return _TORCH_CODES[t.dtype]
    except KeyError:
        raise MoeError(3, f"dtype {t.dtype} is not F32/F16/BF16") from None


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _workspace(nbytes: int, device) -> torch.Tensor:
    # torch allocations are 512-byte aligned, above the ABI's 256-byte rule
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def moe_route(logits: torch.Tensor, top_k: int, renormalize: bool, weights_f32: bool = False,
              stream=None):
    """Routing contract (user guide, section 4).  Returns (idx int32 [T,k],
    weights [T,k] in the logits dtype[, weights_f32 float32 [T,k]])."""
    lib = load()
    T, E = logits.shape
    idx = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, top_k), dtype=logits.dtype, device=logits.device)
    w32 = torch.empty((T, top_k), dtype=torch.float32, device=logits.device) if weights_f32 else None
    _lib.check(lib.moe_route(_ptr(logits), _code(logits), T, E, top_k, int(bool(renormalize)),
                             _ptr(idx), _ptr(w), _ptr(w32), _stream(stream)))
    return (idx, w, w32) if weights_f32 else (idx, w)


def group_options(top_k: int, groups: int, selected_groups: int, group_top_two: bool,
                  renormalize: bool, scale: float = 1.0):
    return _lib.GroupRoutingOptions(top_k, groups, selected_groups, int(bool(group_top_two)),
                                    int(bool(renormalize)), float(scale))


def moe_route_sigmoid_grouped(logits: torch.Tensor, top_k: int, groups: int, selected_groups: int,
                              group_top_two: bool, renormalize: bool, scale: float = 1.0,
                              bias: torch.Tensor | None = None, weights_f32: bool = False,
                              stream=None):
    """Sigmoid group-limited routing (user guide, section 10).  ``bias``: optional
    FP32 [E] correction used for the selection only."""
    lib = load()
    T, E = logits.shape
    if bias is not None and (bias.dtype != torch.float32 or bias.shape != (E,)):
        raise MoeError(1, "bias must be a float32 [E] tensor")
    opt = group_options(top_k, groups, selected_groups, group_top_two, renormalize, scale)
    idx = torch.empty((T, top_k), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, top_k), dtype=logits.dtype, device=logits.device)
    w32 = torch.empty((T, top_k), dtype=torch.float32, device=logits.device) if weights_f32 else None
    _lib.check(lib.moe_route_sigmoid_grouped(_ptr(logits), _code(logits), T, E, _ptr(bias),
                                             ctypes.byref(opt), _ptr(idx), _ptr(w), _ptr(w32),
                                             _stream(stream)))
    return (idx, w, w32) if weights_f32 else (idx, w)


@dataclass
class Dispatched:
    offsets: torch.Tensor      # int32 [E+1]
    row_experts: torch.Tensor  # int32 [N]
    perm: torch.Tensor         # int32 [N], perm[r] = t*k + j
    x_disp: torch.Tensor | None
    workspace: torch.Tensor    # holds the device status word


def moe_dispatch(idx: torch.Tensor, num_experts: int, x: torch.Tensor | None = None,
                 stream=None) -> Dispatched:
    """Stable capacity-free dispatch (user guide, section 5)."""
    lib = load()
    T, k = idx.shape
    dev = idx.device
    N = T * k
    offsets = torch.empty(num_experts + 1, dtype=torch.int32, device=dev)
    row_experts = torch.empty(N, dtype=torch.int32, device=dev)
    perm = torch.empty(N, dtype=torch.int32, device=dev)
    x_disp = None
    H = 0
    xcode = 0
    if x is not None:
        H = x.shape[1]
        xcode = _code(x)
        x_disp = torch.empty((N, H), dtype=x.dtype, device=dev)
    ws = _workspace(lib.moe_dispatch_workspace_size(T, num_experts, k), dev)
    _lib.check(lib.moe_dispatch(_ptr(idx), T, num_experts, k, _ptr(x), xcode, H, _ptr(offsets),
                                _ptr(row_experts), _ptr(perm), _ptr(x_disp), _ptr(ws), ws.numel(),
                                _stream(stream)))
    return Dispatched(offsets, row_experts, perm, x_disp, ws)


def moe_combine(expert_out: torch.Tensor, perm: torch.Tensor, weights: torch.Tensor, top_k: int,
                stream=None) -> torch.Tensor:
    """Weighted combine back to token order (user guide, section 6)."""
    lib = load()
    T = weights.shape[0]
    H = expert_out.shape[1]
    y = torch.empty((T, H), dtype=expert_out.dtype, device=expert_out.device)
    ws = _workspace(lib.moe_combine_workspace_size(T, top_k), expert_out.device)
    _lib.check(lib.moe_combine(_ptr(expert_out), _code(expert_out), _ptr(perm), _ptr(weights),
                               _code(weights), T, top_k, H, _ptr(y), _ptr(ws), ws.numel(),
                               _stream(stream)))
    return y


# --------------------------------------------------------------------------
# first-order training backward (user guide, section 12)
BWD_STRATEGIES = {"scalar": 0, "auto": 1, "tensor_core": 2}
# --------------------------------------------------------------------------

def moe_combine_backward(expert_out: torch.Tensor, perm: torch.Tensor, weights: torch.Tensor,
                         dy: torch.Tensor, top_k: int, stream=None):
    """(dexpert [T*k,H] in expert_out's dtype, dweights [T,k] float32)."""
    lib = load()
    T, H = dy.shape
    dexpert = torch.empty_like(expert_out)
    dweights = torch.empty((T, top_k), dtype=torch.float32, device=dy.device)
    _lib.check(lib.moe_combine_backward(_ptr(expert_out), _code(expert_out), _ptr(perm), _ptr(weights),
                                        _code(weights), _ptr(dy), T, top_k, H, _ptr(dexpert),
                                        _ptr(dweights), _stream(stream)))
    return dexpert, dweights


def moe_dispatch_backward(dinput: torch.Tensor, perm: torch.Tensor, T: int, top_k: int,
                          stream=None) -> torch.Tensor:
    """dx [T,H]: every dispatched row summed back into its token."""
    lib = load()
    H = dinput.shape[1]
    dx = torch.empty((T, H), dtype=dinput.dtype, device=dinput.device)
    ws = _workspace(lib.moe_combine_workspace_size(T, top_k), dinput.device)
    _lib.check(lib.moe_dispatch_backward(_ptr(dinput), _code(dinput), _ptr(perm), T, top_k, H, _ptr(dx),
                                         _ptr(ws), ws.numel(), _stream(stream)))
    return dx


_SCORING = {"softmax": 0, "sigmoid": 1}


def moe_router_weights(logits: torch.Tensor, idx: torch.Tensor, scoring: str = "softmax",
                       renormalize: bool = True, scale: float = 1.0, stream=None) -> torch.Tensor:
    """FP32 router weights [T,k] of a fixed selection idx."""
    lib = load()
    T, E = logits.shape
    k = idx.shape[1]
    w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _lib.check(lib.moe_router_weights(_ptr(logits), _code(logits), _ptr(idx), T, E, k, _SCORING[scoring],
                                      int(bool(renormalize)), float(scale), _ptr(w), _stream(stream)))
    return w


def moe_router_backward(logits: torch.Tensor, idx: torch.Tensor, dweights: torch.Tensor,
                        scoring: str = "softmax", renormalize: bool = True, scale: float = 1.0,
                        stream=None) -> torch.Tensor:
    """dL/dlogits [T,E] (logits dtype) from FP32 dL/dweights [T,k]."""
    lib = load()
    T, E = logits.shape
    k = idx.shape[1]
    dl = torch.empty_like(logits)
    _lib.check(lib.moe_router_backward(_ptr(logits), _code(logits), _ptr(idx), _ptr(dweights), T, E, k,
                                       _SCORING[scoring], int(bool(renormalize)), float(scale), _ptr(dl),
                                       _stream(stream)))
    return dl


def moe_get_device_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronises the stream and returns the workspace's device status code."""
    lib = load()
    st = lib.moe_get_device_status(_ptr(workspace), _stream(stream))
    return int(st)


class SwiGluExperts:
    """Bias-free SwiGLU experts (SwiGluExperts in src/moe/experts.rs): gate and
    up [E,I,H], down [E,H,I].  The handle does not own the tensors; this object
    keeps references to them so they stay alive."""

    def __init__(self, gate: torch.Tensor, up: torch.Tensor, down: torch.Tensor):
        lib = load()
        self._lib = lib
        self.handle = None
        for t in (gate, up, down):
            if t.dim() != 3:
                raise MoeError(2, "MoE expert weights must be rank-three tensors with matching dtype")
        if not (gate.dtype == up.dtype == down.dtype):
            raise MoeError(3, "MoE expert weights must be rank-three tensors with matching dtype")
        E, I, H = gate.shape
        if tuple(up.shape) != (E, I, H) or tuple(down.shape) != (E, H, I):
            raise MoeError(2, "MoE expert weight dimensions do not match")
        self.gate, self.up, self.down = gate, up, down
        self.E, self.I, self.H = E, I, H
        self.dtype = gate.dtype
        h = ctypes.c_void_p()
        with torch.cuda.device(gate.device):
            _lib.check(lib.moe_experts_create(_ptr(gate), _ptr(up), _ptr(down), _code(gate), E, I, H,
                                              ctypes.byref(h)))
        self.handle = h
        self._ws = None

    def __del__(self):
        if getattr(self, "handle", None) is not None and self._lib is not None:
            self._lib.moe_experts_destroy(self.handle)
            self.handle = None

    # -- workspaces -----------------------------------------------------------
    def forward_workspace_size(self, T: int, top_k: int, logits_dtype=torch.bfloat16) -> int:
        return int(self._lib.moe_forward_workspace_size(self.handle, T, top_k, _TORCH_CODES[logits_dtype]))

    def forward_workspace(self, T: int, top_k: int, logits_dtype=torch.bfloat16) -> torch.Tensor:
        return _workspace(self.forward_workspace_size(T, top_k, logits_dtype), self.gate.device)

    def forward_layout(self, T: int, top_k: int, logits_dtype=torch.bfloat16) -> dict:
        lay = _lib.ForwardLayout()
        _lib.check(self._lib.moe_forward_layout(self.handle, T, top_k, _TORCH_CODES[logits_dtype],
                                                ctypes.byref(lay)))
        return {n: int(getattr(lay, n)) for n, _ in lay._fields_}

    # -- compute ----------------------------------------------------------------
    def forward_dispatched(self, x_disp: torch.Tensor, offsets: torch.Tensor, out=None,
                           workspace=None, stream=None) -> torch.Tensor:
        """forward_dispatched: expert outputs [N,H] in dispatch order."""
        N = x_disp.shape[0]
        if out is None:
            out = torch.empty((N, self.H), dtype=self.dtype, device=x_disp.device)
        if workspace is None:
            workspace = _workspace(self._lib.moe_experts_workspace_size(self.handle, N), x_disp.device)
        _lib.check(self._lib.moe_experts_forward(self.handle, _ptr(x_disp), N, _ptr(offsets), _ptr(out),
                                                 _ptr(workspace), workspace.numel(), _stream(stream)))
        return out

    def forward(self, x: torch.Tensor, logits: torch.Tensor, top_k: int, renormalize: bool,
                y=None, workspace=None, stream=None, events=None) -> torch.Tensor:
        """Fused route -> dispatch -> experts -> combine (SwiGluExperts::forward).
        ``events``: optional list of 6 recorded-capable torch.cuda.Event objects
        (or None for a boundary not to record) marking the stage boundaries."""
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.H), dtype=self.dtype, device=x.device)
        if workspace is None:
            workspace = self.forward_workspace(T, top_k, logits.dtype)
        args = (self.handle, _ptr(x), _ptr(logits), _code(logits), T, top_k, int(bool(renormalize)),
                _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream))
        if events is None:
            _lib.check(self._lib.moe_forward(*args))
        else:
            arr = (ctypes.c_void_p * len(events))(
                *[ctypes.c_void_p(e.cuda_event if e is not None else None) for e in events])
            _lib.check(self._lib.moe_forward_timed(*args, arr, len(events)))
        return y

    def backward(self, x_disp: torch.Tensor, offsets: torch.Tensor, dout: torch.Tensor,
                 workspace=None, stream=None, strategy: str = "scalar"):
        """Expert backward (ExpertTrainingCache::backward_with_strategy): returns
        (dinput [N,H] in the weight dtype, dgate [E,I,H], dup [E,I,H], ddown
        [E,H,I] in FP32).  ``strategy``: "scalar" (the default), "auto" or
        "tensor_core" (F16/BF16 experts)."""
        code = BWD_STRATEGIES[strategy]
        N = x_disp.shape[0]
        dev = x_disp.device
        dinput = torch.empty((N, self.H), dtype=self.dtype, device=dev)
        dgate = torch.empty((self.E, self.I, self.H), dtype=torch.float32, device=dev)
        dup = torch.empty_like(dgate)
        ddown = torch.empty((self.E, self.H, self.I), dtype=torch.float32, device=dev)
        if workspace is None:
            workspace = _workspace(self._lib.moe_experts_backward_workspace_size(self.handle, N), dev)
        _lib.check(self._lib.moe_experts_backward_with_strategy(
            self.handle, _ptr(x_disp), N, _ptr(offsets), _ptr(dout), _ptr(dinput), _ptr(dgate), _ptr(dup),
            _ptr(ddown), code, _ptr(workspace), workspace.numel(), _stream(stream)))
        return dinput, dgate, dup, ddown

    def forward_sigmoid_grouped(self, x: torch.Tensor, logits: torch.Tensor, top_k: int, groups: int,
                                selected_groups: int, group_top_two: bool, renormalize: bool,
                                scale: float = 1.0, bias: torch.Tensor | None = None, y=None,
                                workspace=None, stream=None) -> torch.Tensor:
        """Fused forward with sigmoid group-limited routing
        (SwiGluExperts::forward_sigmoid_grouped)."""
        T = x.shape[0]
        if y is None:
            y = torch.empty((T, self.H), dtype=self.dtype, device=x.device)
        if workspace is None:
            workspace = self.forward_workspace(T, top_k, logits.dtype)
        opt = group_options(top_k, groups, selected_groups, group_top_two, renormalize, scale)
        _lib.check(self._lib.moe_forward_sigmoid_grouped(
            self.handle, _ptr(x), _ptr(logits), _code(logits), T, _ptr(bias), ctypes.byref(opt),
            _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream)))
        return y

    def forward_host(self, x_host: torch.Tensor, logits_host: torch.Tensor, top_k: int,
                     renormalize: bool, y_host: torch.Tensor, workspace: torch.Tensor,
                     stream=None) -> torch.Tensor:
        """The fused forward on host (ideally pinned) tensors; copies happen
        inside the call on ``stream``; synchronise before reading ``y_host``."""
        T = x_host.shape[0]
        for t in (x_host, logits_host, y_host):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("forward_host takes contiguous host tensors")
        _lib.check(self._lib.moe_forward_host(
            self.handle, ctypes.c_void_p(x_host.data_ptr()), ctypes.c_void_p(logits_host.data_ptr()),
            _code(logits_host), T, top_k, int(bool(renormalize)), ctypes.c_void_p(y_host.data_ptr()),
            _ptr(workspace), workspace.numel(), _stream(stream)))
        return y_host

    def host_pipeline(self, T_max: int, top_k: int, renormalize: bool, logits_dtype=torch.bfloat16,
                      depth: int = 2, stream=None) -> "HostPipeline":
        """A pipelined host-buffer forward (moe_host_pipeline_*) for a stream of
        batches of up to T_max tokens."""
        return HostPipeline(self, T_max, top_k, renormalize, logits_dtype, depth, stream)

    def forward_host_workspace(self, T: int, top_k: int, logits_dtype=torch.bfloat16) -> torch.Tensor:
        n = self._lib.moe_forward_host_workspace_size(self.handle, T, top_k, _TORCH_CODES[logits_dtype])
        return _workspace(n, self.gate.device)


class HostPipeline:
    """moe_host_pipeline_*: host batches in, host results out; the copies of
    consecutive batches overlap the forward of the batch between them.  Keep
    the host tensors alive and y unread until ``sync()``."""

    def __init__(self, experts: SwiGluExperts, T_max: int, top_k: int, renormalize: bool,
                 logits_dtype, depth: int, stream):
        self._lib = experts._lib
        self.experts = experts
        self.T_max = T_max
        self.H, self.E = experts.H, experts.E
        code = _TORCH_CODES[logits_dtype]
        n = self._lib.moe_host_pipeline_workspace_size(experts.handle, T_max, top_k, code, depth)
        self.workspace = _workspace(n, experts.gate.device)
        self.stream = stream if stream is not None else torch.cuda.current_stream()
        h = ctypes.c_void_p()
        _lib.check(self._lib.moe_host_pipeline_create(
            experts.handle, T_max, top_k, code, int(bool(renormalize)), depth, _ptr(self.workspace),
            self.workspace.numel(), _stream(self.stream), ctypes.byref(h)))
        self.handle = h

    def submit(self, x_host: torch.Tensor, logits_host: torch.Tensor, y_host: torch.Tensor):
        for t in (x_host, logits_host, y_host):
            if t.is_cuda or not t.is_contiguous():
                raise ValueError("submit takes contiguous host tensors")
        _lib.check(self._lib.moe_host_pipeline_submit(
            self.handle, ctypes.c_void_p(x_host.data_ptr()), ctypes.c_void_p(logits_host.data_ptr()),
            ctypes.c_void_p(y_host.data_ptr()), x_host.shape[0]))

    def sync(self):
        _lib.check(self._lib.moe_host_pipeline_sync(self.handle))

    def close(self):
        if self.handle:
            _lib.check(self._lib.moe_host_pipeline_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
