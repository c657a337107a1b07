"""ctypes declarations of the C ABI in include/moe.h.

Loading fails loudly: if ``libmoe_gb300.so`` is missing or cannot be loaded
there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_OK = 0
STATUS_NAMES = {
    0: "MOE_OK",
    1: "MOE_ERR_INVALID_ARG",
    2: "MOE_ERR_SHAPE",
    3: "MOE_ERR_DTYPE",
    4: "MOE_ERR_UNSUPPORTED",
    5: "MOE_ERR_CUDA",
    6: "MOE_ERR_INVALID_INDEX",
    7: "MOE_ERR_DEVICE_TIMEOUT",
}
DTYPE_CODES = {"f32": 0, "f16": 1, "bf16": 2}


class MoeError(RuntimeError):
    """A non-OK moe_status, with the library's message."""

    def __init__(self, status: int, message: str):
        self.status = status
        self.status_name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{self.status_name}: {message}")


class ForwardLayout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("idx", "weights", "offsets", "perm", "x_disp", "h", "slots", "slot_row", "total")]


class GroupRoutingOptions(ctypes.Structure):
    """moe_group_routing_options (user guide, section 10)."""
    _fields_ = [("top_k", ctypes.c_int32), ("groups", ctypes.c_int32),
                ("selected_groups", ctypes.c_int32), ("group_top_two", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("scale", ctypes.c_float)]


_lib = None
_lock = threading.Lock()

P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int32
INT = ctypes.c_int
SZ = ctypes.c_size_t
ST = ctypes.c_int

_SIGNATURES = {
    "moe_last_error": (ctypes.c_char_p, []),
    "moe_status_string": (ctypes.c_char_p, [ST]),
    "moe_route": (ST, [P, INT, I64, I64, I32, INT, P, P, P, P]),
    "moe_route_sigmoid_grouped": (ST, [P, INT, I64, I64, P, ctypes.POINTER(GroupRoutingOptions),
                                       P, P, P, P]),
    "moe_forward_sigmoid_grouped": (ST, [P, P, P, INT, I64, P, ctypes.POINTER(GroupRoutingOptions),
                                         P, P, SZ, P]),
    "moe_dispatch_workspace_size": (SZ, [I64, I64, I32]),
    "moe_dispatch": (ST, [P, I64, I64, I32, P, INT, I64, P, P, P, P, P, SZ, P]),
    "moe_dispatch_noalloc": (ST, [P, I64, I64, I32, P, INT, I64, P, P, P, P, P]),
    "moe_experts_create": (ST, [P, P, P, INT, I64, I64, I64, ctypes.POINTER(P)]),
    "moe_experts_destroy": (None, [P]),
    "moe_experts_workspace_size": (SZ, [P, I64]),
    "moe_experts_forward": (ST, [P, P, I64, P, P, P, SZ, P]),
    "moe_combine_workspace_size": (SZ, [I64, I32]),
    "moe_combine": (ST, [P, INT, P, P, INT, I64, I32, I64, P, P, SZ, P]),
    "moe_forward_workspace_size": (SZ, [P, I64, I32, INT]),
    "moe_forward": (ST, [P, P, P, INT, I64, I32, INT, P, P, SZ, P]),
    "moe_forward_timed": (ST, [P, P, P, INT, I64, I32, INT, P, P, SZ, P, ctypes.POINTER(P), INT]),
    "moe_forward_host_workspace_size": (SZ, [P, I64, I32, INT]),
    "moe_forward_host": (ST, [P, P, P, INT, I64, I32, INT, P, P, SZ, P]),
    "moe_host_pipeline_workspace_size": (SZ, [P, I64, I32, INT, INT]),
    "moe_host_pipeline_create": (ST, [P, I64, I32, INT, INT, INT, P, SZ, P, ctypes.POINTER(P)]),
    "moe_host_pipeline_submit": (ST, [P, P, P, P, I64]),
    "moe_host_pipeline_sync": (ST, [P]),
    "moe_host_pipeline_destroy": (ST, [P]),
    "moe_forward_layout": (ST, [P, I64, I32, INT, ctypes.POINTER(ForwardLayout)]),
    "moe_get_device_status": (ST, [P, P]),
    "moe_combine_backward": (ST, [P, INT, P, P, INT, P, I64, I32, I64, P, P, P]),
    "moe_dispatch_backward": (ST, [P, INT, P, I64, I32, I64, P, P, SZ, P]),
    "moe_experts_backward_workspace_size": (SZ, [P, I64]),
    "moe_experts_backward": (ST, [P, P, I64, P, P, P, P, P, P, P, SZ, P]),
    "moe_experts_backward_with_strategy": (ST, [P, P, I64, P, P, P, P, P, P, I32, P, SZ, P]),
    "moe_router_weights": (ST, [P, INT, P, I64, I64, I32, INT, INT, ctypes.c_float, P, P]),
    "moe_router_backward": (ST, [P, INT, P, P, I64, I64, I32, INT, INT, ctypes.c_float, P, P]),
    "moe_selftest_bounded_wait": (ST, [P, ctypes.c_uint32, P]),
}


def exported_names() -> list[str]:
    return sorted(_SIGNATURES)


def load(path: str | None = None):
    """Load the library (once).  Raises if it is missing: no CPU fallback."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(
                f"{p} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()'); "
                "this package has no CPU fallback")
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def check(status: int) -> None:
    if status != MOE_OK:
        msg = load().moe_last_error().decode(errors="replace")
        raise MoeError(status, msg)
