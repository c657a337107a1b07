"""C-ABI checks that need no GPU: the library builds and loads, exports every
function that include/moe.h declares, and rejects bad arguments on the host
before any CUDA call (the argument checks come first in every entry point)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")

OK, INVALID_ARG, SHAPE, DTYPE, UNSUPPORTED = 0, 1, 2, 3, 4
F32, F16, BF16 = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    from top_routing_grouped_fp32_gb300 import build as native_build
    from top_routing_grouped_fp32_gb300 import _lib
    native_build.build()
    return _lib.load()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_staged_and_fused_calls():
    names = _declared_functions()
    for n in ("moe_route", "moe_dispatch", "moe_experts_create", "moe_experts_forward",
              "moe_combine", "moe_forward"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    from top_routing_grouped_fp32_gb300 import _lib
    declared = _declared_functions()
    missing = [n for n in declared if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"
    # the Python binding declares a signature for every one of them
    assert sorted(_lib.exported_names()) == declared


def test_status_strings(lib):
    for code, name in [(0, b"MOE_OK"), (1, b"MOE_ERR_INVALID_ARG"), (6, b"MOE_ERR_INVALID_INDEX"),
                       (7, b"MOE_ERR_DEVICE_TIMEOUT")]:
        assert lib.moe_status_string(code) == name


FAKE = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails its checks first


def _msg(lib):
    return lib.moe_last_error().decode()


@pytest.mark.parametrize("T,E,k,want", [
    (4, 8, 0, INVALID_ARG),      # top_k < 1
    (4, 8, 9, INVALID_ARG),      # top_k > E
    (4, 0, 1, SHAPE),            # no experts
    (-1, 8, 2, SHAPE),           # negative T
    (4, 1025, 2, UNSUPPORTED),   # E beyond 1024
    (4, 128, 65, UNSUPPORTED),   # top_k beyond 64
    (2 ** 31, 8, 2, UNSUPPORTED),  # T*k beyond 2^31-1
])
def test_route_argument_rules(lib, T, E, k, want):
    st = lib.moe_route(FAKE, BF16, T, E, k, 1, FAKE, FAKE, None, None)
    assert st == want, _msg(lib)


def test_route_rejects_bad_dtype_and_nulls(lib):
    assert lib.moe_route(FAKE, 7, 4, 8, 2, 1, FAKE, FAKE, None, None) == DTYPE
    assert lib.moe_route(None, BF16, 4, 8, 2, 1, FAKE, FAKE, None, None) == INVALID_ARG
    assert lib.moe_route(FAKE, BF16, 4, 8, 2, 1, None, FAKE, None, None) == INVALID_ARG
    assert "non-NULL" in _msg(lib)


def test_route_empty_batch_is_a_noop(lib):
    assert lib.moe_route(None, BF16, 0, 8, 2, 1, None, None, None, None) == OK


def test_dispatch_argument_rules(lib):
    ws = lib.moe_dispatch_workspace_size(1000, 64, 6)
    assert ws > 256
    # x without x_disp
    assert lib.moe_dispatch(FAKE, 10, 8, 2, FAKE, BF16, 64, FAKE, FAKE, FAKE, None, FAKE, ws, None) == INVALID_ARG
    # bad x dtype, zero H
    assert lib.moe_dispatch(FAKE, 10, 8, 2, FAKE, 9, 64, FAKE, FAKE, FAKE, FAKE, FAKE, ws, None) == DTYPE
    assert lib.moe_dispatch(FAKE, 10, 8, 2, FAKE, BF16, 0, FAKE, FAKE, FAKE, FAKE, FAKE, ws, None) == SHAPE
    # workspace too small / misaligned / missing
    assert lib.moe_dispatch(FAKE, 10, 8, 2, None, BF16, 0, FAKE, FAKE, FAKE, None, FAKE, 16, None) == INVALID_ARG
    assert "too small" in _msg(lib)
    assert lib.moe_dispatch(FAKE, 10, 8, 2, None, BF16, 0, FAKE, FAKE, FAKE, None,
                            ctypes.c_void_p(0x10010), 1 << 30, None) == INVALID_ARG
    assert "aligned" in _msg(lib)
    assert lib.moe_dispatch(FAKE, 10, 8, 2, None, BF16, 0, FAKE, FAKE, FAKE, None, None, 1 << 30,
                            None) == INVALID_ARG
    assert lib.moe_dispatch(FAKE, 10, 8, 9, None, BF16, 0, FAKE, FAKE, FAKE, None, FAKE, ws, None) == INVALID_ARG


def test_experts_create_rules(lib):
    h = ctypes.c_void_p()
    # the rules of SwiGluExperts::new: float dtype, non-zero dims
    assert lib.moe_experts_create(FAKE, FAKE, FAKE, 5, 4, 8, 8, ctypes.byref(h)) == DTYPE
    assert lib.moe_experts_create(FAKE, FAKE, FAKE, BF16, 0, 8, 8, ctypes.byref(h)) == SHAPE
    assert lib.moe_experts_create(FAKE, FAKE, FAKE, BF16, 4, 0, 8, ctypes.byref(h)) == SHAPE
    assert lib.moe_experts_create(FAKE, FAKE, FAKE, BF16, 4, 8, 0, ctypes.byref(h)) == SHAPE
    assert "non-zero" in _msg(lib)
    assert lib.moe_experts_create(FAKE, FAKE, FAKE, BF16, 2000, 8, 8, ctypes.byref(h)) == UNSUPPORTED
    assert lib.moe_experts_create(None, FAKE, FAKE, BF16, 4, 8, 8, ctypes.byref(h)) == INVALID_ARG
    assert lib.moe_experts_create(ctypes.c_void_p(0x10002), FAKE, FAKE, BF16, 4, 8, 8,
                                  ctypes.byref(h)) == INVALID_ARG
    assert lib.moe_experts_create(FAKE, FAKE, FAKE, BF16, 4, 8, 8, None) == INVALID_ARG
    assert not h.value


def test_null_handle_rules(lib):
    assert lib.moe_forward(None, FAKE, FAKE, BF16, 4, 2, 1, FAKE, FAKE, 1 << 20, None) == INVALID_ARG
    assert lib.moe_experts_forward(None, FAKE, 4, FAKE, FAKE, FAKE, 1 << 20, None) == INVALID_ARG
    assert lib.moe_forward_workspace_size(None, 4, 2, BF16) == 0
    assert lib.moe_experts_workspace_size(None, 4) == 0
    from top_routing_grouped_fp32_gb300 import _lib
    assert lib.moe_forward_layout(None, 4, 2, BF16, ctypes.byref(_lib.ForwardLayout())) == INVALID_ARG
    lib.moe_experts_destroy(None)  # a no-op


def test_combine_rules(lib):
    ws = lib.moe_combine_workspace_size(10, 2)
    assert ws >= 256 + 10 * 2 * 4
    assert lib.moe_combine(FAKE, 9, FAKE, FAKE, BF16, 10, 2, 64, FAKE, FAKE, ws, None) == DTYPE
    assert lib.moe_combine(FAKE, BF16, FAKE, FAKE, BF16, 10, 0, 64, FAKE, FAKE, ws, None) == INVALID_ARG
    assert lib.moe_combine(FAKE, BF16, FAKE, FAKE, BF16, 10, 2, 0, FAKE, FAKE, ws, None) == SHAPE
    assert lib.moe_combine(FAKE, BF16, None, FAKE, BF16, 10, 2, 64, FAKE, FAKE, ws, None) == INVALID_ARG
    assert lib.moe_combine(FAKE, BF16, FAKE, FAKE, BF16, 10, 2, 64, FAKE, FAKE, 8, None) == INVALID_ARG
    assert lib.moe_combine(None, BF16, None, None, BF16, 0, 2, 64, None, None, 0, None) == OK


def test_workspace_sizes_grow_with_the_problem(lib):
    a = lib.moe_dispatch_workspace_size(256, 64, 6)
    b = lib.moe_dispatch_workspace_size(16384, 64, 6)
    assert b > a > 0
    assert lib.moe_dispatch_workspace_size(10, 0, 1) == 0
    assert lib.moe_combine_workspace_size(-1, 2) == 0


def test_product_has_no_cpu_fallback(tmp_path, monkeypatch):
    """Loading from a path without the library raises instead of degrading."""
    from top_routing_grouped_fp32_gb300 import _lib
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        _lib.load(str(tmp_path / "libmoe_gb300.so"))


def test_product_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "top_routing_grouped_fp32_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), f
                assert "moe_oracle" not in src, f


def _opts(top_k=8, groups=8, sel=4, top_two=1, renorm=1, scale=2.5):
    from top_routing_grouped_fp32_gb300 import _lib
    return _lib.GroupRoutingOptions(top_k, groups, sel, top_two, renorm, scale)


@pytest.mark.parametrize("E,opt,want", [
    (256, dict(), OK),                                   # DeepSeek-style: 8 groups, keep 4, top-two
    (256, dict(groups=0), INVALID_ARG),                  # groups in 1..=128
    (256, dict(groups=256), INVALID_ARG),
    (250, dict(), INVALID_ARG),                          # E divisible by groups
    (256, dict(sel=0), INVALID_ARG),                     # selected groups valid
    (256, dict(sel=9), INVALID_ARG),
    (256, dict(top_k=65), INVALID_ARG),                  # top-k in 1..=64
    (64, dict(top_k=20, groups=8, sel=2), INVALID_ARG),  # top-k <= experts of the kept groups
    (8, dict(top_k=2, groups=8, sel=4, top_two=1), INVALID_ARG),  # top-two needs >= 2 per group
    (256, dict(scale=0.0), INVALID_ARG),                 # scale finite and positive
    (256, dict(scale=float("inf")), INVALID_ARG),
    (2048, dict(), UNSUPPORTED),                         # experts in 1..=1024
])
def test_sigmoid_group_option_rules(lib, E, opt, want):
    o = _opts(**opt)
    # T = 0: only the option rules run, nothing is launched
    st = lib.moe_route_sigmoid_grouped(None, BF16, 0, E, None, ctypes.byref(o), None, None, None, None)
    assert st == want, _msg(lib)
    assert lib.moe_route_sigmoid_grouped(FAKE, BF16, 4, E, None, None, FAKE, FAKE, None, None) == INVALID_ARG


def test_host_pipeline_and_backward_null_rules(lib):
    """The host pipeline and the backward entry points reject null handles and
    bad arguments on the host; destroying a null pipeline is a no-op."""
    out = ctypes.c_void_p()
    assert lib.moe_host_pipeline_workspace_size(None, 16, 2, BF16, 2) == 0
    assert lib.moe_host_pipeline_create(None, 16, 2, BF16, 1, 2, None, 0, None, ctypes.byref(out)) == INVALID_ARG
    assert lib.moe_host_pipeline_submit(None, None, None, None, 4) == INVALID_ARG
    assert lib.moe_host_pipeline_sync(None) == INVALID_ARG
    assert lib.moe_host_pipeline_destroy(None) == OK
    assert lib.moe_experts_backward_workspace_size(None, 16) == 0
    assert lib.moe_experts_backward_with_strategy(None, None, 4, None, None, None, None, None, None, 2,
                                                  None, 0, None) == INVALID_ARG
