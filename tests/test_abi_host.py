"""Host-side checks of the C ABI (no GPU): the library builds, loads and exports every
entry point that include/moe_gb300.h declares; size queries follow the documented
layout; argument validation returns the documented status before any device work."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe_gb300.h")


@pytest.fixture(scope="module")
def moe():
    from moe_expert_layer_route_gb300 import _build
    _build.build()
    import moe_expert_layer_route_gb300 as m
    m.lib()
    return m


def declared_functions() -> list[str]:
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", text)))


def test_header_declares_the_block_entry_points():
    names = declared_functions()
    for required in ("moe_route", "moe_dispatch", "moe_expert_ffn", "moe_combine", "moe_forward",
                     "moe_backward", "moe_workspace_size", "moe_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(moe):
    lib = ctypes.CDLL(moe.LIB_PATH)
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding wires each of them
    from moe_expert_layer_route_gb300 import _SIG
    assert set(declared_functions()) == set(_SIG)


def test_status_strings(moe):
    for code in range(-7, 1):
        assert moe.lib().moe_status_string(code)
    assert moe.lib().moe_status_string(123) == b"unknown status"


def test_padded_rows_formula(moe):
    for T, E, k in ((512, 8, 2), (4096, 128, 8), (4096, 32, 4), (65536, 32, 4), (0, 4, 1), (1, 1, 1)):
        s = moe.shape(T, 64, E, k, 64)
        A = T * k
        assert moe.padded_rows(s) == 128 * ((A + 127) // 128 + E)


def test_workspace_sizes_cover_the_layout(moe):
    s = moe.shape(4096, 2880, 32, 4, 2880)
    R = moe.padded_rows(s)
    inf = moe.workspace_size(s, False)
    tr = moe.workspace_size(s, True)
    assert inf >= R * 2880 * 2 * 2 + R * 2880 * 2        # xp, o, h
    assert tr - inf >= R * 2 * 2880 * 2                   # saved gate|up
    assert moe.backward_scratch_size(s) >= R * (2880 + 2 * 2880 + 2880) * 2


@pytest.mark.parametrize("T,d,E,k,f,status", [
    (16, 64, 8, 9, 64, -1),        # k > E
    (16, 64, 300, 2, 64, -2),      # E > 256
    (16, 64, 32, 17, 64, -2),      # k > 16
    (16, 60, 8, 2, 64, -3),        # d not a multiple of 8
    (16, 64, 8, 2, 36, -3),        # f not a multiple of 8
    (-1, 64, 8, 2, 64, -1),        # negative T
    (1 << 29, 64, 8, 8, 64, -5),   # T*k beyond int32
])
def test_shape_validation(moe, T, d, E, k, f, status):
    s = moe.shape(T, d, E, k, f)
    assert moe.lib().moe_workspace_size(s, 1) == 0
    fake = ctypes.c_void_p(0x10000)
    rc = moe.lib().moe_forward(s, fake, fake, fake, fake, fake, 1, None, fake, 1 << 40, None)
    assert rc == status


def test_pointer_and_workspace_validation(moe):
    L = moe.lib()
    s = moe.shape(64, 64, 8, 2, 64)
    good = ctypes.c_void_p(0x10000)
    odd = ctypes.c_void_p(0x10008)
    null = ctypes.c_void_p(None)
    need = L.moe_workspace_size(s, 1)
    assert L.moe_forward(s, null, good, good, good, good, 1, None, good, need, None) == -1
    assert L.moe_forward(s, odd, good, good, good, good, 1, None, good, need, None) == -3
    assert L.moe_forward(s, good, good, good, good, good, 1, None, good, need - 1, None) == -4
    bad_opts = moe._RouteOptions(odd, None)
    assert L.moe_forward(s, good, good, good, good, good, 1, ctypes.byref(bad_opts), good, need,
                         None) == -3
    scratch = L.moe_backward_scratch_size(s)
    assert L.moe_backward(s, good, good, good, good, need, good, good, good, null, good,
                          scratch - 1, None) == -4
    assert L.moe_backward(s, good, good, good, good, need - 1, good, good, good, null, good,
                          scratch, None) == -4
    assert L.moe_backward(s, good, good, good, good, need, good, good, good, odd, good,
                          scratch, None) == -3
    assert L.moe_combine(s, good, good, good, null, None) == -1
    assert L.moe_route(s, good, good, odd, None, None) == -3
    assert L.moe_router_route(s, good, odd, good, good, good, None, None) == -3
    assert L.moe_router_route(s, good, null, good, good, good, None, None) == -1
    assert L.moe_forward_router(s, good, null, good, good, good, good, 1, None, good, need,
                                None) == -1
    assert L.moe_forward_router(s, good, good, odd, good, good, good, 1, None, good, need,
                                None) == -3
    assert L.moe_forward_router(s, good, good, good, good, good, good, 1, None, good, need - 1,
                                None) == -4
    rneed = L.moe_router_backward_scratch_size(s)
    assert rneed >= 16
    assert L.moe_router_backward(s, good, good, good, good, good, good, rneed - 1, None) == -4
    assert L.moe_router_backward(s, good, good, good, good, odd, good, rneed, None) == -3
    assert L.moe_router_backward(s, good, null, good, good, good, good, rneed, None) == -1


def test_router_backward_scratch_is_fixed_by_the_shape(moe):
    L = moe.lib()
    # 2880 columns in 12 blocks of 256, 32 experts in one block: ceil(304 / 12) = 26
    # token splits of 160 tokens, E * d floats each
    assert L.moe_router_backward_scratch_size(moe.shape(4096, 2880, 32, 4, 2880)) == \
        26 * 32 * 2880 * 4
    assert L.moe_router_backward_scratch_size(moe.shape(32, 64, 8, 2, 64)) == 16  # one split
    assert L.moe_router_backward_scratch_size(moe.shape(16, 60, 8, 2, 64)) == 0   # bad shape


def test_views_follow_the_layout(moe):
    s = moe.shape(100, 64, 8, 2, 64)
    v = moe._Views()
    base = 1 << 20
    n = moe.workspace_size(s, True)
    assert moe.lib().moe_workspace_views(s, 1, ctypes.c_void_p(base), n, ctypes.byref(v)) == 0
    ptrs = [getattr(v, f) for f, _ in v._fields_]
    assert all(p is not None and p % 256 == 0 and base <= p < base + n for p in ptrs)
    assert len(set(ptrs)) == len(ptrs)
    assert moe.lib().moe_workspace_views(s, 0, ctypes.c_void_p(base), n, ctypes.byref(v)) == 0
    assert v.gu is None


def test_product_path_refuses_missing_library(monkeypatch, moe):
    monkeypatch.setattr(moe, "_lib", None)
    monkeypatch.setattr(moe, "LIB_PATH", "/nonexistent/libmoe_gb300.so")
    with pytest.raises(RuntimeError):
        moe.lib()


def test_product_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "moe_expert_layer_route_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in text and "from oracle" not in text, fn
    for fn in os.listdir(os.path.join(ROOT, "oracle")):
        if fn.endswith(".py"):
            text = open(os.path.join(ROOT, "oracle", fn)).read()
            assert "moe_expert_layer_route_gb300" not in text, fn
