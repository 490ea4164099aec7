"""The C-ABI library builds, loads without a GPU, and exports every entry
point declared in include/*.h; host-side argument checks run without a GPU."""
import ctypes
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z0-9_]+)\s*\(",
                             text, flags=re.M):
            names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def lib():
    from moe_expert_layer_gb300 import build
    build.build()
    import moe_expert_layer_gb300 as moe
    return moe.load_library()


def test_header_declares_entry_points():
    names = declared_functions()
    assert {"moe_layer_fwd", "moe_layer_workspace_size", "moe_route_sort", "moe_quant_tokens",
            "moe_gmm1", "moe_swiglu_quant", "moe_gmm2", "moe_combine_unpermute"} <= names


def test_library_exports_every_declared_symbol(lib):
    import moe_expert_layer_gb300 as moe
    for name in declared_functions():
        assert hasattr(lib, name), "missing export %s" % name
    assert set(moe.EXPORTS) == declared_functions()


def test_workspace_size_and_shape_checks(lib):
    import moe_expert_layer_gb300 as moe
    ok = moe.dims(128, 7168, 2048, 256, 8)
    assert moe.moe_layer_workspace_size(ok) > 0
    assert moe.moe_layer_host_workspace_size(ok) > moe.moe_layer_workspace_size(ok)
    for bad in [moe.dims(0, 256, 256, 8, 2), moe.dims(16, 100, 256, 8, 2), moe.dims(16, 256, 100, 8, 2),
                moe.dims(16, 256, 256, 8, 9), moe.dims(16, 256, 256, 1024, 2),
                moe.dims(16, 32768, 256, 8, 2), moe.dims(1 << 22, 256, 256, 8, 8)]:
        assert moe.moe_layer_workspace_size(bad) == 0


def test_entry_points_reject_before_touching_the_device(lib):
    import moe_expert_layer_gb300 as moe
    d = moe.dims(16, 256, 256, 8, 2)
    bad = moe.dims(16, 100, 256, 8, 2)
    # invalid shape -> MOE_ERR_SHAPE, NULL pointers -> MOE_ERR_NULL; no GPU needed for either
    assert lib.moe_layer_fwd(ctypes.byref(bad), *([None] * 9), 0, None) == -2
    assert lib.moe_layer_fwd(ctypes.byref(d), *([None] * 9), 0, None) == -1
    assert lib.moe_quant_tokens(ctypes.byref(d), *([None] * 7)) == -1
    assert lib.moe_gmm1(ctypes.byref(bad), *([None] * 8), 0, None) == -2
    assert lib.moe_quant_dispatch(ctypes.byref(d), *([None] * 7)) == -1
    assert lib.moe_front_reorder(ctypes.byref(d), *([None] * 10), 0, None) == -1
    assert lib.moe_front_reorder(ctypes.byref(bad), *([None] * 10), 0, None) == -2
    assert lib.moe_status_string(-5) == b"workspace missing or too small"
    h = ctypes.c_void_p(1234)
    assert lib.moe_layer_graph_create(ctypes.byref(d), *([None] * 9), 0, None, ctypes.byref(h)) == -1
    assert h.value is None  # the handle is cleared on failure
    assert lib.moe_layer_graph_create(ctypes.byref(bad), *([None] * 9), 0, None, ctypes.byref(h)) == -2
    assert lib.moe_layer_graph_create_host(ctypes.byref(d), *([None] * 9), 0, None, ctypes.byref(h)) == -1
    assert lib.moe_layer_graph_launch(None, None) == -1
    assert lib.moe_layer_graph_destroy(None) == 0
    # misaligned pointers -> MOE_ERR_ALIGN
    p = 4096 + 2
    assert lib.moe_layer_fwd(ctypes.byref(d), p, p, p, p, p, p, p, p, 4096, 1 << 30, None) == -3
