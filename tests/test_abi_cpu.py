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


def test_route_sort_workspace_is_one_histogram_per_block(lib):
    """The multi-block sort's scratch: one (E + 1)-bucket int32 histogram per block of
    1024 routes (the scatter blocks scan them themselves), nothing up to 8192 routes."""
    import moe_expert_layer_gb300 as moe
    assert moe.moe_route_sort_workspace_size(moe.dims(1024, 256, 256, 8, 8)) == 0  # 8192 routes: one block
    assert moe.moe_route_sort_workspace_size(moe.dims(8192, 4096, 1408, 64, 6)) == 48 * 65 * 4  # prefill
    assert moe.moe_route_sort_workspace_size(moe.dims(2048, 7168, 2048, 256, 8)) == 16 * 257 * 4  # skewed
    # past 64 blocks of 1024 routes the blocks grow (2048 routes each for 131072 routes)
    assert moe.moe_route_sort_workspace_size(moe.dims(16384, 256, 256, 1023, 8)) == 64 * 1024 * 4


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
    # the pipelined executor: size, depth, NULL and alignment checks before any CUDA call
    assert lib.moe_layer_pipeline_workspace_size(ctypes.byref(d), 2) > lib.moe_layer_workspace_size(ctypes.byref(d))
    assert lib.moe_layer_pipeline_workspace_size(ctypes.byref(d), 0) == 0
    assert lib.moe_layer_pipeline_workspace_size(ctypes.byref(d), 9) == 0
    assert lib.moe_layer_pipeline_workspace_size(ctypes.byref(bad), 2) == 0
    assert lib.moe_layer_pipeline_create(ctypes.byref(d), *([None] * 5), 0, 2, None) == -1
    assert lib.moe_layer_pipeline_create(ctypes.byref(d), *([None] * 5), 0, 2, ctypes.byref(h)) == -1
    assert h.value is None
    assert lib.moe_layer_pipeline_create(ctypes.byref(bad), *([None] * 5), 0, 2, ctypes.byref(h)) == -2
    assert lib.moe_layer_pipeline_create(ctypes.byref(d), *([4096] * 5), 1 << 30, 0, ctypes.byref(h)) == -2
    assert lib.moe_layer_pipeline_create(ctypes.byref(d), *([4096] * 5), 1 << 30, 9, ctypes.byref(h)) == -2
    assert lib.moe_layer_pipeline_create(ctypes.byref(d), 4096 + 4, *([4096] * 4), 1 << 30, 2, ctypes.byref(h)) == -3
    assert lib.moe_layer_pipeline_create(ctypes.byref(d), *([4096] * 4), 4096 + 16, 1 << 30, 2, ctypes.byref(h)) == -3
    assert lib.moe_layer_pipeline_create(ctypes.byref(d), *([4096] * 5), 1024, 2, ctypes.byref(h)) == -5
    t = ctypes.c_uint64()
    assert lib.moe_layer_pipeline_submit(None, 1, 1, 1, 1, ctypes.byref(t)) == -1
    assert lib.moe_layer_pipeline_wait(None, 0) == -1
    assert lib.moe_layer_pipeline_destroy(None) == 0
    # misaligned pointers -> MOE_ERR_ALIGN
    p = 4096 + 2
    assert lib.moe_layer_fwd(ctypes.byref(d), p, p, p, p, p, p, p, p, 4096, 1 << 30, None) == -3


def test_weight_tiles_sizes_and_checks(lib):
    """Tile-buffer sizes follow the documented layout (E * N/128 * KB * 16 KiB, KB =
    2 * ceil(D / 256)); invalid layouts and GEMM numbers are refused on the host."""
    import moe_expert_layer_gb300 as moe
    d = moe.dims(128, 7168, 2048, 256, 8)
    assert moe.moe_weight_tiles_bytes(d, 1) == 256 * (4096 // 128) * 56 * 16384   # GMM1: N = 2I, D = K
    assert moe.moe_weight_tiles_bytes(d, 2) == 256 * (7168 // 128) * 16 * 16384   # GMM2: N = K, D = I
    p = moe.dims(8192, 4096, 1408, 64, 6)
    assert moe.moe_weight_tiles_bytes(p, 2) == 64 * 32 * 12 * 16384   # I = 1408: 11 tiles padded to 12
    assert moe.moe_weight_tiles_bytes(moe.dims(16, 256, 192, 8, 2), 1) == 8 * 3 * 2 * 16384
    assert moe.moe_weight_tiles_bytes(d, 0) == 0 and moe.moe_weight_tiles_bytes(d, 3) == 0
    assert moe.moe_weight_tiles_bytes(moe.dims(16, 100, 256, 8, 2), 1) == 0
    # the layout field: tiles accepted, anything else refused; the size queries ignore it
    t = moe.dims(128, 7168, 2048, 256, 8, moe.WEIGHTS_TILES)
    assert moe.moe_layer_workspace_size(t) == moe.moe_layer_workspace_size(d) > 0
    assert moe.moe_layer_workspace_size(moe.dims(128, 7168, 2048, 256, 8, 2)) == 0
    assert moe.moe_weight_tiles_bytes(moe.dims(128, 7168, 2048, 256, 8, 7), 1) == moe.moe_weight_tiles_bytes(d, 1)
    bad_layout = moe.dims(16, 256, 256, 8, 2, -1)
    assert lib.moe_layer_fwd(ctypes.byref(bad_layout), *([None] * 9), 0, None) == -2
    assert lib.moe_gmm1(ctypes.byref(bad_layout), *([None] * 8), 0, None) == -2
    small = moe.dims(16, 256, 256, 8, 2)
    assert lib.moe_pack_weight_tiles(ctypes.byref(small), 3, 4096, 4096, None) == -2
    assert lib.moe_pack_weight_tiles(ctypes.byref(small), 1, None, 4096, None) == -1
    assert lib.moe_pack_weight_tiles(ctypes.byref(small), 1, 4096 + 8, 4096, None) == -3


def test_binding_refuses_strided_tensors():
    """The binding hands the library raw pointers of dense row-major arrays; a view
    with other strides is refused before anything reaches the library."""
    import torch
    import moe_expert_layer_gb300 as moe
    a = torch.zeros(8, 16, dtype=torch.float16)
    assert moe._p(a) == a.data_ptr()
    assert moe._p(a[2:]) == a[2:].data_ptr()          # a row range is still dense
    assert moe._p(None) is None and moe._p(4096) == 4096
    for bad in (a.t(), a[:, :8], torch.zeros(16, dtype=torch.float16).expand(8, 16)):
        with pytest.raises(ValueError):
            moe._p(bad)


def test_stage_entry_points_check_every_device_pointer_alignment(lib):
    """Index, scale and bounds arrays are checked for 16-byte alignment too, before any
    device call (so this runs without a GPU); optional arguments may be NULL."""
    import moe_expert_layer_gb300 as moe
    d = moe.dims(16, 256, 256, 8, 2)
    A, U = 4096, 4096 + 4  # aligned, 4-byte aligned only (a valid int32/fp32 address)
    assert lib.moe_route_sort(ctypes.byref(d), A, A, A, A, U, None, 0, None) == -3
    assert lib.moe_quant_tokens(ctypes.byref(d), A, None, None, A, U, None, None) == -3
    assert lib.moe_quant_dispatch(ctypes.byref(d), A, A, U, A, A, None, None) == -3
    assert lib.moe_front_reorder(ctypes.byref(d), A, A, A, A, A, A, A, A, U, None, 0, None) == -3
    assert lib.moe_gmm1(ctypes.byref(d), A, None, U, None, A, A, A, A, 256, None) == -3
    assert lib.moe_gmm1(ctypes.byref(d), A, None, A, None, A, U, A, A, 256, None) == -3
    assert lib.moe_swiglu_quant(ctypes.byref(d), A, A, U, A, None, None, A, A, None, None) == -3
    assert lib.moe_gmm2(ctypes.byref(d), A, A, U, A, A, A, A, 256, None) == -3
    assert lib.moe_combine_unpermute(ctypes.byref(d), A, A, A, U, A, None) == -3


def test_noalloc_sort_host_refusals(lib):
    """moe_route_sort_noalloc makes moe_route_sort's host checks (shape, NULL, 16-byte
    alignment of its five device pointers) plus its own size limit, all before any
    device call (so this runs without a GPU)."""
    import moe_expert_layer_gb300 as moe
    d = moe.dims(16, 256, 256, 8, 2)
    A, U = 4096, 4096 + 4
    f = lib.moe_route_sort_noalloc
    assert f(None, A, A, A, A, A, None) == -1
    for bad in (moe.dims(0, 256, 256, 8, 2), moe.dims(16, 256, 256, 8, 9), moe.dims(16, 256, 256, 1024, 2),
                moe.dims(16, 100, 256, 8, 2), moe.dims(16, 256, 256, 8, 2, 5)):
        assert f(ctypes.byref(bad), A, A, A, A, A, None) == -2
    big = moe.dims(moe.ROUTE_SORT_NOALLOC_MAX_ROUTES // 8 + 1, 256, 256, 16, 8)
    assert f(ctypes.byref(big), A, A, A, A, A, None) == -2
    for i in range(5):
        ptrs = [A] * 5
        ptrs[i] = None
        assert f(ctypes.byref(d), *ptrs, None) == -1
        ptrs[i] = U
        assert f(ctypes.byref(d), *ptrs, None) == -3
    # the regular sort refuses the same misaligned pointers the same way
    assert lib.moe_route_sort(ctypes.byref(d), U, A, A, A, A, None, 0, None) == -3


C_CLIENT = r"""
#include <stdio.h>
#include "moe_layer.h"

int main(void) {
  moe_dims_t ok = {128, 7168, 2048, 256, 8, MOE_WEIGHTS_ROWS};
  moe_dims_t bad = {16, 100, 256, 8, 2, MOE_WEIGHTS_ROWS};
  moe_layer_graph_t* g = 0;
  printf("%zu %zu %zu\n", moe_layer_workspace_size(&ok), moe_layer_workspace_size(&bad),
         moe_weight_tiles_bytes(&ok, 1));
  printf("%d %d %d\n", (int)moe_layer_fwd(&bad, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0),
         (int)moe_layer_fwd(&ok, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0),
         (int)moe_layer_graph_create(&ok, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, 0, &g));
  printf("%s|%s\n", moe_status_string(MOE_ERR_SHAPE), moe_status_string(MOE_ERR_TIMEOUT));
  return g != 0;
}
"""


def test_plain_c_client_compiles_links_and_runs(lib, tmp_path):
    """The ABI is consumable from C alone: a C99 program (-pedantic -Werror) includes the
    header, links against the library and gets the documented host-side results without
    a GPU (sizes, shape and null-pointer codes, status strings)."""
    import subprocess
    from moe_expert_layer_gb300 import build
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(build.LIB_PATH)
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror",
                           "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                           "-L", libdir, "-lmoe_layer", "-Wl,-rpath," + libdir])
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    import moe_expert_layer_gb300 as moe
    ok = moe.dims(128, 7168, 2048, 256, 8)
    sizes = [int(v) for v in out[0].split()]
    assert sizes == [moe.moe_layer_workspace_size(ok), 0, 256 * 32 * 56 * 16384]
    assert out[1].split() == ["-2", "-1", "-1"]
    assert out[2] == "unsupported dimensions|device-side wait timed out"
