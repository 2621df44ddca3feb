"""The C-ABI library without a GPU: it builds, loads, exports every entry
point ``include/*.h`` declares, sizes workspaces on the host, and rejects bad
arguments before enqueuing anything.  Only calls that must fail argument
checks are made here, so no kernel is ever launched."""
import ctypes
import glob
import os
import re

import pytest

import combine_moe_dispatch_gb300 as moe
from combine_moe_dispatch_gb300 import Shape, Status, make_shape

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    moe.build()
    return moe.load_library()


def declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(moe_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert "moe_plan" in names and "moe_dispatch" in names and "moe_combine" in names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"
        assert n in moe.SIGNATURES, f"{n} has no binding"


def test_status_strings(lib):
    for s in Status:
        assert moe.status_string(s) and moe.status_string(s) != "unknown status"
    assert moe.status_string(99) == "unknown status"


def test_workspace_size(lib):
    s = make_shape(8, 128, 7168, 256, 8, 1024, moe.PAYLOAD_FP8_E4M3)
    ws = moe.workspace_size(s)
    # 256-byte header + tags + 2 count rows per tile (8 ranks x 1 tile of 128 tokens)
    assert ws == 256 + 256 + 2 * 8 * 256 * 4
    assert moe.workspace_size(make_shape(0, 1, 8, 1, 1, 1)) == 0
    assert moe.workspace_size(make_shape(1, 1, 8, 1, 33, 1)) == 0          # K > 32
    assert moe.workspace_size(make_shape(1, 1, 8, 4096, 1, 1)) == 0        # E > 2048
    assert moe.workspace_size(make_shape(1, 1, 12, 1, 1, 1)) == 0          # H % 8
    assert moe.workspace_size(make_shape(1, 1, 136, 1, 1, 1, moe.PAYLOAD_FP8_E4M3)) == 0
    assert moe.workspace_size(make_shape(1, 1, 136, 1, 1, 1, moe.PAYLOAD_FP8_E4M3_TSCALE)) == 0
    assert moe.workspace_size(make_shape(1, 1, 128, 1, 1, 1, moe.PAYLOAD_FP8_E4M3_TSCALE)) > 0
    assert moe.workspace_size(make_shape(1, 1, 128, 1, 1, 1, 3)) == 0      # no such payload
    assert moe.workspace_size(make_shape(1, 1, 8, 2, 1, 1 << 30)) == 0     # E*cap >= 2^31
    assert moe.workspace_size(make_shape(1, 1, 8, 1, 1, 1, 7)) == 0        # payload


def _p(v):
    return ctypes.c_void_p(v)


def test_host_rejections_enqueue_nothing(lib):
    s = make_shape(2, 4, 256, 8, 2, 8)
    ws_bytes = moe.workspace_size(s)
    A = 0x100000   # aligned fake address: never dereferenced, every call below fails its checks
    sp = ctypes.byref(s)
    # null pointers
    assert lib.moe_plan(sp, None, _p(A), _p(A), _p(A), _p(A), _p(A), ws_bytes, None) == Status.INVALID_ARG
    assert lib.moe_dispatch(sp, None, _p(A), _p(A), _p(A), None, _p(A), None) == Status.INVALID_ARG
    assert lib.moe_combine(sp, _p(A), _p(A), _p(A), None, _p(A), _p(A), None) == Status.INVALID_ARG
    # workspace too small / missing
    assert lib.moe_plan(sp, _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), ws_bytes - 1, None) == Status.WORKSPACE
    assert lib.moe_dispatch(sp, _p(A), _p(A), _p(A), _p(A), None, None, None) == Status.WORKSPACE
    # misaligned pointers
    assert lib.moe_plan(sp, _p(A + 2), _p(A), _p(A), _p(A), _p(A), _p(A), ws_bytes, None) == Status.ALIGNMENT
    assert lib.moe_dispatch(sp, _p(A + 8), _p(A), _p(A), _p(A), None, _p(A), None) == Status.ALIGNMENT
    assert lib.moe_combine(sp, _p(A), _p(A), _p(A), _p(A), _p(A + 4), _p(A), None) == Status.ALIGNMENT
    # fp8 payload needs the scale array
    s8 = make_shape(2, 4, 256, 8, 2, 8, moe.PAYLOAD_FP8_E4M3)
    assert lib.moe_dispatch(ctypes.byref(s8), _p(A), _p(A), _p(A), _p(A), None, _p(A), None) \
        == Status.INVALID_ARG
    # bad shapes
    bad = make_shape(2, 4, 256, 8, 0, 8)
    assert lib.moe_plan(ctypes.byref(bad), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), 1 << 20, None) \
        == Status.INVALID_ARG
    big_k = make_shape(2, 4, 256, 64, 40, 8)
    assert lib.moe_combine(ctypes.byref(big_k), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None) \
        == Status.UNSUPPORTED
    assert lib.moe_plan(None, _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), 1 << 20, None) == Status.INVALID_ARG
    # activation: intermediate size, null pointers, alignment, workspace
    assert lib.moe_silu_mul_quant(sp, 200, _p(A), _p(A), _p(A), _p(A), _p(A), None) == Status.UNSUPPORTED
    assert lib.moe_silu_mul_quant(sp, 0, _p(A), _p(A), _p(A), _p(A), _p(A), None) == Status.INVALID_ARG
    assert lib.moe_silu_mul_quant(sp, 256, None, _p(A), _p(A), _p(A), _p(A), None) == Status.INVALID_ARG
    assert lib.moe_silu_mul_quant(sp, 256, _p(A), _p(A), _p(A + 1), _p(A), _p(A), None) == Status.ALIGNMENT
    assert lib.moe_silu_mul_quant(sp, 256, _p(A), _p(A), _p(A), _p(A), None, None) == Status.WORKSPACE
    # plan + dispatch in one call: the checks of both
    pd = lib.moe_plan_dispatch
    assert pd(sp, None, _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None, _p(A), ws_bytes, None) \
        == Status.INVALID_ARG
    assert pd(sp, _p(A), None, _p(A), _p(A), _p(A), _p(A), _p(A), None, _p(A), ws_bytes, None) \
        == Status.INVALID_ARG
    assert pd(sp, _p(A + 8), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None, _p(A), ws_bytes, None) \
        == Status.ALIGNMENT
    assert pd(sp, _p(A), _p(A + 2), _p(A), _p(A), _p(A), _p(A), _p(A), None, _p(A), ws_bytes, None) \
        == Status.ALIGNMENT
    assert pd(sp, _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None, _p(A), ws_bytes - 1, None) \
        == Status.WORKSPACE
    assert pd(ctypes.byref(s8), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None, _p(A), ws_bytes,
              None) == Status.INVALID_ARG
    assert pd(ctypes.byref(bad), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None, _p(A), 1 << 20,
              None) == Status.INVALID_ARG
    out = ctypes.c_int(0)
    assert lib.moe_read_status(None, None, ctypes.byref(out)) == Status.INVALID_ARG
    assert lib.moe_workspace_init(None, 256, None) == Status.INVALID_ARG
    assert lib.moe_workspace_init(_p(A + 4), 256, None) == Status.ALIGNMENT
    assert lib.moe_workspace_set_debug(None, 1, 0, None) == Status.INVALID_ARG
    # moe_dispatch_ex: moe_dispatch's checks, and no flag bit but EARLY_X
    dx = lib.moe_dispatch_ex
    assert dx(sp, None, _p(A), _p(A), _p(A), None, _p(A), None, 1) == Status.INVALID_ARG
    assert dx(sp, _p(A + 8), _p(A), _p(A), _p(A), None, _p(A), None, 1) == Status.ALIGNMENT
    assert dx(sp, _p(A), _p(A), _p(A), _p(A), None, None, None, 0) == Status.WORKSPACE
    for flags in (2, 4, 1 | 8, 0x80000000):
        assert dx(sp, _p(A), _p(A), _p(A), _p(A), None, _p(A), None, flags) == Status.INVALID_ARG
    assert dx(ctypes.byref(Shape(3, 0, 256, 8, 2, 4, 1)), None, None, None, None, None, None, None,
              moe.DISPATCH_EARLY_X) == Status.OK


@pytest.mark.parametrize("fields,over,under", [
    # (R, T, H, E, K, cap, payload) of a shape just over a limit, and just under it
    ("N*K < 2^31", (1, 1 << 28, 256, 8, 8, 8, 0), (1, (1 << 28) - 1, 256, 8, 8, 8, 0)),
    ("E*cap < 2^31", (1, 4, 256, 2048, 2, 1 << 20, 0), (1, 4, 256, 2048, 2, (1 << 20) - 1, 0)),
    ("E <= 2048", (1, 4, 256, 2049, 2, 8, 0), (1, 4, 256, 2048, 2, 8, 0)),
    ("K <= 32", (1, 4, 256, 64, 33, 8, 0), (1, 4, 256, 64, 32, 8, 0)),
    ("H % 8 == 0", (1, 4, 260, 8, 2, 8, 0), (1, 4, 264, 8, 2, 8, 0)),
    ("fp8: H % 16 == 0", (1, 4, 264, 8, 2, 8, 1), (1, 4, 272, 8, 2, 8, 1)),
    ("fp8, transposed scales: H % 16 == 0", (1, 4, 392, 8, 2, 8, 2), (1, 4, 400, 8, 2, 8, 2)),
])
def test_shape_limits(lib, fields, over, under):
    """Each limit of the shape check, from both sides: just over it the
    limit's own code; just under it the shape passes and the call fails at
    the next check (a null x).  No pointer is dereferenced."""
    A = 0x100000
    s = Shape(*over)
    assert lib.moe_dispatch(ctypes.byref(s), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None) \
        == Status.UNSUPPORTED, fields
    s = Shape(*under)
    assert lib.moe_dispatch(ctypes.byref(s), None, _p(A), _p(A), _p(A), _p(A), _p(A), None) \
        == Status.INVALID_ARG, fields


def test_shape_values_out_of_range(lib):
    A = 0x100000
    for bad in [(0, 4, 256, 8, 2, 8, 0), (1, -1, 256, 8, 2, 8, 0), (1, 4, 0, 8, 2, 8, 0),
                (1, 4, 256, 0, 2, 8, 0), (1, 4, 256, 8, 0, 8, 0), (1, 4, 256, 8, 2, 0, 0),
                (1, 4, 256, 8, 2, 8, 3), (1, 4, 256, 8, 2, 8, -1)]:
        s = Shape(*bad)
        assert lib.moe_dispatch(ctypes.byref(s), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None) \
            == Status.INVALID_ARG, bad


def test_empty_batch_touches_nothing(lib):
    # T = 0: the shape is valid and there is nothing to read or write, so even
    # null buffers are accepted and nothing is enqueued
    s = Shape(3, 0, 256, 8, 2, 4, 1)
    assert lib.moe_dispatch(ctypes.byref(s), None, None, None, None, None, None, None) == Status.OK


def test_router_limits(lib):
    A = 0x100000
    r = lib.moe_router_topk
    for over, code in [((1, 4, 256, 8, 9, 8, 0), Status.UNSUPPORTED),        # K > E
                       ((1, 4, 256, 1025, 8, 8, 0), Status.UNSUPPORTED)]:    # E above 1024
        s = Shape(*over)
        assert r(ctypes.byref(s), _p(A), _p(A), _p(A), None) == code, over
    for under in [(1, 4, 256, 8, 8, 8, 0), (1, 4, 256, 1024, 8, 8, 0)]:
        s = Shape(*under)
        assert r(ctypes.byref(s), None, _p(A), _p(A), None) == Status.INVALID_ARG, under
    s = Shape(1, 4, 256, 64, 8, 8, 0)
    assert r(ctypes.byref(s), _p(A + 2), _p(A), _p(A), None) == Status.ALIGNMENT
    s = Shape(2, 0, 256, 64, 8, 8, 0)
    assert r(ctypes.byref(s), None, None, None, None) == Status.OK      # empty batch


def test_activation_size_limit(lib):
    # E * cap * 2I elements of expert_h must stay below 2^46
    A = 0x100000
    act = lib.moe_silu_mul_quant
    s = Shape(1, 4, 256, 2048, 2, 1 << 20, 0)          # E * cap = 2^31 - too large for the shape check
    assert act(ctypes.byref(s), 128, _p(A), _p(A), _p(A), _p(A), _p(A), _p(A)) == Status.UNSUPPORTED
    s = Shape(1, 4, 256, 1024, 2, 1 << 20, 0)          # E * cap = 2^30: 2^31 * I >= 2^46 from I = 2^15
    assert act(ctypes.byref(s), 1 << 15, _p(A), _p(A), _p(A), _p(A), _p(A), _p(A)) == Status.UNSUPPORTED
    assert act(ctypes.byref(s), (1 << 15) - 128, None, _p(A), _p(A), _p(A), _p(A), _p(A)) \
        == Status.INVALID_ARG


@pytest.mark.parametrize("payload", [0, 1, 2])
def test_plan_noalloc_host_checks(lib, payload):
    A = 0x100000
    na = lib.moe_plan_noalloc
    assert na(None, _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None) == Status.INVALID_ARG
    s = Shape(1, 4, 256, 0, 2, 8, payload)               # no experts
    assert na(ctypes.byref(s), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None) == Status.INVALID_ARG
    s = Shape(1, 4, 256, 4096, 2, 8, payload)            # more experts than supported
    assert na(ctypes.byref(s), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None) == Status.UNSUPPORTED
    s = Shape(64, 4096, 256, 256, 8, 8, payload)         # a workspace above the 1 MiB scratch
    assert moe.workspace_size(s) > (1 << 20)
    assert na(ctypes.byref(s), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None) == Status.WORKSPACE
    s = Shape(1, 4, 256, 8, 2, 8, payload)
    assert na(ctypes.byref(s), _p(A), _p(A), _p(A), _p(A), _p(A), None, None) == Status.INVALID_ARG
    assert na(ctypes.byref(s), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A + 2), None) == Status.ALIGNMENT
    # routes and slots are required unless the batch is empty (T = 0, tested on the GPU)
    assert na(ctypes.byref(s), None, _p(A), _p(A), _p(A), _p(A), _p(A), None) == Status.INVALID_ARG
    assert na(ctypes.byref(s), _p(A), _p(A), _p(A), None, _p(A), _p(A), None) == Status.INVALID_ARG


def test_masked_plan_and_shared_combine_host_checks(lib):
    A = 0x100000
    s = Shape(2, 4, 256, 8, 2, 8, 0)
    ws = moe.workspace_size(s)
    pm = lib.moe_plan_masked
    # num_tokens may be null (every token valid) but, if given, 4-byte aligned
    assert pm(ctypes.byref(s), _p(A), _p(A + 2), _p(A), _p(A), _p(A), _p(A), _p(A), ws, None) \
        == Status.ALIGNMENT
    assert pm(ctypes.byref(s), None, None, _p(A), _p(A), _p(A), _p(A), _p(A), ws, None) \
        == Status.INVALID_ARG
    cs = lib.moe_combine_shared
    # the shared expert's output is required, 16-byte aligned
    assert cs(ctypes.byref(s), _p(A), _p(A), _p(A), _p(A), None, _p(A), _p(A), None) \
        == Status.INVALID_ARG
    assert cs(ctypes.byref(s), _p(A), _p(A), _p(A), _p(A), _p(A + 8), _p(A), _p(A), None) \
        == Status.ALIGNMENT
    # the rest as moe_combine: y aligned, shape checked
    assert cs(ctypes.byref(s), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A + 8), _p(A), None) \
        == Status.ALIGNMENT
    big_k = Shape(2, 4, 256, 64, 40, 8, 0)
    assert cs(ctypes.byref(big_k), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), _p(A), None) \
        == Status.UNSUPPORTED
    # an empty batch needs nothing
    e = Shape(2, 0, 256, 8, 2, 8, 0)
    assert cs(ctypes.byref(e), None, None, None, None, None, None, None, None) == Status.OK


def test_missing_library_fails_loudly(tmp_path):
    saved = moe._lib
    moe._lib = None
    try:
        with pytest.raises(moe.LibraryNotBuilt):
            moe.load_library(str(tmp_path / "nope.so"))
    finally:
        moe._lib = saved


def test_bench_knows_the_fused_limit():
    """bench.py counts one launch for moe_plan_dispatch up to the library's
    fused limit and two beyond it: the two constants must agree."""
    import importlib.util
    src = open(os.path.join(ROOT, "combine_moe_dispatch_gb300", "csrc", "moe_common.cuh")).read()
    m = re.search(r"kFusedMaxEntries\s*=\s*(\d+)", src)
    assert m, "kFusedMaxEntries not found"
    spec = importlib.util.spec_from_file_location("bench_for_test", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert bench.FUSED_MAX_ENTRIES == int(m.group(1))
