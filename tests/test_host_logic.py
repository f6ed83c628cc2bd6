"""Host-side checks that need no GPU: the C ABI exports every entry point
include/rr.h declares, arguments are rejected before anything touches a
device, the tier dispatch picks what the header documents, and the
multi-rank timing of bench.py aggregates correctly over two gloo ranks."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from cluster_reductions_gb300 import build
    build.build()
    import cluster_reductions_gb300 as rr
    return rr.load()


def declared_functions():
    with open(os.path.join(ROOT, "include", "rr.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+char\s*\*|int)\s*(rr_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("rr_reduce", "rr_reduce_ex", "rr_softmax", "rr_layernorm_stats",
                 "rr_cluster_allreduce_selftest", "rr_splitk_combine", "rr_device_status"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    from cluster_reductions_gb300._lib import SIGNATURES
    for name in declared_functions():
        assert hasattr(lib, name), f"librr.so does not export {name}"
        assert name in SIGNATURES, f"binding has no signature for {name}"


def test_arguments_rejected_on_the_host(lib):
    INVALID = 1
    null = None
    assert lib.rr_reduce(null, -1, 4, 0, 0, null, null) == INVALID
    assert lib.rr_reduce(null, 4, -1, 0, 0, null, null) == INVALID
    assert lib.rr_reduce(null, 4, 4, 7, 0, null, null) == INVALID      # bad op
    assert lib.rr_reduce(null, 4, 4, 0, 2, null, null) == INVALID      # bf16 not reducible
    assert lib.rr_reduce(null, 4, 4, 0, 0, null, null) == INVALID      # null pointers
    assert lib.rr_reduce(null, 0, 4, 0, 0, null, null) == 0            # empty: no-op
    buf = (ctypes.c_float * 64)()
    p = ctypes.addressof(buf)
    assert lib.rr_reduce(p, 4, 8, 0, 0, p + 16, null) == INVALID       # out overlaps x
    from cluster_reductions_gb300._lib import rr_reduce_opts
    bad = rr_reduce_opts(1, 0, 0, 5, None)                             # tile width 5
    assert lib.rr_reduce_ex(p, 1, 64, 0, 0, p + 256, null, ctypes.byref(bad)) == INVALID
    bad = rr_reduce_opts(4, 3, 0, 0, None)                             # cluster size 3
    assert lib.rr_reduce_ex(p, 1, 8, 0, 0, p + 64, null, ctypes.byref(bad)) == INVALID
    assert lib.rr_softmax(p, 2, 0, 2, p, null) == INVALID              # cols == 0
    assert lib.rr_softmax(p, 2, 4, 0, p, null) == INVALID              # out overlaps x
    assert lib.rr_layernorm_stats(p, 2, 4, 2, ctypes.c_float(-1.0), p, p, null) == INVALID
    assert lib.rr_splitk_combine(p, p, p, 17, 4, 8, ctypes.c_float(1.0), p, null) == INVALID
    assert lib.rr_splitk_combine(p, p, p, 2, 4, 0, ctypes.c_float(1.0), p, null) == INVALID
    assert lib.rr_splitk_combine(p, p, p, 2, 4, 8, ctypes.c_float(float("inf")), p, null) == INVALID
    assert lib.rr_cluster_allreduce(p, 1, 2, 3, 0, 0, 4, 0, 0, p, null, null) == INVALID
    # iters * clusters * cluster_size * width elements would not fit a size_t
    assert lib.rr_cluster_allreduce(p, 1 << 30, 16, 8, 0, 0, 1 << 30, 0, 0, p + 4096, null,
                                    null) == INVALID
    n = ctypes.c_int64(-1)
    assert lib.rr_cluster_allreduce_selftest(2, 1, 0, 0, 0, 0, 1, null, ctypes.byref(n)) == INVALID
    assert lib.rr_cluster_allreduce_selftest_noalloc(16, 8, 0, 0, 1025, 1, 1, null,
                                                     ctypes.byref(n)) == INVALID
    assert n.value == -1
    assert lib.rr_test_wait_timeout(-1, null) == INVALID
    # reduction over a non-last axis
    from cluster_reductions_gb300._lib import rr_axis_opts
    assert lib.rr_reduce_axis(null, -1, 4, 4, 0, 0, null, null) == INVALID
    assert lib.rr_reduce_axis(null, 2, 4, -4, 0, 0, null, null) == INVALID
    assert lib.rr_reduce_axis(null, 2, 4, 4, 3, 0, null, null) == INVALID    # bad op
    assert lib.rr_reduce_axis(null, 2, 4, 4, 0, 2, null, null) == INVALID    # bf16
    assert lib.rr_reduce_axis(null, 0, 4, 4, 0, 0, null, null) == 0          # empty: no-op
    assert lib.rr_reduce_axis(null, 2, 4, 0, 0, 0, null, null) == 0
    assert lib.rr_reduce_axis(null, 2, 4, 4, 0, 0, null, null) == INVALID    # null pointers
    assert lib.rr_reduce_axis(p, 1, 2, 4, 0, 0, p + 16, null) == INVALID     # out overlaps x
    assert lib.rr_reduce_axis(p + 2, 1, 2, 4, 0, 0, p + 128, null) == INVALID  # x not 4-aligned
    assert lib.rr_reduce_axis(p, 1 << 40, 1 << 40, 4, 0, 0, p + 128, null) == INVALID
    bad = rr_axis_opts(2, 0, 3)                                            # tile width 3
    assert lib.rr_reduce_axis_ex(p, 1, 2, 4, 0, 0, p + 64, null, ctypes.byref(bad)) == INVALID
    bad = rr_axis_opts(4, 5, 0)                                            # cluster size 5
    assert lib.rr_reduce_axis_ex(p, 1, 2, 4, 0, 0, p + 64, null, ctypes.byref(bad)) == INVALID
    bad = rr_axis_opts(9, 0, 0)                                            # no such tier
    assert lib.rr_reduce_axis_ex(p, 1, 2, 4, 0, 0, p + 64, null, ctypes.byref(bad)) == INVALID


def test_status_strings(lib):
    import cluster_reductions_gb300 as rr
    assert rr._lib.status_string(0) == "ok"
    assert rr._lib.status_string(4) == "device wait timed out"
    assert rr._lib.status_string(99) == "unknown status"


@pytest.mark.parametrize("rows,cols,sms,maxc,expect", [
    (1 << 20, 8, 152, 16, ("tiled", 1)),
    (1 << 20, 12, 152, 16, ("tiled", 1)),
    (1 << 20, 16, 152, 16, ("warp", 1)),        # 16 and 29-32: the warp tier
    (5, 0, 152, 16, ("tiled", 1)),
    (1 << 20, 17, 152, 16, ("tiled", 1)),       # 17-28: a thread per row
    (1 << 20, 24, 152, 16, ("tiled", 1)),
    (1 << 20, 28, 152, 16, ("tiled", 1)),
    (1 << 20, 29, 152, 16, ("warp", 1)),
    (1 << 20, 32, 152, 16, ("warp", 1)),
    (8192, 8192, 152, 16, ("block", 1)),
    (1 << 20, 33, 152, 16, ("warp", 1)),       # medium rows: warp segments
    (1 << 20, 64, 152, 16, ("warp", 1)),
    (65536, 1024, 152, 16, ("warp", 1)),
    (152, 4095, 152, 16, ("warp", 1)),
    (16384, 4096, 152, 16, ("block", 1)),
    (151, 1000, 152, 16, ("block", 1)),        # too few rows for warps
    (16, 1 << 24, 152, 16, ("splitk", 16)),
    (16, 1 << 24, 152, 8, ("splitk", 8)),
    (64, 4096, 152, 16, ("splitk", 4)),
    (100, 5000, 152, 16, ("splitk", 2)),
    (151, 4096, 152, 16, ("splitk", 2)),
    (152, 4096, 152, 16, ("block", 1)),
    (16, 4095, 152, 16, ("block", 1)),
    (16, 1 << 24, 152, 1, ("block", 1)),   # no clusters: block tier
    (1, 1 << 20, 148, 16, ("splitk", 16)),
])
def test_tier_dispatch(lib, rows, cols, sms, maxc, expect):
    import cluster_reductions_gb300 as rr
    assert rr.plan_reduce(rows, cols, sms, maxc) == expect


@pytest.mark.parametrize("rows,cols,op,dtype,aligned,maxc,expect", [
    # split-K for a few long rows, the smallest C that covers the SMs
    # (with rows that fit the streamed ring form: as many CTAs per row as
    # there are SMs per row, any cluster size up to 16; one row per SM: a
    # CTA per row)
    (16, 1 << 20, "softmax", "bf16", True, 16, ("splitk", 9)),
    (16, 1 << 20, "layernorm", "bf16", True, 8, ("splitk", 8)),
    (16, 1 << 20, "layernorm", "bf16", True, 16, ("splitk", 16)),   # the rewrite: pow2 rule
    (151, 16384, "lnstats", "bf16", True, 16, ("block", 1)),
    (76, 16384, "lnstats", "bf16", True, 16, ("splitk", 2)),
    (16, 1 << 20, "softmax", "f32", True, 16, ("splitk", 9)),
    (16, 1 << 20 | 4, "softmax", "f32", True, 16, ("splitk", 16)),  # not whole 8-element units
    (100, 1 << 20, "softmax", "bf16", True, 16, ("splitk", 2)),     # 200 MB: beyond L2
    (100, 1 << 20, "lnstats", "bf16", True, 16, ("block", 1)),
    (16, 1 << 20, "softmax", "bf16", True, 1, ("block", 1)),      # no clusters
    (151, 16376, "softmax", "bf16", True, 16, ("block", 1)),      # below 16384 columns
    # a CTA per row once rows fill the SMs and do not fit a warp segment
    (32768, 4096, "softmax", "bf16", True, 16, ("block", 1)),
    (16384, 8192, "layernorm", "bf16", True, 16, ("block", 1)),
    (65536, 2048, "softmax", "f32", True, 16, ("block", 1)),      # 512 vectors > 256
    # warp segments: about 4 vectors per lane, 2 for short rows and the rewrite
    (65536, 2048, "softmax", "bf16", True, 16, ("warp", 32)),
    (65536, 1024, "lnstats", "f32", True, 16, ("warp", 32)),
    (1 << 20, 128, "softmax", "bf16", True, 16, ("warp", 4)),
    (1 << 20, 128, "layernorm", "bf16", True, 16, ("warp", 8)),
    (1 << 20, 64, "lnstats", "bf16", True, 16, ("warp", 4)),
    (1 << 20, 16, "lnstats", "bf16", True, 16, ("warp", 1)),
    (1 << 20, 4, "softmax", "f32", True, 16, ("warp", 1)),
    # enough rows: 4 per SM, 8 for the rewrite
    (607, 256, "softmax", "bf16", True, 16, ("block", 1)),
    (608, 256, "softmax", "bf16", True, 16, ("warp", 8)),
    (1215, 256, "layernorm", "bf16", True, 16, ("block", 1)),
    (1216, 256, "layernorm", "bf16", True, 16, ("warp", 16)),
    # alignment: operands or a width that is not a vector multiple take the
    # chunked warp form (whole 16-byte chunks over the lanes as vectors, the
    # rewrite at 2 a lane) up to 256 chunks, the rewrite's rows of under 32
    # elements the element-wise form (4 elements a lane below 32 lanes)
    (1 << 20, 128, "softmax", "bf16", False, 16, ("warp", 4)),
    (1 << 20, 100, "softmax", "bf16", True, 16, ("warp", 4)),
    (1 << 20, 6, "lnstats", "f32", True, 16, ("warp", 1)),
    (1 << 20, 64, "layernorm", "bf16", False, 16, ("warp", 4)),
    (1 << 20, 65, "layernorm", "bf16", False, 16, ("warp", 4)),
    (1 << 20, 250, "layernorm", "bf16", False, 16, ("warp", 16)),
    (1 << 20, 20, "layernorm", "bf16", False, 16, ("warp", 8)),
    (1 << 20, 1, "softmax", "f32", False, 16, ("warp", 1)),
    (1 << 20, 1025, "lnstats", "f32", False, 16, ("warp", 32)),
    (1 << 20, 2055, "lnstats", "bf16", False, 16, ("warp", 32)),
    (1 << 20, 2057, "lnstats", "bf16", False, 16, ("block", 1)),
    (607, 100, "softmax", "bf16", True, 16, ("block", 1)),
    (608, 100, "softmax", "bf16", True, 16, ("warp", 4)),
    (1215, 100, "layernorm", "bf16", True, 16, ("block", 1)),
    (1216, 100, "layernorm", "bf16", True, 16, ("warp", 8)),
])
def test_rowwise_dispatch(lib, rows, cols, op, dtype, aligned, maxc, expect):
    import torch
    import cluster_reductions_gb300 as rr
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    assert rr.plan_rowwise(rows, cols, op, 152, maxc, dtype=dt, aligned=aligned) == expect


@pytest.mark.parametrize("rows,cols,op,dtype,aligned,maxc,expect", [
    # staged in shared memory: softmax beyond 1024 vectors, layernorm beyond 2048
    (4096, 32768, "softmax", "bf16", True, 16, ("block", 1, "staged")),
    (8192, 16384, "softmax", "bf16", True, 16, ("block", 1, "staged")),
    (8192, 16384, "lnstats", "bf16", True, 16, ("block", 1, "direct")),   # register form
    (16384, 8192, "softmax", "bf16", True, 16, ("block", 1, "direct")),
    (4096, 16384, "layernorm", "f32", True, 16, ("block", 1, "staged")),  # 64 KiB rows
    (304, 524288, "layernorm", "bf16", True, 16, ("splitk", 16, "staged")),
    (608, 262144, "softmax", "bf16", True, 16, ("splitk", 8, "staged")),
    # the statistics of rows beyond the register form: a CTA per row, streamed
    (2048, 65536, "lnstats", "bf16", True, 16, ("block", 1, "ring")),
    (608, 262144, "lnstats", "bf16", True, 16, ("block", 1, "ring")),
    (1216, 131072, "lnstats", "bf16", True, 16, ("block", 1, "ring")),
    (4096, 32768, "lnstats", "bf16", True, 16, ("block", 1, "staged")),   # 64 KiB rows stage
    (4096, 32776, "lnstats", "f32", True, 16, ("block", 1, "ring")),
    (4096, 32772, "lnstats", "f32", True, 16, ("splitk", 2, "staged")),   # not whole 8-element units
    # a few long rows: split-K, streamed
    (16, 1 << 20, "lnstats", "bf16", True, 16, ("splitk", 9, "ring")),
    (16, 1 << 20, "layernorm", "bf16", True, 16, ("splitk", 16, "direct")),  # the rewrite: not
    # not stageable: split-K over global memory
    (304, 524288, "layernorm", "bf16", True, 8, ("splitk", 8, "direct")),  # slices > 96 KiB
    (152, 1 << 20, "softmax", "bf16", True, 16, ("splitk", 16, "direct")),
    (4096, 32767, "softmax", "bf16", True, 16, ("block", 1, "staged")),    # not a vector multiple:
    (4096, 32768, "softmax", "bf16", False, 16, ("block", 1, "staged")),   # misaligned rows staged
    (4096, 50257, "softmax", "bf16", True, 16, ("splitk", 2, "staged")),
    (4096, 49148, "softmax", "bf16", False, 16, ("splitk", 2, "staged")),  # + 8 elements > 96 KiB
    (16384, 4100, "softmax", "bf16", True, 16, ("block", 1, "chunked")),   # 8-byte vector rows:
    (16384, 4092, "softmax", "bf16", True, 16, ("block", 1, "direct")),    # registers up to 1024
    (16384, 8188, "layernorm", "bf16", True, 16, ("block", 1, "direct")),  # 8-byte vectors for
    (16384, 8196, "layernorm", "bf16", True, 16, ("block", 1, "chunked")), # softmax, 2048 for the
    (16384, 4100, "lnstats", "bf16", True, 16, ("block", 1, "direct")),    # statistics / rewrite;
    (16384, 4098, "lnstats", "bf16", True, 16, ("block", 1, "chunked")),   # the statistics and the
    (16384, 4098, "layernorm", "bf16", True, 16, ("block", 1, "chunked")), # rewrite of rows not
    (16384, 4099, "layernorm", "bf16", True, 16, ("block", 1, "chunked")), # 8-byte aligned (or
    (16384, 4095, "layernorm", "f32", True, 16, ("block", 1, "chunked")),  # past the 8-byte form):
    (16384, 4098, "softmax", "bf16", True, 16, ("block", 1, "chunked")),   # chunked registers to
    (8192, 6148, "softmax", "bf16", True, 16, ("block", 1, "staged")),     # (softmax to 4096
    (16384, 4095, "softmax", "f32", True, 16, ("block", 1, "chunked")),    # elements: 512 bf16 /
    (8192, 4105, "softmax", "f32", True, 16, ("block", 1, "staged")),      # 1024 fp32 vectors)
    (8192, 8204, "lnstats", "bf16", True, 16, ("block", 1, "staged")),     # 1024 vectors, then
    (8192, 8190, "lnstats", "bf16", False, 16, ("block", 1, "chunked")),   # staged (the statistics)
    (8192, 8190, "layernorm", "bf16", False, 16, ("block", 1, "chunked")), # or the scalar form
    (8192, 8204, "layernorm", "bf16", True, 16, ("block", 1, "direct")),   # (the rewrite, to 2048),
    (4096, 16396, "layernorm", "bf16", True, 16, ("block", 1, "staged")),  # staged beyond
    (4096, 32768, "softmax", "bf16", True, 1, ("block", 1, "staged")),     # no clusters: C = 1 fits
    (4096, 40000, "softmax", "f32", True, 1, ("block", 1, "direct")),      # no clusters, too long
])
def test_rowwise_staged_dispatch(lib, rows, cols, op, dtype, aligned, maxc, expect):
    import torch
    import cluster_reductions_gb300 as rr
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    assert rr.plan_rowwise(rows, cols, op, 152, maxc, dtype=dt, aligned=aligned,
                           form=True) == expect


@pytest.mark.parametrize("rows,cols,op,dtype,aligned,expect", [
    # fewer rows than SMs, at least 16384 aligned elements whole 8-element
    # units: the grid form, G = floor(4 * 152 / rows) CTAs per row (one
    # wave), slices of at least 2048 elements
    (16, 1 << 20, "softmax", "bf16", True, ("splitk", 38, "grid")),
    (16, 1 << 20, "lnstats", "bf16", True, ("splitk", 38, "grid")),
    (16, 1 << 20, "layernorm", "bf16", True, ("splitk", 38, "grid")),
    (16, 1 << 20, "softmax", "f32", True, ("splitk", 38, "grid")),
    (1, 1 << 20, "softmax", "bf16", True, ("splitk", 512, "grid")),     # slices >= 2048
    (1, 1 << 24, "lnstats", "bf16", True, ("splitk", 608, "grid")),
    (3, 16384, "layernorm", "bf16", True, ("splitk", 8, "grid")),
    (151, 16384, "softmax", "bf16", True, ("splitk", 4, "grid")),
    (64, 262144, "layernorm", "f32", True, ("splitk", 9, "grid")),
    # not the grid form: as many rows as SMs, short rows, misaligned rows
    (152, 16384, "softmax", "bf16", True, ("block", 1, "staged")),
    (16, 8192, "softmax", "bf16", True, ("block", 1, "direct")),
    (16, 65536, "softmax", "bf16", False, ("splitk", 16, "direct")),
    (16, 65540, "softmax", "f32", True, ("splitk", 16, "direct")),       # not whole 8-element units
    # the rewrite of at least as many rows as SMs, rows of 256 KiB and more:
    # ring statistics, then a rewrite pass (two passes); the statistics and
    # softmax of the same rows, shorter rows, misaligned rows: not
    (608, 262144, "layernorm", "bf16", True, ("block", 1, "twopass")),
    (152, 131072, "layernorm", "bf16", True, ("block", 1, "twopass")),
    (1000, 65536, "layernorm", "f32", True, ("block", 1, "twopass")),
    (608, 262144, "lnstats", "bf16", True, ("block", 1, "ring")),
    (608, 262144, "softmax", "bf16", True, ("splitk", 8, "staged")),
    (2048, 65536, "layernorm", "bf16", True, ("splitk", 2, "staged")),    # 128 KiB rows
    (608, 262148, "layernorm", "bf16", True, ("splitk", 8, "staged")),    # not whole units
])
def test_rowwise_grid_dispatch(lib, rows, cols, op, dtype, aligned, expect):
    import torch
    import cluster_reductions_gb300 as rr
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    assert rr.plan_rowwise(rows, cols, op, 152, 16, dtype=dt, aligned=aligned, form=True,
                           with_workspace=True) == expect


def test_rowwise_grid_needs_a_workspace(lib):
    # without a workspace the same shapes plan as before (ring or split-K)
    import cluster_reductions_gb300 as rr
    for op in ("softmax", "lnstats", "layernorm"):
        assert rr.plan_rowwise(16, 1 << 20, op, 152, 16, form=True)[2] != "grid"
        assert rr.plan_rowwise(16, 1 << 20, op, 152, 16, form=True, with_workspace=True)[2] == "grid"


def test_rowwise_warp_reach_for_unaligned_rows(lib):
    # many rows that are not aligned vectors plan onto the warp tier exactly
    # while their whole 16-byte chunks fit 32 lanes x 8 (2055 bf16 / 1027
    # fp32 elements), with a power-of-two lane count; longer rows do not
    import torch
    import cluster_reductions_gb300 as rr
    for dt, top in ((torch.bfloat16, 2055), (torch.float32, 1027)):
        widths = list(range(1, 100)) + [250, 513, 1000, top - 8, top - 1, top, top + 1, top + 9, 4100]
        for cols in widths:
            for op in ("softmax", "lnstats", "layernorm"):
                tier, width = rr.plan_rowwise(1 << 20, cols, op, 152, 16, dtype=dt, aligned=False)
                if cols <= top:
                    assert tier == "warp" and width in (1, 2, 4, 8, 16, 32), (dt, cols, op, tier, width)
                else:
                    assert tier != "warp", (dt, cols, op, tier, width)


def test_rowwise_plan_rejects_bad_arguments(lib):
    t, w = ctypes.c_int(), ctypes.c_int()
    bt, bw = ctypes.byref(t), ctypes.byref(w)
    RR_BF16, RR_I32 = 2, 1
    assert lib.rr_plan_rowwise(-1, 8, RR_BF16, 0, 1, 152, 16, 0, bt, bw, None) == 1
    assert lib.rr_plan_rowwise(8, -8, RR_BF16, 0, 1, 152, 16, 0, bt, bw, None) == 1
    assert lib.rr_plan_rowwise(8, 8, RR_I32, 0, 1, 152, 16, 0, bt, bw, None) == 1
    assert lib.rr_plan_rowwise(8, 8, RR_BF16, 3, 1, 152, 16, 0, bt, bw, None) == 1
    assert lib.rr_plan_rowwise(8, 8, RR_BF16, 0, 1, 0, 16, 0, bt, bw, None) == 1
    assert lib.rr_plan_rowwise(8, 8, RR_BF16, 0, 1, 152, 0, 0, bt, bw, None) == 1
    assert lib.rr_plan_rowwise(8, 8, RR_BF16, 0, 1, 152, 16, 0, None, bw, None) == 1
    assert lib.rr_plan_rowwise(0, 8, RR_BF16, 0, 1, 152, 16, 0, bt, bw, None) == 0
    n = ctypes.c_size_t(0)
    assert lib.rr_rowwise_workspace_size(-1, 8, RR_BF16, 0, ctypes.byref(n)) == 1
    assert lib.rr_rowwise_workspace_size(8, 8, RR_I32, 0, ctypes.byref(n)) == 1
    assert lib.rr_rowwise_workspace_size(8, 8, RR_BF16, 3, ctypes.byref(n)) == 1
    assert lib.rr_rowwise_workspace_size(8, 8, RR_BF16, 0, None) == 1


def test_rowwise_grid_options_rejected_on_the_host(lib):
    # the grid form's options: splits only as split-K without a cluster and
    # with a workspace; a workspace 16-byte aligned, sized, not overlapping
    from cluster_reductions_gb300._lib import rr_rowwise_opts
    buf = (ctypes.c_float * 4096)()
    p = ctypes.addressof(buf)
    p = (p + 255) // 256 * 256
    x, y, ws = p, p + 4096, p + 12288
    SPLITK, BLOCK, AUTO, BF16 = 4, 3, 0, 2

    def sm(o, xp=x, yp=y):
        return lib.rr_softmax_ex(xp, 2, 512, BF16, yp, None, ctypes.byref(o))

    assert sm(rr_rowwise_opts(AUTO, 0, 0, 4, ws, 1024)) == 1        # splits need split-K
    assert sm(rr_rowwise_opts(BLOCK, 0, 0, 4, ws, 1024)) == 1
    assert sm(rr_rowwise_opts(SPLITK, 2, 0, 4, ws, 1024)) == 1      # ... without a cluster
    assert sm(rr_rowwise_opts(SPLITK, 0, 0, 4, None, 0)) == 1       # ... and a workspace
    assert sm(rr_rowwise_opts(SPLITK, 0, 0, -1, ws, 1024)) == 1
    assert sm(rr_rowwise_opts(SPLITK, 0, 0, 1025, ws, 1024)) == 1   # at most 1024 CTAs per row
    assert sm(rr_rowwise_opts(SPLITK, 0, 0, 4, ws + 8, 1024)) == 1  # workspace 16-byte aligned
    assert sm(rr_rowwise_opts(AUTO, 0, 0, 0, ws, 0)) == 1           # a workspace of no bytes
    assert sm(rr_rowwise_opts(SPLITK, 0, 0, 4, x + 64, 1024)) == 1  # overlapping x
    assert sm(rr_rowwise_opts(SPLITK, 0, 0, 4, y + 64, 1024)) == 1  # ... or the output
    assert lib.rr_layernorm_stats_ex(x, 2, 512, BF16, ctypes.c_float(1e-5), y, y + 64, None,
                                     ctypes.byref(rr_rowwise_opts(SPLITK, 0, 0, 4, y + 32, 64))) == 1
    assert lib.rr_layernorm_ex(x, 2, 512, BF16, ctypes.c_float(1e-5), ws, ws + 2048, y, None,
                               None, None,
                               ctypes.byref(rr_rowwise_opts(SPLITK, 0, 0, 4, ws + 1024, 64))) == 1


@pytest.mark.parametrize("shape,align,ws,expect", [
    # (tier, cluster_size, emit_tile_width, tile_rows, splits)
    ((262144, 16, 16), 16, True, ("tiled", 1, 4, 0, 1)),       # many short lines: no combine
    ((262144, 16, 16), 8, True, ("tiled", 1, 2, 0, 1)),        # 8-byte aligned: pairs
    ((32768, 256, 8), 16, True, ("warp", 1, 0, 8, 1)),
    ((32768, 256, 8), 4, True, ("warp", 1, 0, 8, 1)),          # unaligned: scalar lanes
    ((256, 1024, 256), 16, True, ("block", 1, 0, 128, 1)),
    ((1, 8192, 8192), 16, True, ("block", 1, 0, 16, 1)),       # tiles narrowed to 64 bytes
    ((16, 4096, 1024), 16, True, ("block", 1, 0, 32, 1)),
    ((1, 65536, 1024), 16, True, ("splitk", 8, 0, 16, 1)),
    ((64, 65536, 64), 16, True, ("splitk", 2, 0, 16, 1)),
    ((1, 1 << 22, 16), 16, True, ("splitk", 8, 0, 16, 57)),    # one tile: G clusters
    ((1, 1 << 22, 16), 16, False, ("splitk", 16, 0, 16, 1)),   # no workspace: one cluster
    ((1, 1 << 22, 16), 16, True, ("splitk", 8, 0, 16, 57)),
    ((2, 4096, 3), 4, True, ("splitk", 8, 0, 4, 2)),
    ((21845, 1024, 3), 16, True, ("warp", 1, 0, 3, 1)),          # a warp per slab
    ((13107, 1024, 5), 16, True, ("warp", 1, 0, 5, 1)),
    ((1216, 1022, 6), 16, True, ("block", 1, 0, 6, 1)),          # 2-15 slabs per SM: a CTA each
    ((1216, 1021, 6), 16, True, ("block", 1, 0, 8, 1)),          # slabs not 16-byte aligned
    ((21845, 1024, 3), 8, True, ("warp", 1, 0, 4, 1)),           # x 8-byte aligned: lanes
    ((2432, 1024, 7), 16, True, ("warp", 1, 0, 7, 1)),
    ((303, 1024, 3), 16, True, ("splitk", 2, 0, 4, 1)),          # < 2 slabs per SM: tiles
])
def test_axis_dispatch(lib, shape, align, ws, expect):
    import cluster_reductions_gb300 as rr
    p = rr.plan_reduce_axis(*shape, 152, 16, x_align=align, with_workspace=ws)
    got = (p["tier"], p["cluster_size"], p["emit_tile_width"], p["tile_rows"], p["splits"])
    assert got == expect
    outer, _, inner = shape
    assert p["workspace_bytes"] == (p["splits"] * outer * inner * 4 if p["splits"] > 1 else 0)


def test_axis_dispatch_last_axis_and_limits(lib):
    import cluster_reductions_gb300 as rr
    # inner == 1 is the row reduction's plan
    p = rr.plan_reduce_axis(1 << 20, 32, 1, 152, 16)
    assert (p["tier"], p["cluster_size"]) == rr.plan_reduce(1 << 20, 32, 152, 16)
    p = rr.plan_reduce_axis(16, 1 << 24, 1, 152, 16)
    assert (p["tier"], p["cluster_size"]) == ("splitk", 16)
    # no clusters on the device: block, with the split workspace when one tile
    p = rr.plan_reduce_axis(1, 1 << 22, 16, 152, 1)
    assert (p["tier"], p["cluster_size"], p["splits"]) == ("block", 1, 456)
    # G never exceeds 1024 and every split folds at least 256 positions
    p = rr.plan_reduce_axis(1, 1 << 14, 4, 4096, 8)
    assert p["splits"] == (1 << 14) // (8 * 256)
    with pytest.raises(RuntimeError, match="invalid"):
        rr.plan_reduce_axis(1, 2, 3, 152, 16, x_align=2)


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import sys
    sys.path.insert(0, ROOT)
    import bench
    ms = [12.5, 20.0][rank]              # rank 1 is the slow one
    slowest = bench.max_over_ranks(ms, world)
    bench.barrier(world)
    q.put((rank, slowest, bench.job_gbs(1_000_000_000, 10, world, slowest)))
    dist.destroy_process_group()


def test_two_rank_replica_timing_gloo():
    import socket

    import torch.multiprocessing as mp
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, gbs in got:
        assert slowest == 20.0
        # both replicas' bytes over the slowest rank's time: 2 * 10 GB / 20 ms
        assert abs(gbs - 2 * 10 / 0.020) < 1e-9


@pytest.mark.parametrize("epv", [8, 4], ids=["bf16", "f32"])
def test_chunk_image_slots_conflict_free(epv):
    # k_layernorm_ck's gamma / beta image: column j at slot j + j // EPV,
    # 8-byte slots.  A half warp's 16 lanes read one column each, EPV apart
    # (lane t: h + EPV (c0 + t) + e, h the row's head length), so the slots
    # are EPV + 1 apart: 16 distinct 8-byte bank pairs (slot % 16) for every
    # head length, element and starting vector; and every slot stays below
    # the image's cols + cols // EPV + 1.
    for cols in (9, 1029, 2057, 4095, 4099, 8191, 8199):
        nslots = cols + cols // epv + 1
        for h in range(min(epv, cols)):
            nvec = (cols - h) // epv
            for c0 in range(0, max(1, nvec - 15), 16):
                for e in range(epv):
                    js = [h + epv * (c0 + t) + e for t in range(16) if c0 + t < nvec]
                    if not js:
                        continue
                    slots = [j + j // epv for j in js]
                    assert max(slots) < nslots
                    assert len({s % 16 for s in slots}) == len(slots), (cols, h, c0, e)
