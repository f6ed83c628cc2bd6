"""ctypes binding of librr.so (the C ABI declared in include/rr.h).

Argument marshalling only: every step of every operation runs in the CUDA
kernels of librr.so.  There is no CPU fallback: if the library has not been
built, or no CUDA device is present, the calls raise.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "librr.so")

RR_OK, RR_ERR_INVALID, RR_ERR_UNSUPPORTED, RR_ERR_CUDA, RR_ERR_TIMEOUT, RR_ERR_MISMATCH = range(6)
RR_OP_SUM, RR_OP_MAX, RR_OP_MIN = 0, 1, 2
RR_F32, RR_I32, RR_BF16 = 0, 1, 2
RR_TIER_AUTO, RR_TIER_WARP, RR_TIER_TILED, RR_TIER_BLOCK, RR_TIER_SPLITK = range(5)

TIER_NAMES = {RR_TIER_AUTO: "auto", RR_TIER_WARP: "warp", RR_TIER_TILED: "tiled",
              RR_TIER_BLOCK: "block", RR_TIER_SPLITK: "splitk"}


class rr_reduce_opts(ctypes.Structure):
    _fields_ = [("tier", ctypes.c_int), ("cluster_size", ctypes.c_int),
                ("two_slot", ctypes.c_int), ("emit_tile_width", ctypes.c_int),
                ("rank_out", ctypes.c_void_p)]


class rr_rowwise_opts(ctypes.Structure):
    _fields_ = [("tier", ctypes.c_int), ("cluster_size", ctypes.c_int),
                ("lanes_per_row", ctypes.c_int), ("splits", ctypes.c_int),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


class rr_axis_opts(ctypes.Structure):
    _fields_ = [("tier", ctypes.c_int), ("cluster_size", ctypes.c_int),
                ("emit_tile_width", ctypes.c_int), ("tile_rows", ctypes.c_int),
                ("splits", ctypes.c_int), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


class rr_axis_plan(ctypes.Structure):
    _fields_ = [("tier", ctypes.c_int), ("cluster_size", ctypes.c_int),
                ("emit_tile_width", ctypes.c_int), ("tile_rows", ctypes.c_int),
                ("splits", ctypes.c_int), ("workspace_bytes", ctypes.c_size_t)]


# name -> (restype, argtypes), mirroring include/rr.h
_i64, _int, _vp, _f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_float
SIGNATURES = {
    "rr_reduce": (_int, [_vp, _i64, _i64, _int, _int, _vp, _vp]),
    "rr_reduce_ex": (_int, [_vp, _i64, _i64, _int, _int, _vp, _vp,
                            ctypes.POINTER(rr_reduce_opts)]),
    "rr_reduce_splitk_multi": (_int, [_vp, _i64, _i64, _int, _int, _vp, _int, _int, _vp,
                                      ctypes.c_size_t, _vp]),
    "rr_reduce_axis": (_int, [_vp, _i64, _i64, _i64, _int, _int, _vp, _vp]),
    "rr_reduce_axis_ex": (_int, [_vp, _i64, _i64, _i64, _int, _int, _vp, _vp,
                                 ctypes.POINTER(rr_axis_opts)]),
    "rr_plan_reduce_axis": (_int, [_i64, _i64, _i64, _int, _int, _int, _int,
                                   ctypes.POINTER(rr_axis_plan)]),
    "rr_reduce_axis_workspace_size": (_int, [_i64, _i64, _i64, _int,
                                             ctypes.POINTER(ctypes.c_size_t)]),
    "rr_softmax": (_int, [_vp, _i64, _i64, _int, _vp, _vp]),
    "rr_layernorm_stats": (_int, [_vp, _i64, _i64, _int, _f32, _vp, _vp, _vp]),
    "rr_softmax_ex": (_int, [_vp, _i64, _i64, _int, _vp, _vp, ctypes.POINTER(rr_rowwise_opts)]),
    "rr_layernorm_stats_ex": (_int, [_vp, _i64, _i64, _int, _f32, _vp, _vp, _vp,
                                     ctypes.POINTER(rr_rowwise_opts)]),
    "rr_layernorm": (_int, [_vp, _i64, _i64, _int, _f32, _vp, _vp, _vp, _vp, _vp, _vp]),
    "rr_layernorm_ex": (_int, [_vp, _i64, _i64, _int, _f32, _vp, _vp, _vp, _vp, _vp, _vp,
                               ctypes.POINTER(rr_rowwise_opts)]),
    "rr_cluster_allreduce": (_int, [_vp, _int, _int, _int, _int, _int, _int, _int, _i64,
                                    _vp, _vp, _vp]),
    "rr_cluster_allreduce_selftest": (_int, [_int, _int, _int, _int, _int, _int,
                                             ctypes.c_uint64, _vp,
                                             ctypes.POINTER(ctypes.c_int64)]),
    "rr_cluster_allreduce_selftest_noalloc": (_int, [_int, _int, _int, _int, _int, _int,
                                                     ctypes.c_uint64, _vp,
                                                     ctypes.POINTER(ctypes.c_int64)]),
    "rr_cluster_allreduce_selftest_ex": (_int, [_int, _int, _int, _int, _int, _int,
                                                ctypes.c_uint64, _vp,
                                                ctypes.POINTER(ctypes.c_int64), _vp, _vp]),
    "rr_cluster_allreduce_selftest_noalloc_ex": (_int, [_int, _int, _int, _int, _int, _int,
                                                        ctypes.c_uint64, _vp,
                                                        ctypes.POINTER(ctypes.c_int64), _vp,
                                                        _vp]),
    "rr_splitk_combine": (_int, [_vp, _vp, _vp, _int, _i64, _int, _f32, _vp, _vp]),
    "rr_splitk_combine_ex": (_int, [_vp, _vp, _vp, _int, _i64, _int, _f32, _vp, _vp, _int]),
    "rr_device_status": (_int, [_vp]),
    "rr_last_tier": (_int, []),
    "rr_status_string": (ctypes.c_char_p, [_int]),
    "rr_plan_rowwise": (_int, [_i64, _i64, _int, _int, _int, _int, _int, _int,
                               ctypes.POINTER(_int), ctypes.POINTER(_int), ctypes.POINTER(_int)]),
    "rr_rowwise_workspace_size": (_int, [_i64, _i64, _int, _int, ctypes.POINTER(ctypes.c_size_t)]),
    "rr_plan_reduce": (_int, [_i64, _i64, _int, _int, ctypes.POINTER(_int),
                              ctypes.POINTER(_int)]),
    "rr_test_wait_timeout": (_int, [_i64, _vp]),
    "rr_test_inject_error": (_int, [_int]),
}

_lib = None


class RRError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


def load() -> ctypes.CDLL:
    """Load the in-tree librr.so.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"librr.so is not built ({LIB_PATH} missing); run "
                "`python -c 'import __graft_entry__ as g; g.build()'` first")
        lib = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load().rr_status_string(int(status)).decode()


def check(status: int, what: str) -> None:
    if status != RR_OK:
        raise RRError(status, what)
