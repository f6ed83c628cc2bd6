"""CPU oracle for the row-reduction hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  The product library
(``cluster_reductions_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, fp64, ``-ffp-contract=off``,
serial per row); this module only builds and loads it and marshals numpy
arrays.  Every function states the definition it computes; the sources are
the three Mojo API pages "cluster_allreduce", "reduce" (algorithm/gpu/rowwise)
and "fa4_splitk_reduce_scatter_write".

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
against closed forms, brute force, library routines or hand-worked examples.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

SUM, MAX, MIN = 0, 1, 2
_OPS = {"sum": SUM, "max": MAX, "min": MIN}

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, -O2, no fast-math, no FMA
    contraction).  Returns the library path."""
    stale = (not os.path.exists(_LIB)
             or os.path.getmtime(_LIB) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call([
            "gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
            "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_reduce_f32.argtypes = [vp, i64, i64, i32, vp]
        lib.oracle_reduce_i32.argtypes = [vp, i64, i64, i32, vp]
        lib.oracle_cluster_fold.argtypes = [vp, i32, i32, i32, i32, vp]
        lib.oracle_softmax.argtypes = [vp, i32, i64, i64, vp]
        lib.oracle_layernorm_stats.argtypes = [vp, i32, i64, i64, ctypes.c_double,
                                               vp, vp, vp]
        lib.oracle_splitk_combine.argtypes = [vp, vp, vp, i32, i64, i32,
                                              ctypes.c_float, vp, vp]
        lib.oracle_layernorm.argtypes = [vp, i32, i64, i64, ctypes.c_double, vp, vp,
                                         vp, vp, vp, vp]
        lib.oracle_layernorm.restype = None
        lib.oracle_reduce_axis.argtypes = [vp, i64, i64, i64, i32, i32, vp]
        lib.oracle_reduce_axis.restype = None
        lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        for f in (lib.oracle_reduce_f32, lib.oracle_reduce_i32,
                  lib.oracle_cluster_fold, lib.oracle_softmax,
                  lib.oracle_layernorm_stats, lib.oracle_splitk_combine):
            f.restype = None
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _op(op) -> int:
    return _OPS[op] if isinstance(op, str) else int(op)


def reduce_rows(x: np.ndarray, op) -> np.ndarray:
    """Row-wise reduction of a 2-D array ("reduce" page, state-carrying
    overload: every element of the row folded into one monoid state).

    float32 input: sum -> fp64 sum in index order; max/min -> the exact fp32
    result as float64 (+0 beats -0 for max, -0 beats +0 for min, NaN
    propagates).  int32 input: sum wraps modulo 2^32; max/min exact.
    Empty rows give the identity (0, -inf/INT_MIN, +inf/INT_MAX)."""
    x = np.ascontiguousarray(x)
    assert x.ndim == 2
    rows, cols = x.shape
    lib = _load()
    if x.dtype == np.float32:
        out = np.empty(rows, np.float64)
        lib.oracle_reduce_f32(_ptr(x), rows, cols, _op(op), _ptr(out))
    elif x.dtype == np.int32:
        out = np.empty(rows, np.int32)
        lib.oracle_reduce_i32(_ptr(x), rows, cols, _op(op), _ptr(out))
    else:
        raise TypeError(f"oracle reduce: unsupported dtype {x.dtype}")
    return out


def reduce_axis(x: np.ndarray, op) -> np.ndarray:
    """Reduction over the middle axis of a 3-D [outer, axis, inner] array
    ("reduce" page: the reduce axis is ctx.axis, the other coordinates are
    pinned), folding in axis order.  float32 -> float64 [outer, inner] (sum
    in fp64, max/min exact); int32 -> int32 (sum wraps)."""
    x = np.ascontiguousarray(x)
    assert x.ndim == 3
    outer, axis, inner = x.shape
    if x.dtype == np.float32:
        out = np.empty((outer, inner), np.float64)
        dt = 0
    elif x.dtype == np.int32:
        out = np.empty((outer, inner), np.int32)
        dt = 1
    else:
        raise TypeError(f"oracle reduce_axis: unsupported dtype {x.dtype}")
    _load().oracle_reduce_axis(_ptr(x), outer, axis, inner, _op(op), dt, _ptr(out))
    return out


def cluster_fold(vals: np.ndarray, op) -> np.ndarray:
    """Rank-order fold of per-rank vectors ("cluster_allreduce" page:
    every CTA gathers every peer and folds in rank order).  ``vals`` is
    [C, W] float32 or int32; returns [W] of the same dtype, folded
    left to right in that dtype."""
    vals = np.ascontiguousarray(vals)
    C, W = vals.shape
    dt = {np.dtype(np.float32): 0, np.dtype(np.int32): 1}[vals.dtype]
    out = np.empty(W, vals.dtype)
    _load().oracle_cluster_fold(_ptr(vals), C, W, _op(op), dt, _ptr(out))
    return out


def _x_dtype(x: np.ndarray) -> int:
    if x.dtype == np.float32:
        return 0
    if x.dtype == np.uint16:      # raw bf16 bit patterns
        return 2
    raise TypeError(f"oracle: expected float32 or uint16 (bf16 bits), got {x.dtype}")


def softmax(x: np.ndarray) -> np.ndarray:
    """Two-pass row softmax in fp64 ("reduce" page: pass 1 reduces
    (max, sum), pass 2 maps).  ``x`` is float32 or uint16 holding bf16
    bit patterns; returns float64 [rows, cols]."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    y = np.empty((rows, cols), np.float64)
    _load().oracle_softmax(_ptr(x), _x_dtype(x), rows, cols, _ptr(y))
    return y


def layernorm_stats(x: np.ndarray, eps: float = 1e-5):
    """Per-row mean, population variance and rstd = 1/sqrt(var + eps) in
    fp64, variance taken about the mean in a second pass.  Returns
    (mean, var, rstd) as float64 [rows]."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    mean = np.empty(rows, np.float64)
    var = np.empty(rows, np.float64)
    rstd = np.empty(rows, np.float64)
    _load().oracle_layernorm_stats(_ptr(x), _x_dtype(x), rows, cols, float(eps),
                                   _ptr(mean), _ptr(var), _ptr(rstd))
    return mean, var, rstd


def layernorm(x: np.ndarray, gamma: np.ndarray, beta: np.ndarray, eps: float = 1e-5):
    """Layernorm rewrite ("reduce" page: the map pass after the statistics):
    y = (x - mean) * rstd * gamma + beta per row, fp64, then rounded once to
    bf16.  x float32 or uint16 (bf16 bits) [rows, cols]; gamma, beta float32
    [cols].  Returns (y_f64, y_bf16_bits, mean, rstd)."""
    x = np.ascontiguousarray(x)
    rows, cols = x.shape
    g = np.ascontiguousarray(gamma, dtype=np.float32)
    b = np.ascontiguousarray(beta, dtype=np.float32)
    assert g.shape == (cols,) and b.shape == (cols,)
    y64 = np.empty((rows, cols), np.float64)
    y16 = np.empty((rows, cols), np.uint16)
    mean = np.empty(rows, np.float64)
    rstd = np.empty(rows, np.float64)
    _load().oracle_layernorm(_ptr(x), _x_dtype(x), rows, cols, float(eps), _ptr(g), _ptr(b),
                             _ptr(y64), _ptr(y16), _ptr(mean), _ptr(rstd))
    return y64, y16, mean, rstd


def splitk_combine(O: np.ndarray, m: np.ndarray, l: np.ndarray,
                   scale_log2e: float):
    """Split-K attention-output combine ("fa4_splitk_reduce_scatter_write"
    page).  O [P, rows, D], m and l [P, rows] float32.  Returns
    (out_f64 [rows, D], out_bf16_bits [rows, D] uint16) where
    out = sum_p w_p O_p / sum_p w_p l_p, w_p = 2^((m_p - max m) * scale_log2e),
    rounded once to bf16 nearest-even; rows with max m = -inf or L = 0 give 0."""
    O = np.ascontiguousarray(O, dtype=np.float32)
    m = np.ascontiguousarray(m, dtype=np.float32)
    l = np.ascontiguousarray(l, dtype=np.float32)
    P, rows, D = O.shape
    assert m.shape == (P, rows) and l.shape == (P, rows) and 1 <= P <= 64
    out64 = np.empty((rows, D), np.float64)
    out16 = np.empty((rows, D), np.uint16)
    _load().oracle_splitk_combine(_ptr(O), _ptr(m), _ptr(l), P, rows, D,
                                  ctypes.c_float(scale_log2e), _ptr(out64),
                                  _ptr(out16))
    return out64, out16


def f64_to_bf16_bits(x: float) -> int:
    """Round one double to bf16 (nearest-even, directly from fp64)."""
    return int(_load().oracle_f64_to_bf16(float(x)))
