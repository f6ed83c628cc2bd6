"""cluster_reductions_gb300 -- deterministic row-wise monoid reductions on
NVIDIA GB300 (sm_103a), behind the C ABI of librr.so (include/rr.h).

Python names mirror the C entry points.  Tensors are torch tensors used only
as device memory (and their current CUDA stream); every computation runs in
the library's CUDA kernels.  Passing CPU tensors stages them through device
memory (host -> device copy, kernel, device -> host copy) on the current
stream, which is what an end-to-end call from host buffers costs.
"""
from __future__ import annotations

import ctypes
import functools
from typing import Optional, Tuple

import numpy as np
import torch

from . import _lib
from ._lib import (RR_BF16, RR_F32, RR_I32, RR_OP_MAX, RR_OP_MIN, RR_OP_SUM,  # noqa: F401
                   RR_TIER_AUTO, RR_TIER_BLOCK, RR_TIER_SPLITK, RR_TIER_TILED,
                   RR_TIER_WARP, RRError, TIER_NAMES, check, load)

_OPS = {"sum": RR_OP_SUM, "max": RR_OP_MAX, "min": RR_OP_MIN}
_TIERS = {None: RR_TIER_AUTO, "auto": RR_TIER_AUTO, "warp": RR_TIER_WARP,
          "tiled": RR_TIER_TILED, "serial": RR_TIER_TILED, "block": RR_TIER_BLOCK,
          "splitk": RR_TIER_SPLITK}
_DT = {torch.float32: RR_F32, torch.int32: RR_I32, torch.bfloat16: RR_BF16}


def _op(op) -> int:
    return _OPS[op] if isinstance(op, str) else int(op)


def _stream() -> int:
    return torch.cuda.current_stream().cuda_stream


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _as_2d(x: torch.Tensor) -> torch.Tensor:
    if x.dim() == 1:
        x = x.unsqueeze(0)
    if x.dim() != 2:
        raise ValueError(f"expected a 2-D [rows, cols] tensor, got shape {tuple(x.shape)}")
    if not x.is_contiguous():
        raise ValueError("expected a contiguous (row-major) tensor")
    return x


def _device_of(x: torch.Tensor) -> torch.device:
    if x.is_cuda:
        return x.device
    return torch.device("cuda", torch.cuda.current_device())


def _to_device(x: torch.Tensor) -> torch.Tensor:
    return x if x.is_cuda else x.to(_device_of(x), non_blocking=True)


def _to_host(y: torch.Tensor, like: torch.Tensor) -> torch.Tensor:
    if like.is_cuda:
        return y
    h = torch.empty(y.shape, dtype=y.dtype, pin_memory=like.is_pinned())
    h.copy_(y, non_blocking=like.is_pinned())
    return h


def _on_input_device(fn):
    """Run a binding call with the first argument's GPU as the current device
    (the library launches on the current device and stream)."""
    @functools.wraps(fn)
    def call(x, *args, **kwargs):
        if isinstance(x, torch.Tensor) and x.is_cuda and x.device.index != torch.cuda.current_device():
            with torch.cuda.device(x.device):
                return fn(x, *args, **kwargs)
        return fn(x, *args, **kwargs)
    return call


def _same_device(device, *ts):
    for t in ts:
        if t is not None and t.is_cuda and t.device != device:
            raise ValueError(f"tensor on {t.device}, the input on {device}")


def _out_buf(out: Optional[torch.Tensor], shape, dtype, device) -> torch.Tensor:
    """Device buffer a kernel writes: `out` itself when it is a CUDA tensor,
    else a fresh device tensor (copied into a CPU `out` by _deliver).  A given
    `out` must have exactly the result's shape and dtype and be contiguous:
    the kernels write every element of it and nothing else."""
    shape = tuple(shape)
    if out is not None:
        if tuple(out.shape) != shape or out.dtype != dtype or not out.is_contiguous():
            raise ValueError(f"out must be a contiguous {dtype} tensor of shape {shape}, "
                             f"got {out.dtype} {tuple(out.shape)}")
        if out.is_cuda:
            if out.device != device:
                raise ValueError(f"out is on {out.device}, the input on {device}")
            return out
    return torch.empty(shape, dtype=dtype, device=device)


def _deliver(y: torch.Tensor, out: Optional[torch.Tensor], like: torch.Tensor) -> torch.Tensor:
    """The result where the caller asked for it.  A CPU `out` receives a
    copy, asynchronous when it is pinned (like torch's non_blocking copies:
    valid once the current stream has passed this point); with no `out`, a
    CPU input gets a CPU result the same way."""
    if out is not None:
        if not out.is_cuda:
            out.copy_(y, non_blocking=out.is_pinned())
        return out
    return _to_host(y, like)


@_on_input_device
def reduce(x: torch.Tensor, op="sum", *, out: Optional[torch.Tensor] = None, tier=None,
           cluster_size: int = 0, emit_tile_width: int = 0,
           rank_out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """rr_reduce / rr_reduce_ex: reduce every row of a [rows, cols] fp32 or
    int32 tensor with sum, max or min.  Returns [rows] of the same dtype."""
    x = _as_2d(x)
    xd = _to_device(x)
    rows, cols = xd.shape
    dt = _DT.get(xd.dtype)
    if dt not in (RR_F32, RR_I32):
        raise TypeError(f"reduce: dtype {xd.dtype} not supported (float32, int32)")
    o = _out_buf(out, (rows,), xd.dtype, xd.device)
    lib = load()
    if tier is None and cluster_size == 0 and emit_tile_width == 0 and rank_out is None:
        st = lib.rr_reduce(_ptr(xd), rows, cols, _op(op), dt, _ptr(o), _stream())
    else:
        opts = _lib.rr_reduce_opts(_TIERS[tier] if not isinstance(tier, int) else tier,
                                   int(cluster_size), 0, int(emit_tile_width), _ptr(rank_out))
        st = lib.rr_reduce_ex(_ptr(xd), rows, cols, _op(op), dt, _ptr(o), _stream(),
                              ctypes.byref(opts))
    check(st, "rr_reduce")
    return _deliver(o, out, x)


@_on_input_device
def reduce_splitk_multi(x: torch.Tensor, op="sum", *, cluster_size: int = 0,
                        clusters_per_row: int = 0, out: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """rr_reduce_splitk_multi: the split-K reduction with several clusters
    per row (for very few, very long rows).  The workspace (rows * G
    elements) is allocated here when not given."""
    x = _as_2d(x)
    xd = _to_device(x)
    rows, cols = xd.shape
    dt = _DT.get(xd.dtype)
    if dt not in (RR_F32, RR_I32):
        raise TypeError(f"reduce: dtype {xd.dtype} not supported (float32, int32)")
    o = _out_buf(out, (rows,), xd.dtype, xd.device)
    g = clusters_per_row if clusters_per_row > 0 else 1024
    ws = workspace if workspace is not None else torch.empty(max(1, rows * g), dtype=torch.int32,
                                                             device=xd.device)
    check(load().rr_reduce_splitk_multi(_ptr(xd), rows, cols, _op(op), dt, _ptr(o),
                                        int(cluster_size), int(clusters_per_row), _ptr(ws),
                                        ws.numel() * ws.element_size(), _stream()),
          "rr_reduce_splitk_multi")
    return _deliver(o, out, x)


@_on_input_device
def reduce_axis(x: torch.Tensor, op="sum", dim: int = 0, *, out: Optional[torch.Tensor] = None,
                tier=None, cluster_size: int = 0, emit_tile_width: int = 0, tile_rows: int = 0,
                splits: int = 0, workspace: Optional[torch.Tensor] = None) -> torch.Tensor:
    """rr_reduce_axis_ex: reduce a contiguous fp32 or int32 tensor over
    dimension `dim` (viewed as [outer, axis, inner]).  Returns the tensor's
    shape without `dim`, same dtype.  The workspace the automatic plan asks
    for (rr_reduce_axis_workspace_size; shapes with too few output tiles to
    cover the GPU) is allocated here when not given."""
    if not x.is_contiguous():
        raise ValueError("reduce_axis: x must be contiguous")
    if x.dim() == 0:
        raise ValueError("reduce_axis: x must have at least one dimension")
    dim = dim % x.dim()
    shape = tuple(x.shape)
    outer = 1
    for n in shape[:dim]:
        outer *= n
    inner = 1
    for n in shape[dim + 1:]:
        inner *= n
    axis = shape[dim]
    xd = _to_device(x)
    dt = _DT.get(xd.dtype)
    if dt not in (RR_F32, RR_I32):
        raise TypeError(f"reduce_axis: dtype {xd.dtype} not supported (float32, int32)")
    oshape = shape[:dim] + shape[dim + 1:]
    o = _out_buf(out, oshape, xd.dtype, xd.device)
    lib = load()
    ws = workspace
    if ws is None and inner > 1 and (tier is None or splits > 1):
        addr = xd.data_ptr()
        align = 16 if addr % 16 == 0 else (8 if addr % 8 == 0 else 4)
        nbytes = ctypes.c_size_t(0)
        check(lib.rr_reduce_axis_workspace_size(outer, axis, inner, align, ctypes.byref(nbytes)),
              "rr_reduce_axis_workspace_size")
        need = nbytes.value
        if splits > 1:
            need = max(need, splits * outer * inner * 4)
        if need:
            ws = torch.empty((need + 3) // 4, dtype=torch.int32, device=xd.device)
    opts = _lib.rr_axis_opts(_TIERS[tier] if not isinstance(tier, int) else tier,
                             int(cluster_size), int(emit_tile_width), int(tile_rows), int(splits),
                             _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size())
    st = lib.rr_reduce_axis_ex(_ptr(xd), outer, axis, inner, _op(op), dt, _ptr(o), _stream(),
                               ctypes.byref(opts))
    check(st, "rr_reduce_axis")
    return _deliver(o, out, x)


def _rowwise_opts(tier, cluster_size, lanes_per_row=0, splits=0, ws=None):
    if tier is None and not cluster_size and not lanes_per_row and not splits and ws is None:
        return None
    return ctypes.byref(_lib.rr_rowwise_opts(_TIERS[tier] if not isinstance(tier, int) else tier,
                                             int(cluster_size), int(lanes_per_row), int(splits),
                                             _ptr(ws),
                                             0 if ws is None else ws.numel() * ws.element_size()))


@functools.lru_cache(maxsize=256)
def _row_ws_bytes(device: int, rows: int, cols: int, dt: int, row_op: int) -> int:
    n = ctypes.c_size_t(0)
    with torch.cuda.device(device):
        check(load().rr_rowwise_workspace_size(rows, cols, dt, row_op, ctypes.byref(n)),
              "rr_rowwise_workspace_size")
    return n.value


def _row_ws(xd: torch.Tensor, row_op: str, tier, splits: int, workspace):
    """The workspace of a row op (the grid form's partial states, the
    layernorm two-pass form's statistics): the
    caller's tensor, none (workspace=False), or one of the size the
    automatic plan (or a forced `splits`) asks for, allocated here on the
    current stream."""
    if workspace is False:
        return None
    if workspace is not None:
        return workspace
    rows, cols = xd.shape
    if splits > 0:
        need = rows * splits * 16
    elif tier is None or tier == "auto":
        if xd.data_ptr() % 16 or rows == 0:
            return None
        need = _row_ws_bytes(xd.device.index, rows, cols, _DT[xd.dtype], _ROW_OPS[row_op])
    else:
        return None
    if not need:
        return None
    return torch.empty((need + 15) // 16 * 4, dtype=torch.int32, device=xd.device)


@_on_input_device
def softmax(x: torch.Tensor, *, out: Optional[torch.Tensor] = None, tier=None,
            cluster_size: int = 0, lanes_per_row: int = 0, splits: int = 0,
            workspace=None) -> torch.Tensor:
    """rr_softmax / rr_softmax_ex: row softmax of a bf16 or fp32 [rows, cols]
    tensor, fp32 out.  tier: None/"auto", "warp", "block" or "splitk";
    cluster_size for split-K, lanes_per_row for the warp tier; splits (with
    tier "splitk") forces the grid form with that many CTAs per row.
    workspace: None (allocated here when the plan wants one), False (none),
    or a device tensor."""
    x = _as_2d(x)
    xd = _to_device(x)
    rows, cols = xd.shape
    dt = _DT.get(xd.dtype)
    if dt not in (RR_BF16, RR_F32):
        raise TypeError(f"softmax: dtype {xd.dtype} not supported (bfloat16, float32)")
    o = _out_buf(out, (rows, cols), torch.float32, xd.device)
    ws = _row_ws(xd, "softmax", tier, splits, workspace)
    opts = _rowwise_opts(tier, cluster_size, lanes_per_row, splits, ws)
    if opts is None:
        st = load().rr_softmax(_ptr(xd), rows, cols, dt, _ptr(o), _stream())
    else:
        st = load().rr_softmax_ex(_ptr(xd), rows, cols, dt, _ptr(o), _stream(), opts)
    check(st, "rr_softmax")
    return _deliver(o, out, x)


@_on_input_device
def layernorm_stats(x: torch.Tensor, eps: float = 1e-5, *,
                    mean: Optional[torch.Tensor] = None,
                    rstd: Optional[torch.Tensor] = None, tier=None,
                    cluster_size: int = 0, lanes_per_row: int = 0, splits: int = 0,
                    workspace=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """rr_layernorm_stats / rr_layernorm_stats_ex: per-row mean and
    1/sqrt(var + eps), fp32.  tier: None/"auto", "warp", "block" or
    "splitk"; splits / workspace as for softmax."""
    x = _as_2d(x)
    xd = _to_device(x)
    rows, cols = xd.shape
    dt = _DT.get(xd.dtype)
    if dt not in (RR_BF16, RR_F32):
        raise TypeError(f"layernorm_stats: dtype {xd.dtype} not supported")
    mu = _out_buf(mean, (rows,), torch.float32, xd.device)
    rs = _out_buf(rstd, (rows,), torch.float32, xd.device)
    ws = _row_ws(xd, "lnstats", tier, splits, workspace)
    opts = _rowwise_opts(tier, cluster_size, lanes_per_row, splits, ws)
    if opts is None:
        st = load().rr_layernorm_stats(_ptr(xd), rows, cols, dt, float(eps), _ptr(mu), _ptr(rs),
                                       _stream())
    else:
        st = load().rr_layernorm_stats_ex(_ptr(xd), rows, cols, dt, float(eps), _ptr(mu),
                                          _ptr(rs), _stream(), opts)
    check(st, "rr_layernorm_stats")
    return _deliver(mu, mean, x), _deliver(rs, rstd, x)


@_on_input_device
def layernorm(x: torch.Tensor, gamma: torch.Tensor, beta: torch.Tensor, eps: float = 1e-5, *,
              out: Optional[torch.Tensor] = None, mean: Optional[torch.Tensor] = None,
              rstd: Optional[torch.Tensor] = None, tier=None,
              cluster_size: int = 0, lanes_per_row: int = 0, splits: int = 0,
              workspace=None) -> torch.Tensor:
    """rr_layernorm / rr_layernorm_ex: bf16 (x - mean) * rstd * gamma + beta per
    row of a bf16 or fp32 [rows, cols] tensor; gamma, beta fp32 [cols].
    mean / rstd (fp32 [rows]) are filled when given; splits / workspace as
    for softmax."""
    x = _as_2d(x)
    xd = _to_device(x)
    rows, cols = xd.shape
    dt = _DT.get(xd.dtype)
    if dt not in (RR_BF16, RR_F32):
        raise TypeError(f"layernorm: dtype {xd.dtype} not supported")
    if gamma.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("gamma and beta must be float32")
    if gamma.numel() != cols or beta.numel() != cols:
        raise ValueError("gamma and beta must have cols elements")
    _same_device(xd.device, gamma, beta)
    gd, bd = _to_device(gamma.contiguous()), _to_device(beta.contiguous())
    o = _out_buf(out, (rows, cols), torch.bfloat16, xd.device)
    mu = None if mean is None else _out_buf(mean, (rows,), torch.float32, xd.device)
    rs = None if rstd is None else _out_buf(rstd, (rows,), torch.float32, xd.device)
    ws = _row_ws(xd, "layernorm", tier, splits, workspace)
    opts = _rowwise_opts(tier, cluster_size, lanes_per_row, splits, ws)
    args = (_ptr(xd), rows, cols, dt, float(eps), _ptr(gd), _ptr(bd), _ptr(o), _ptr(mu),
            _ptr(rs), _stream())
    st = load().rr_layernorm(*args) if opts is None else load().rr_layernorm_ex(*args, opts)
    check(st, "rr_layernorm")
    if mu is not None:
        _deliver(mu, mean, x)
    if rs is not None:
        _deliver(rs, rstd, x)
    return _deliver(o, out, x)


@_on_input_device
def cluster_allreduce(vals: torch.Tensor, op="sum", *, two_slot: bool = False,
                      skew_cycles: int = 0, res: Optional[torch.Tensor] = None,
                      mismatches: Optional[torch.Tensor] = None) -> torch.Tensor:
    """rr_cluster_allreduce: vals is [iters, clusters, C, W] fp32 or int32 on
    the device; returns res of the same shape (each rank's combined copy).
    `mismatches` (int64 [1] on the device) accumulates per-thread bit
    differences from the rank-order fold."""
    if vals.dim() != 4 or not vals.is_contiguous() or not vals.is_cuda:
        raise ValueError("vals must be a contiguous CUDA tensor [iters, clusters, C, W]")
    iters, clusters, C, W = vals.shape
    dt = _DT.get(vals.dtype)
    if dt not in (RR_F32, RR_I32):
        raise TypeError("cluster_allreduce: float32 or int32 values")
    r = res if res is not None else torch.empty_like(vals)
    check(load().rr_cluster_allreduce(_ptr(vals), clusters, C, W, _op(op), dt, iters,
                                      1 if two_slot else 0, int(skew_cycles), _ptr(r),
                                      _ptr(mismatches), _stream()), "rr_cluster_allreduce")
    return r


def cluster_allreduce_selftest(cluster_size: int, width: int = 1, op="sum",
                               dtype: torch.dtype = torch.float32, iters: int = 1000,
                               two_slot: bool = True, seed: int = 1) -> int:
    """rr_cluster_allreduce_selftest (blocking): number of values that differ
    from the rank-order fold (0 on success)."""
    n = ctypes.c_int64(-1)
    st = load().rr_cluster_allreduce_selftest(int(cluster_size), int(width), _op(op),
                                              _DT[dtype], int(iters), 1 if two_slot else 0,
                                              int(seed), _stream(), ctypes.byref(n))
    if st not in (_lib.RR_OK, _lib.RR_ERR_MISMATCH):
        check(st, "rr_cluster_allreduce_selftest")
    return int(n.value)


def cluster_allreduce_selftest_noalloc(cluster_size: int, width: int = 1, op="sum",
                                       dtype: torch.dtype = torch.float32, iters: int = 1000,
                                       two_slot: bool = True, seed: int = 1) -> int:
    """rr_cluster_allreduce_selftest_noalloc (blocking): the same self-test as
    cluster_allreduce_selftest, run out of the library's fixed device array
    instead of freshly allocated memory, for callers that cannot allocate.
    iters * 2 * cluster_size * width must be at most 262144."""
    n = ctypes.c_int64(-1)
    st = load().rr_cluster_allreduce_selftest_noalloc(int(cluster_size), int(width), _op(op),
                                                      _DT[dtype], int(iters),
                                                      1 if two_slot else 0, int(seed),
                                                      _stream(), ctypes.byref(n))
    if st not in (_lib.RR_OK, _lib.RR_ERR_MISMATCH):
        check(st, "rr_cluster_allreduce_selftest_noalloc")
    return int(n.value)


def cluster_allreduce_selftest_dump(cluster_size: int, width: int = 1, op="sum",
                                    dtype: torch.dtype = torch.float32, iters: int = 1000,
                                    two_slot: bool = True, seed: int = 1,
                                    noalloc: bool = False):
    """rr_cluster_allreduce_selftest_ex (or its no-allocation twin, noalloc
    = True), blocking: (mismatch count, inputs, every rank's result), the
    arrays numpy [iters, 2, cluster_size, width] of `dtype`, for a check of
    the run on the host."""
    np_dt = {torch.float32: np.float32, torch.int32: np.int32}[dtype]
    shape = (int(iters), 2, int(cluster_size), int(width))
    vals = np.zeros(shape, np_dt)
    res = np.zeros(shape, np_dt)
    n = ctypes.c_int64(-1)
    fn = (load().rr_cluster_allreduce_selftest_noalloc_ex if noalloc
          else load().rr_cluster_allreduce_selftest_ex)
    st = fn(int(cluster_size), int(width), _op(op), _DT[dtype], int(iters), 1 if two_slot else 0,
            int(seed), _stream(), ctypes.byref(n), vals.ctypes.data, res.ctypes.data)
    if st not in (_lib.RR_OK, _lib.RR_ERR_MISMATCH):
        check(st, "rr_cluster_allreduce_selftest_ex")
    return int(n.value), vals, res


COMBINE_MODES = {None: 0, "auto": 0, "pull": 1, "push": 2, "generic": 3, "direct": 4}


@_on_input_device
def splitk_combine(O: torch.Tensor, m: torch.Tensor, l: torch.Tensor, scale_log2e: float, *,
                   out: Optional[torch.Tensor] = None, mode=None) -> torch.Tensor:
    """rr_splitk_combine / rr_splitk_combine_ex: O [P, rows, D], m and l
    [P, rows] fp32 -> bf16 [rows, D].  mode: None/"auto", "pull", "push" or
    "generic" (see rr_combine_mode in rr.h)."""
    if O.dim() != 3 or m.dim() != 2 or l.dim() != 2:
        raise ValueError("O must be [P, rows, D], m and l [P, rows]")
    P, rows, D = O.shape
    if tuple(m.shape) != (P, rows) or tuple(l.shape) != (P, rows):
        raise ValueError("m and l must be [P, rows]")
    for t in (O, m, l):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise TypeError("O, m, l must be contiguous float32")
    Od = _to_device(O)
    _same_device(Od.device, m, l)
    md, ld = _to_device(m), _to_device(l)
    o = _out_buf(out, (rows, D), torch.bfloat16, Od.device)
    if mode is None:
        st = load().rr_splitk_combine(_ptr(Od), _ptr(md), _ptr(ld), P, rows, D,
                                      float(scale_log2e), _ptr(o), _stream())
    else:
        st = load().rr_splitk_combine_ex(_ptr(Od), _ptr(md), _ptr(ld), P, rows, D,
                                         float(scale_log2e), _ptr(o), _stream(),
                                         COMBINE_MODES[mode])
    check(st, "rr_splitk_combine")
    return _deliver(o, out, O)


def device_status() -> int:
    """rr_device_status on the current stream (RR_OK or RR_ERR_TIMEOUT)."""
    return int(load().rr_device_status(_stream()))


def last_tier() -> Tuple[str, int]:
    """(tier, width) of the last reduce / softmax / layernorm call."""
    v = int(load().rr_last_tier())
    return TIER_NAMES.get(v & 0xff, "?"), ((v >> 8) & 0xff) | (((v >> 19) & 0xff) << 8)


def last_staged() -> bool:
    """Whether the last row operation staged its rows in shared memory."""
    return bool((int(load().rr_last_tier()) >> 16) & 1)


def last_form() -> str:
    """How the last row operation read its rows: "grid" (split-K over a
    plain grid, partial states through the workspace), "ring" (streamed
    through a shared-memory ring), "staged" (held in shared memory),
    "chunked" (a row not 16-byte aligned in registers as head + vectors +
    tail), "twopass" (the layernorm rewrite of many long rows: the
    statistics streamed through the ring, then x read again for the
    rewrite) or "direct"."""
    v = int(load().rr_last_tier())
    if (v >> 28) & 1:
        return "twopass"
    if (v >> 27) & 1:
        return "chunked"
    if (v >> 18) & 1:
        return "grid"
    return "ring" if (v >> 17) & 1 else ("staged" if (v >> 16) & 1 else "direct")


def plan_reduce(rows: int, cols: int, sm_count: int, max_cluster: int) -> Tuple[str, int]:
    """rr_plan_reduce (host only): the tier and cluster size rr_reduce picks."""
    t, c = ctypes.c_int(), ctypes.c_int()
    check(load().rr_plan_reduce(int(rows), int(cols), int(sm_count), int(max_cluster),
                                ctypes.byref(t), ctypes.byref(c)), "rr_plan_reduce")
    return TIER_NAMES[t.value], c.value


_ROW_OPS = {"softmax": 0, "lnstats": 1, "layernorm_stats": 1, "layernorm": 2}


def plan_rowwise(rows: int, cols: int, row_op: str, sm_count: int, max_cluster: int,
                 dtype=torch.bfloat16, aligned: bool = True, staged: bool = False,
                 form: bool = False, with_workspace: bool = False):
    """rr_plan_rowwise (host only): the tier and width (lanes per row, cluster
    size, CTAs per row of the grid form, or 1) that softmax / layernorm_stats
    / layernorm pick -- with a workspace (with_workspace=True, as the
    functions here pass one) or without; with staged=True also whether the
    rows are staged in shared memory, with form=True how they are read
    ("direct", "staged", "ring" or "grid")."""
    dt = _DT.get(dtype)
    if dt not in (RR_BF16, RR_F32):
        raise TypeError(f"plan_rowwise: dtype {dtype} not supported")
    t, w, st = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    check(load().rr_plan_rowwise(int(rows), int(cols), dt, _ROW_OPS[row_op], 1 if aligned else 0,
                                 int(sm_count), int(max_cluster), 1 if with_workspace else 0,
                                 ctypes.byref(t), ctypes.byref(w), ctypes.byref(st)),
          "rr_plan_rowwise")
    if staged:
        return TIER_NAMES[t.value], w.value, st.value == 1
    if form:
        return TIER_NAMES[t.value], w.value, ("direct", "staged", "ring", "grid", "chunked", "twopass")[st.value]
    return TIER_NAMES[t.value], w.value


def plan_reduce_axis(outer: int, axis: int, inner: int, sm_count: int, max_cluster: int,
                     x_align: int = 16, with_workspace: bool = True) -> dict:
    """rr_plan_reduce_axis (host only): the launch rr_reduce_axis_ex picks."""
    p = _lib.rr_axis_plan()
    check(load().rr_plan_reduce_axis(int(outer), int(axis), int(inner), int(sm_count),
                                     int(max_cluster), int(x_align), 1 if with_workspace else 0,
                                     ctypes.byref(p)), "rr_plan_reduce_axis")
    return {"tier": TIER_NAMES[p.tier], "cluster_size": p.cluster_size,
            "emit_tile_width": p.emit_tile_width, "tile_rows": p.tile_rows,
            "splits": p.splits, "workspace_bytes": p.workspace_bytes}


def test_wait_timeout(budget_iters: int = 64) -> None:
    """rr_test_wait_timeout: enqueue the bounded-wait probe (see rr.h)."""
    check(load().rr_test_wait_timeout(int(budget_iters), _stream()), "rr_test_wait_timeout")


def test_inject_error(count: int = 1) -> None:
    """rr_test_inject_error: the next `count` calls fail with RR_ERR_CUDA
    after validating their arguments (see rr.h)."""
    check(load().rr_test_inject_error(int(count)), "rr_test_inject_error")
