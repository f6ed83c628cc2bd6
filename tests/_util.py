"""Shared helpers of the tests: tolerance checks stated once, host copies of
device tensors for the oracle, bf16 ordinal distance."""
from __future__ import annotations

import numpy as np
import torch


def to_np(t: torch.Tensor) -> np.ndarray:
    """Host numpy copy; bf16 becomes its raw uint16 bit patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def f32_bits(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float32)).view(np.uint32)


def assert_sum_close(gpu: np.ndarray, ref: np.ndarray, x: np.ndarray, rtol: float = 1e-5):
    """fp32 sum vs the fp64 oracle: |gpu - ref| <= rtol * max(|ref|, ||x_row||_2).
    The row norm is in the bound because a sum of signed values may cancel
    to near zero, where plain relative error is meaningless."""
    gpu = np.asarray(gpu, np.float64)
    norm = np.sqrt((np.asarray(x, np.float64) ** 2).sum(axis=1)) if x.shape[1] else np.zeros(len(ref))
    bound = rtol * np.maximum(np.abs(ref), norm)
    err = np.abs(gpu - ref)
    bad = np.nonzero(~(err <= bound))[0]
    assert bad.size == 0, (f"{bad.size} rows out of tolerance; first {bad[:5]}: "
                           f"gpu={gpu[bad[:5]]} ref={ref[bad[:5]]} bound={bound[bad[:5]]}")


def assert_bits_equal(gpu: np.ndarray, ref: np.ndarray):
    """Exact equality of fp32 / int32 results, bit for bit."""
    g = np.ascontiguousarray(gpu)
    r = np.ascontiguousarray(ref)
    if g.dtype == np.float32 or r.dtype in (np.float32, np.float64):
        g, r = f32_bits(g), f32_bits(r)
    bad = np.nonzero(g != r)[0]
    assert bad.size == 0, f"{bad.size} mismatches; first {bad[:5]}: gpu={g[bad[:5]]} ref={r[bad[:5]]}"


def assert_rel_close(gpu, ref, rtol: float, floor: float = 0.0, what: str = ""):
    """Plain relative error |gpu - ref| <= rtol * |ref| on elements with
    |ref| >= floor."""
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    m = np.abs(ref) >= floor
    err = np.abs(gpu - ref)
    ok = err <= rtol * np.abs(ref)
    bad = np.nonzero(m & ~ok)
    assert bad[0].size == 0, (f"{what}: {bad[0].size} elements out of tolerance; first at "
                              f"{tuple(b[:3] for b in bad)}: gpu={gpu[bad][:3]} ref={ref[bad][:3]}")


def bf16_ord(bits: np.ndarray) -> np.ndarray:
    """Monotone integer image of bf16 bit patterns (+0 and -0 both map to 0)."""
    b = np.asarray(bits, np.int64) & 0xffff
    return np.where(b & 0x8000, -(b & 0x7fff), b)


def assert_bf16_ulp(gpu_bits: np.ndarray, ref_bits: np.ndarray, ulp: int = 1):
    d = np.abs(bf16_ord(gpu_bits) - bf16_ord(ref_bits))
    bad = np.nonzero(d > ulp)
    assert bad[0].size == 0, (f"{bad[0].size} bf16 values more than {ulp} ulp off; first at "
                              f"{tuple(b[:3] for b in bad)}: gpu={gpu_bits[bad][:3]} "
                              f"ref={ref_bits[bad][:3]}")


def assert_layernorm_close(gpu_bits, ref_f64, ref_bits, x_f64, gamma, beta, mean, rstd,
                           max_relaxed_frac: float = 1e-3):
    """Layernorm rewrite parity: each output within 1 bf16 ulp of the
    oracle's correctly rounded value, or -- where (x - mean) * rstd * gamma
    cancels against beta -- within one ulp plus the fp32 bound
        64u (|x - mean| rstd |gamma| + |beta|) + 64u rstd |gamma| sum|x| / N,
    u = 2^-24: the kernel's mean carries the fp32 summation error of the
    row (serial per-thread chains plus a tree, well under 64u sum|x| / N),
    and each of the few roundings after it adds u relative to its operand.
    At most `max_relaxed_frac` of the outputs may need the second form."""
    d = np.abs(bf16_ord(gpu_bits) - bf16_ord(ref_bits))
    strict = d <= 1
    g = bf16_value(gpu_bits)
    ref = np.asarray(ref_f64, np.float64)
    a = np.abs(ref)
    ex = np.floor(np.log2(np.where(a > 0, a, 2.0 ** -133)))
    ulp = 2.0 ** (np.maximum(ex, -126) - 7)
    u = 2.0 ** -24
    xc = np.asarray(x_f64, np.float64) - np.asarray(mean, np.float64)[:, None]
    rs = np.asarray(rstd, np.float64)[:, None]
    gm = np.abs(np.asarray(gamma, np.float64))[None, :]
    bt = np.abs(np.asarray(beta, np.float64))[None, :]
    sabs = np.abs(np.asarray(x_f64, np.float64)).sum(axis=1, keepdims=True) / x_f64.shape[1]
    bound = ulp + 64 * u * (np.abs(xc) * rs * gm + bt) + 64 * u * rs * gm * sabs
    relaxed = np.abs(g - ref) <= bound
    bad = np.nonzero(~(strict | relaxed))
    assert bad[0].size == 0, (f"{bad[0].size} layernorm outputs out of tolerance; first at "
                              f"{tuple(b[:3] for b in bad)}: gpu={g[bad][:3]} ref={ref[bad][:3]}")
    n_relaxed = int((~strict).sum())
    assert n_relaxed <= max(2, max_relaxed_frac * strict.size), (
        f"{n_relaxed} of {strict.size} outputs needed the cancellation bound")


def bf16_value(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def combine_fp32_bound(O, m, l, scale_log2e) -> np.ndarray:
    """Bound on the fp32 rounding error of a combine output before its bf16
    rounding, [rows, D].  The kernel forms w_q = ex2.approx((m_q - M) * s)
    (relative error <= 2^-22 from the instruction plus <= 2 * 2^-24 * |arg|
    * ln 2 from the rounded argument; 2^-20 covers |arg| <= 8), folds
    L = sum w_q l_q and acc = sum w_q O_q with P fused multiply-adds each,
    and multiplies acc by the rounded 1/L.  So
        |err| <= (e_w + P u) * sum_q w_q |O_q| / L + (e_w + (P + 2) u) |out|
    with u = 2^-24, e_w = 2^-20.  The first term is what cancellation in
    sum_q w_q O_q exposes: an output far below its summands can be many bf16
    ulps off in any fp32 evaluation."""
    O = np.asarray(O, np.float64)
    m = np.asarray(m, np.float64)
    l = np.asarray(l, np.float64)
    P = O.shape[0]
    M = m.max(axis=0)
    with np.errstate(invalid="ignore", over="ignore"):
        w = np.exp2((m - M) * float(scale_log2e))
    w = np.where(np.isfinite(w), w, 0.0)
    L = (w * l).sum(axis=0)
    Ls = np.where(L > 0, L, np.inf)
    absum = (w[:, :, None] * np.abs(O)).sum(axis=0) / Ls[:, None]
    out = (w[:, :, None] * O).sum(axis=0) / Ls[:, None]
    u, ew = 2.0 ** -24, 2.0 ** -20
    return (ew + P * u) * absum + (ew + (P + 2) * u) * np.abs(out)


def assert_combine_close(gpu_bits, ref_f64, ref_bits, O, m, l, scale_log2e,
                         max_relaxed_frac: float = 1e-3):
    """Combine parity: each output within 1 bf16 ulp of the oracle's
    correctly rounded value, or -- only where the weighted sum cancels --
    within one bf16 ulp of |ref| plus the fp32 error bound above.  At most
    `max_relaxed_frac` of the outputs may need the second form."""
    d = np.abs(bf16_ord(gpu_bits) - bf16_ord(ref_bits))
    strict = d <= 1
    g = bf16_value(gpu_bits)
    ref = np.asarray(ref_f64, np.float64)
    a = np.abs(ref)
    ex = np.floor(np.log2(np.where(a > 0, a, 2.0 ** -133)))
    ulp = 2.0 ** (np.maximum(ex, -126) - 7)
    bound = ulp + combine_fp32_bound(O, m, l, scale_log2e)
    relaxed = np.abs(g - ref) <= bound
    bad = np.nonzero(~(strict | relaxed))
    assert bad[0].size == 0, (f"{bad[0].size} combine outputs out of tolerance; first at "
                              f"{tuple(b[:3] for b in bad)}: gpu={g[bad][:3]} ref={ref[bad][:3]} "
                              f"bound={bound[bad][:3]}")
    n_relaxed = int((~strict).sum())
    assert n_relaxed <= max(2, max_relaxed_frac * strict.size), (
        f"{n_relaxed} of {strict.size} outputs needed the cancellation bound")
