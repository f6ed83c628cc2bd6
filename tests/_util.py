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


def _bf16_half_ulp(a) -> np.ndarray:
    """Half the bf16 spacing at magnitude |a| (8 significant bits; the
    subnormal spacing 2^-133 below 2^-126)."""
    a = np.abs(np.asarray(a, np.float64))
    ex = np.floor(np.log2(np.where(a > 0, a, 2.0 ** -133)))
    return 2.0 ** (np.maximum(ex, -126) - 8)


def layernorm_rewrite_bound(x_f64, gamma, beta, k_mean, k_rstd):
    """(z, e): the exact value z = (x - mu_k) * rs_k * gamma + beta of the
    rewrite given the kernel's own fp32 statistics mu_k, rs_k, and the bound
    e on |f - z| for the fp32 value f the kernel rounds to bf16.  Every form
    of the kernel evaluates f = fmaf(fl(fl(x - mu_k) * rs_k), gamma, beta):
    two roundings inside the product and one in the fused multiply-add, so
        |f - z| <= (2u + u^2)(1 + u) |(x - mu_k) rs_k gamma| + u |z| + 2^-149
    with u = 2^-24 (the last term: fp32 subnormal spacing)."""
    u = 2.0 ** -24
    xc = np.asarray(x_f64, np.float64) - np.asarray(k_mean, np.float64)[:, None]
    t = xc * np.asarray(k_rstd, np.float64)[:, None] * np.asarray(gamma, np.float64)[None, :]
    z = t + np.asarray(beta, np.float64)[None, :]
    e = (2 * u + u * u) * (1 + u) * np.abs(t) + u * np.abs(z) + 2.0 ** -149
    return z, e


def assert_layernorm_close(gpu_bits, ref_f64, ref_bits, x_f64, gamma, beta, mean, rstd,
                           k_mean, k_rstd, max_relaxed_frac: float = 1e-3):
    """Layernorm rewrite parity, in three steps (mean / rstd: the oracle's
    fp64 statistics; k_mean / k_rstd: the kernel's fp32 ones, same rows).
    1. The kernel's statistics are within the statistics tolerance:
       |mu_k - mean| <= 1e-5 max(|mean|, ||x||_2 / N), |rs_k - rstd| <= 1e-5 rstd.
    2. Every output is the bf16 rounding of the rewrite evaluated from those
       statistics: |y - z| <= e + half a bf16 spacing at |z| + e
       (layernorm_rewrite_bound), with no exception.
    3. Against the oracle's correctly rounded value: within 1 bf16 ulp, or,
       where (x - mean) rstd gamma cancels against beta, within what the
       statistics tolerance of step 1 admits: z - ref equals
       -(mu_k - mean) rs_k gamma + (x - mean)(rs_k - rstd) gamma exactly, so
       |y - ref| <= |y - z| + 1e-5 max(|mean|, ||x||_2 / N) rs_k |gamma|
       + 1e-5 |x - mean| rstd |gamma|.  At most `max_relaxed_frac` of the
       outputs may need this second form.
    Returns the number of outputs that needed it."""
    x_f64 = np.asarray(x_f64, np.float64)
    n = x_f64.shape[1]
    mean = np.asarray(mean, np.float64)
    rstd = np.asarray(rstd, np.float64)
    km = np.asarray(k_mean, np.float32).astype(np.float64)
    kr = np.asarray(k_rstd, np.float32).astype(np.float64)
    mb = 1e-5 * np.maximum(np.abs(mean), np.sqrt((x_f64 ** 2).sum(axis=1)) / n)
    badm = np.nonzero(~(np.abs(km - mean) <= mb))[0]
    assert badm.size == 0, f"{badm.size} kernel means out of tolerance; rows {badm[:5]}"
    badr = np.nonzero(~(np.abs(kr - rstd) <= 1e-5 * rstd))[0]
    assert badr.size == 0, f"{badr.size} kernel rstd out of tolerance; rows {badr[:5]}"
    g = bf16_value(gpu_bits)
    z, e = layernorm_rewrite_bound(x_f64, gamma, beta, km, kr)
    step2 = np.abs(g - z) <= e + _bf16_half_ulp(np.abs(z) + e)
    bad = np.nonzero(~step2)
    assert bad[0].size == 0, (f"{bad[0].size} rewrite outputs are not the rounding of the rewrite "
                              f"of the kernel's own statistics; first at {tuple(b[:3] for b in bad)}: "
                              f"gpu={g[bad][:3]} z={z[bad][:3]} e={e[bad][:3]}")
    d = np.abs(bf16_ord(gpu_bits) - bf16_ord(ref_bits))
    strict = d <= 1
    ref = np.asarray(ref_f64, np.float64)
    gm = np.abs(np.asarray(gamma, np.float64))[None, :]
    prop = (mb[:, None] * kr[:, None] * gm +
            np.abs(x_f64 - mean[:, None]) * (1e-5 * rstd)[:, None] * gm)
    relaxed = np.abs(g - ref) <= np.abs(g - z) + prop + 2.0 ** -50 * np.abs(ref)
    bad = np.nonzero(~(strict | relaxed))
    assert bad[0].size == 0, (f"{bad[0].size} layernorm outputs out of tolerance; first at "
                              f"{tuple(b[:3] for b in bad)}: gpu={g[bad][:3]} ref={ref[bad][:3]}")
    n_relaxed = int((~strict).sum())
    assert n_relaxed <= max(2, max_relaxed_frac * strict.size), (
        f"{n_relaxed} of {strict.size} outputs needed the cancellation bound")
    return n_relaxed


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


_M64 = (1 << 64) - 1


def splitmix64(z: np.ndarray) -> np.ndarray:
    """splitmix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
    number generators", OOPSLA 2014), elementwise on uint64, written from its
    published definition: add the golden-ratio increment, then two
    xor-shift-multiply rounds and a final xor-shift."""
    z = np.asarray(z, np.uint64) + np.uint64(0x9E3779B97F4A7C15)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
    return z ^ (z >> np.uint64(31))


def selftest_values(n: int, seed: int, dtype) -> np.ndarray:
    """The cluster self-test's seeded inputs as the C ABI documents them:
    value i comes from u = splitmix64(seed ^ splitmix64(i)); int32 takes the
    high 32 bits of u, fp32 ldexp((u >> 40) * 2^-23 - 1, (u >> 8) % 41 - 20)."""
    with np.errstate(over="ignore"):
        i = np.arange(n, dtype=np.uint64)
        u = splitmix64(np.uint64(seed & _M64) ^ splitmix64(i))
    if dtype == np.int32:
        return (u >> np.uint64(32)).astype(np.uint32).view(np.int32)
    mant = (u >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -23) - np.float32(1.0)
    ex = ((u >> np.uint64(8)) % np.uint64(41)).astype(np.int64) - 20
    return np.ldexp(mant, ex).astype(np.float32)
