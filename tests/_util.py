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
