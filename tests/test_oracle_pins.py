"""Pins for the CPU oracle: closed forms, brute force, library routines and
hand-worked examples -- never the oracle's own formula retyped.  Each case is
chosen so that a plausible slip in the oracle (a dropped term, a wrong sign or
index, a transposed operand, the wrong rounding) fails at least one of them.
"""
import math
import os
import random
import struct
from fractions import Fraction

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def f32_bits(x) -> int:
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


# ---------------------------------------------------------------- reduce

def test_sum_constant_rows_exact(oracle_mod):
    # sum of c over n is n*c; with c = 1 and n <= 2^24 every partial is exact
    n = 1 << 24
    x = np.ones((1, n), np.float32)
    assert oracle_mod.reduce_rows(x, "sum")[0] == float(n)
    # rows are independent: row r holds the constant r
    x = np.repeat(np.arange(5, dtype=np.float32)[:, None], 1000, axis=1)
    np.testing.assert_array_equal(oracle_mod.reduce_rows(x, "sum"),
                                  1000.0 * np.arange(5))


def test_sum_arange_closed_form(oracle_mod):
    for n in (1, 2, 31, 32, 33, 4096):
        x = np.arange(n, dtype=np.float32)[None, :]
        assert oracle_mod.reduce_rows(x, "sum")[0] == n * (n - 1) / 2
        xi = np.arange(n, dtype=np.int32)[None, :]
        assert oracle_mod.reduce_rows(xi, "sum")[0] == n * (n - 1) // 2


def test_sum_matches_fsum(oracle_mod):
    rng = np.random.default_rng(1)
    x = rng.standard_normal((7, 3001)).astype(np.float32)
    got = oracle_mod.reduce_rows(x, "sum")
    for r in range(7):
        exact = math.fsum(float(v) for v in x[r])
        bound = 3001 * 2.0 ** -52 * float(np.abs(x[r].astype(np.float64)).sum())
        assert abs(got[r] - exact) <= bound


def test_sum_transposed_layout_detected(oracle_mod):
    # a column-major slip would sum columns: use a non-square, non-symmetric x
    x = np.arange(12, dtype=np.float32).reshape(3, 4)
    np.testing.assert_array_equal(oracle_mod.reduce_rows(x, "sum"), [6.0, 22.0, 38.0])


def test_max_min_shuffled_arange(oracle_mod):
    rng = np.random.default_rng(2)
    for n in (1, 7, 32, 1000):
        v = rng.permutation(n).astype(np.float32)[None, :]
        assert oracle_mod.reduce_rows(v, "max")[0] == n - 1
        assert oracle_mod.reduce_rows(v, "min")[0] == 0
        vi = v.astype(np.int32) - 5
        assert oracle_mod.reduce_rows(vi, "max")[0] == n - 6
        assert oracle_mod.reduce_rows(vi, "min")[0] == -5


def test_max_min_match_numpy_and_permutation(oracle_mod):
    rng = np.random.default_rng(3)
    x = rng.standard_normal((9, 517)).astype(np.float32)
    mx = oracle_mod.reduce_rows(x, "max")
    mn = oracle_mod.reduce_rows(x, "min")
    np.testing.assert_array_equal(mx, x.max(axis=1).astype(np.float64))
    np.testing.assert_array_equal(mn, x.min(axis=1).astype(np.float64))
    xp = x[:, rng.permutation(517)]
    np.testing.assert_array_equal(oracle_mod.reduce_rows(xp, "max"), mx)
    np.testing.assert_array_equal(oracle_mod.reduce_rows(xp, "min"), mn)
    for r in range(9):                  # the result is an element of the row
        assert np.float32(mx[r]) in x[r] and np.float32(mn[r]) in x[r]


def test_signed_zero_and_nan(oracle_mod):
    pz, nz = 0.0, -0.0
    for row in ([pz, nz], [nz, pz], [nz, nz, pz, nz]):
        x = np.array([row], np.float32)
        mx = np.float32(oracle_mod.reduce_rows(x, "max")[0])
        mn = np.float32(oracle_mod.reduce_rows(x, "min")[0])
        assert f32_bits(mx) == 0x00000000
        assert f32_bits(mn) == 0x80000000
    x = np.array([[1.0, np.nan, 5.0], [np.nan, -1.0, 2.0]], np.float32)
    assert np.isnan(oracle_mod.reduce_rows(x, "max")).all()
    assert np.isnan(oracle_mod.reduce_rows(x, "min")).all()
    assert np.isnan(oracle_mod.reduce_rows(x, "sum")).all()


def test_empty_rows_give_identity(oracle_mod):
    x = np.zeros((3, 0), np.float32)
    np.testing.assert_array_equal(oracle_mod.reduce_rows(x, "sum"), [0, 0, 0])
    assert (oracle_mod.reduce_rows(x, "max") == -np.inf).all()
    assert (oracle_mod.reduce_rows(x, "min") == np.inf).all()
    xi = np.zeros((2, 0), np.int32)
    np.testing.assert_array_equal(oracle_mod.reduce_rows(xi, "sum"), [0, 0])
    np.testing.assert_array_equal(oracle_mod.reduce_rows(xi, "max"), [-2**31] * 2)
    np.testing.assert_array_equal(oracle_mod.reduce_rows(xi, "min"), [2**31 - 1] * 2)
    assert oracle_mod.reduce_rows(np.zeros((0, 5), np.float32), "sum").shape == (0,)


def test_int32_sum_wraps_like_modular_arithmetic(oracle_mod):
    rng = np.random.default_rng(4)
    x = rng.integers(-2**31, 2**31, size=(6, 300), dtype=np.int64).astype(np.int32)
    got = oracle_mod.reduce_rows(x, "sum")
    for r in range(6):
        s = sum(int(v) for v in x[r]) % (1 << 32)
        if s >= 1 << 31:
            s -= 1 << 32
        assert int(got[r]) == s
    # bounded workload values never wrap: |x| <= 2^15, N <= 8192
    xb = rng.integers(-2**15, 2**15 + 1, size=(4, 8192)).astype(np.int32)
    np.testing.assert_array_equal(oracle_mod.reduce_rows(xb, "sum"),
                                  xb.astype(np.int64).sum(axis=1))


def test_reduce_axis_matches_numpy_and_closed_forms(oracle_mod):
    rng = np.random.default_rng(15)
    x = rng.standard_normal((3, 50, 7)).astype(np.float32)
    np.testing.assert_allclose(oracle_mod.reduce_axis(x, "sum"),
                               x.astype(np.float64).sum(axis=1), rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(oracle_mod.reduce_axis(x, "max"), x.max(axis=1))
    np.testing.assert_array_equal(oracle_mod.reduce_axis(x, "min"), x.min(axis=1))
    # sum over the axis of arange along the axis: axis * (axis - 1) / 2 in every column
    a = np.broadcast_to(np.arange(64, dtype=np.int32)[None, :, None], (2, 64, 5)).copy()
    np.testing.assert_array_equal(oracle_mod.reduce_axis(a, "sum"), np.full((2, 5), 64 * 63 // 2))
    # the reduce runs over the middle index only: a value planted at (o, a, i)
    # shows up in out[o, i] and nowhere else
    z = np.zeros((4, 9, 6), np.float32)
    z[2, 5, 3] = 7.0
    got = oracle_mod.reduce_axis(z, "sum")
    assert got[2, 3] == 7.0 and got.sum() == 7.0
    # inner == 1 is the row reduction
    r = rng.standard_normal((5, 33, 1)).astype(np.float32)
    np.testing.assert_array_equal(oracle_mod.reduce_axis(r, "max")[:, 0],
                                  oracle_mod.reduce_rows(r[:, :, 0], "max"))
    ri = rng.integers(-2**31, 2**31, (2, 40, 3), dtype=np.int64).astype(np.int32)
    wrap = (ri.astype(np.int64).sum(axis=1) + 2**31) % 2**32 - 2**31
    np.testing.assert_array_equal(oracle_mod.reduce_axis(ri, "sum"), wrap)


# ---------------------------------------------------------------- cluster fold

def _golden_fold_cases():
    with open(os.path.join(GOLDEN, "cluster_fold_order.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            lhs, rhs = line.split("->")
            op, dt, C, *vals = lhs.split()
            yield op, dt, int(C), vals, rhs.strip()


@pytest.mark.parametrize("case", list(_golden_fold_cases()),
                         ids=lambda c: f"{c[0]}-{c[1]}-{c[2]}")
def test_cluster_fold_golden(oracle_mod, case):
    op, dt, C, vals, expect = case
    if dt == "f32":
        v = np.array([float(s) for s in vals], np.float32).reshape(C, 1)
        got = oracle_mod.cluster_fold(v, op)[0]
        assert f32_bits(got) == f32_bits(np.float32(float(expect)))
    else:
        v = np.array([int(s) for s in vals], np.int64).astype(np.int32).reshape(C, 1)
        assert int(oracle_mod.cluster_fold(v, op)[0]) == int(expect)


def test_cluster_fold_single_rank_is_broadcast(oracle_mod):
    rng = np.random.default_rng(5)
    v = rng.standard_normal((1, 8)).astype(np.float32)
    for op in ("sum", "max", "min"):
        np.testing.assert_array_equal(oracle_mod.cluster_fold(v, op), v[0])


def test_cluster_fold_matches_numpy_fp32_sequential(oracle_mod):
    rng = np.random.default_rng(6)
    for C in (2, 3, 8, 16):
        v = (rng.standard_normal((C, 4)) * 10.0 ** rng.integers(-3, 6, (C, 4))
             ).astype(np.float32)
        got = oracle_mod.cluster_fold(v, "sum")
        acc = v[0].copy()
        for r in range(1, C):
            acc = (acc + v[r]).astype(np.float32)   # numpy fp32 IEEE add
        assert [f32_bits(a) for a in got] == [f32_bits(a) for a in acc]
        np.testing.assert_array_equal(oracle_mod.cluster_fold(v, "max"), v.max(0))
        np.testing.assert_array_equal(oracle_mod.cluster_fold(v, "min"), v.min(0))


# ---------------------------------------------------------------- softmax

def test_softmax_constant_row(oracle_mod):
    for n in (1, 5, 4096):
        x = np.full((2, n), 3.25, np.float32)
        np.testing.assert_allclose(oracle_mod.softmax(x), 1.0 / n, rtol=1e-15)


def test_softmax_matches_scipy_and_sums_to_one(oracle_mod):
    scipy_special = pytest.importorskip("scipy.special")
    rng = np.random.default_rng(7)
    x = (3.0 * rng.standard_normal((5, 777))).astype(np.float32)
    y = oracle_mod.softmax(x)
    ref = scipy_special.softmax(x.astype(np.float64), axis=1)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=0)
    np.testing.assert_allclose(y.sum(axis=1), 1.0, rtol=0, atol=777 * 2.0 ** -52)


def test_softmax_two_element_logistic(oracle_mod):
    a = 1.5
    y = oracle_mod.softmax(np.array([[0.0, a]], np.float32))[0]
    assert abs(y[1] - 1.0 / (1.0 + math.exp(-a))) < 1e-15
    assert abs(y[0] - 1.0 / (1.0 + math.exp(a))) < 1e-15
    # the running max keeps exp finite: e^800 overflows fp64, e^(800-800) does not
    y = oracle_mod.softmax(np.array([[799.0, 800.0], [-800.0, -799.0]],
                                    np.float32))
    for r in range(2):
        assert abs(y[r, 1] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15


def test_softmax_bf16_widening(oracle_mod):
    import torch
    g = torch.Generator().manual_seed(8)
    xb = (3.0 * torch.randn(4, 300, generator=g)).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    xf = xb.to(torch.float32).numpy()
    np.testing.assert_array_equal(oracle_mod.softmax(bits), oracle_mod.softmax(xf))
    # shift invariance, on small integers so that x + 8 is exact in fp32
    xi = np.random.default_rng(8).integers(-20, 21, (3, 50)).astype(np.float32)
    np.testing.assert_allclose(oracle_mod.softmax(xi + np.float32(8.0)),
                               oracle_mod.softmax(xi), rtol=1e-13)


# ---------------------------------------------------------------- layernorm

def test_layernorm_constant_and_alternating(oracle_mod):
    eps = 1e-5
    x = np.full((1, 64), 2.5, np.float32)
    mean, var, rstd = oracle_mod.layernorm_stats(x, eps)
    assert mean[0] == 2.5 and var[0] == 0.0
    assert rstd[0] == 1.0 / math.sqrt(eps)
    a = 1.75
    x = np.tile(np.array([a, -a], np.float32), 40)[None, :]
    mean, var, rstd = oracle_mod.layernorm_stats(x, eps)
    assert mean[0] == 0.0 and var[0] == a * a
    assert abs(rstd[0] - 1.0 / math.sqrt(a * a + eps)) < 1e-15


def test_layernorm_matches_numpy(oracle_mod):
    import torch
    g = torch.Generator().manual_seed(9)
    xb = torch.randn(6, 1000, generator=g).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    xf = xb.to(torch.float64).numpy()
    mean, var, rstd = oracle_mod.layernorm_stats(bits, 1e-5)
    np.testing.assert_allclose(mean, xf.mean(axis=1), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(var, xf.var(axis=1, ddof=0), rtol=1e-12)
    np.testing.assert_allclose(rstd, 1.0 / np.sqrt(xf.var(axis=1) + 1e-5), rtol=1e-12)


def test_layernorm_rewrite_closed_forms(oracle_mod):
    rng = np.random.default_rng(12)
    cols = 96
    # constant row: x - mean = 0, so y = beta exactly
    x = np.full((2, cols), 1.25, np.float32)
    g = rng.standard_normal(cols).astype(np.float32)
    b = rng.standard_normal(cols).astype(np.float32)
    y64, y16, mean, rstd = oracle_mod.layernorm(x, g, b, 1e-5)
    np.testing.assert_array_equal(y64, np.broadcast_to(b.astype(np.float64), (2, cols)))
    # +-a alternating, gamma = 1, beta = 0: y = +-a / sqrt(a^2 + eps)
    a = 2.0
    x = np.tile(np.array([a, -a], np.float32), cols // 2)[None, :]
    ones, zeros = np.ones(cols, np.float32), np.zeros(cols, np.float32)
    y64, _, _, _ = oracle_mod.layernorm(x, ones, zeros, 1e-5)
    expect = np.tile([a, -a], cols // 2) / np.sqrt(a * a + 1e-5)
    np.testing.assert_allclose(y64[0], expect, rtol=1e-14)
    # gamma scales and beta shifts column-wise: index, not row, dependent
    x = rng.standard_normal((3, cols)).astype(np.float32)
    y1, _, m1, r1 = oracle_mod.layernorm(x, ones, zeros, 1e-5)
    y2, _, _, _ = oracle_mod.layernorm(x, g, b, 1e-5)
    np.testing.assert_allclose(y2, y1 * g.astype(np.float64) + b.astype(np.float64), rtol=1e-13,
                               atol=1e-13)


def test_layernorm_rewrite_matches_numpy_and_rounds_once(oracle_mod):
    import torch
    gen = torch.Generator().manual_seed(13)
    xb = torch.randn(5, 700, generator=gen).to(torch.bfloat16)
    bits = xb.view(torch.int16).numpy().view(np.uint16)
    xf = xb.to(torch.float64).numpy()
    rng = np.random.default_rng(14)
    g = rng.standard_normal(700).astype(np.float32)
    b = rng.standard_normal(700).astype(np.float32)
    y64, y16, mean, rstd = oracle_mod.layernorm(bits, g, b, 1e-5)
    mu = xf.mean(axis=1, keepdims=True)
    ref = (xf - mu) / np.sqrt(xf.var(axis=1, keepdims=True) + 1e-5) * g + b
    np.testing.assert_allclose(y64, ref, rtol=1e-12, atol=1e-12)
    # y_bf16 is the single rounding of y_f64
    for i in range(0, 700, 37):
        assert y16[2, i] == oracle_mod.f64_to_bf16_bits(y64[2, i])


# ---------------------------------------------------------------- combine

def _golden_combine_cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "combine_worked.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            if key == "case":
                cur = {"name": vals[0]}
                cases.append(cur)
            else:
                cur[key] = vals
    return cases


@pytest.mark.parametrize("case", _golden_combine_cases(), ids=lambda c: c["name"])
def test_combine_golden(oracle_mod, case):
    P, rows, D = int(case["P"][0]), int(case["rows"][0]), int(case["D"][0])
    m = np.array(case["m"], np.float32).reshape(P, rows)
    l = np.array(case["l"], np.float32).reshape(P, rows)
    O = np.array(case["O"], np.float32).reshape(P, rows, D)
    out64, out16 = oracle_mod.splitk_combine(O, m, l, float(case["scale_log2e"][0]))
    np.testing.assert_array_equal(out64.ravel(), np.array(case["out"], np.float64))
    np.testing.assert_array_equal(out16.ravel(),
                                  np.array([int(h, 16) for h in case["out_bf16"]]))


def test_combine_special_cases(oracle_mod):
    rng = np.random.default_rng(10)
    rows, D, s = 9, 16, 0.12752743
    O1 = rng.standard_normal((1, rows, D)).astype(np.float32)
    m1 = rng.standard_normal((1, rows)).astype(np.float32)
    l1 = rng.uniform(1, 64, (1, rows)).astype(np.float32)
    # P = 1: O / l
    out64, _ = oracle_mod.splitk_combine(O1, m1, l1, s)
    np.testing.assert_array_equal(out64, O1[0].astype(np.float64) / l1[0, :, None])
    # identical partials: O / l
    O4, m4, l4 = np.repeat(O1, 4, 0), np.repeat(m1, 4, 0), np.repeat(l1, 4, 0)
    out64, _ = oracle_mod.splitk_combine(O4, m4, l4, s)
    np.testing.assert_allclose(out64, O1[0].astype(np.float64) / l1[0, :, None],
                               rtol=1e-14)
    # all m equal: sum O / sum l
    O3 = rng.standard_normal((3, rows, D)).astype(np.float32)
    l3 = rng.uniform(1, 64, (3, rows)).astype(np.float32)
    m3 = np.full((3, rows), 0.7, np.float32)
    out64, _ = oracle_mod.splitk_combine(O3, m3, l3, s)
    np.testing.assert_allclose(out64, O3.astype(np.float64).sum(0)
                               / l3.astype(np.float64).sum(0)[:, None], rtol=1e-14)
    # one partition higher by 1000: that partition's O / l
    m3b = m3.copy()
    m3b[1] += 1000.0
    out64, _ = oracle_mod.splitk_combine(O3, m3b, l3, s)
    np.testing.assert_allclose(out64, O3[1] / l3[1, :, None].astype(np.float64),
                               rtol=1e-14)


def test_combine_dead_rows_zero(oracle_mod):
    O = np.ones((2, 2, 4), np.float32)
    m = np.array([[-np.inf, 0.0], [-np.inf, 1.0]], np.float32)
    l = np.array([[1.0, 0.0], [1.0, 0.0]], np.float32)
    out64, out16 = oracle_mod.splitk_combine(O, m, l, 1.0)
    assert (out64 == 0).all() and (out16 == 0).all()


# ---------------------------------------------------------------- bf16 rounding

def _golden_bf16():
    with open(os.path.join(GOLDEN, "bf16_rounding.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            v, bits, *_ = line.split()
            x = float.fromhex(v) if "0x" in v else float(v)
            yield x, int(bits, 16)


@pytest.mark.parametrize("case", list(_golden_bf16()), ids=lambda c: repr(c[0]))
def test_bf16_rounding_golden(oracle_mod, case):
    x, bits = case
    assert oracle_mod.f64_to_bf16_bits(x) == bits


def _bf16_value(bits: int) -> Fraction:
    f = struct.unpack("<f", struct.pack("<I", bits << 16))[0]
    return Fraction(f)


def test_bf16_rounding_brute_force(oracle_mod):
    # nearest of all candidate bf16 neighbours, ties to the even bit pattern,
    # decided in exact rational arithmetic
    rnd = random.Random(11)
    for _ in range(3000):
        x = rnd.uniform(-1, 1) * 2.0 ** rnd.randint(-140, 120)
        if rnd.random() < 0.2:   # near-halfway cases
            b = f32_bits(abs(x)) >> 16
            lo, hi = _bf16_value(b), _bf16_value(b + 1)
            x = math.copysign(float((lo + hi) / 2 + Fraction(rnd.choice((-1, 0, 1)),
                                                              2 ** 160)), x)
        got = oracle_mod.f64_to_bf16_bits(x)
        ax, sign = Fraction(abs(x)), (0x8000 if x < 0 else 0)
        b = f32_bits(abs(x)) >> 16
        cands = [c for c in (b - 1, b, b + 1, b + 2) if 0 <= c < 0x7f80]
        best = min(cands, key=lambda c: (abs(_bf16_value(c) - ax), c & 1))
        assert got == (sign | best), (x, hex(got), hex(sign | best))
