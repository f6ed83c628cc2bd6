"""Inputs of more than 2^31 elements for every tier and operation, so that an
element offset held in 32 bits anywhere would show.  Each test holds 9 to
13 GB on the device; the oracle checks rows (or columns) whose offsets lie
past 2^31, and the first ones."""
import numpy as np
import pytest
import torch

from _util import (assert_bits_equal, assert_combine_close, assert_layernorm_close,
                   assert_rel_close, assert_sum_close, to_np)

pytestmark = pytest.mark.gpu
BIG = 1 << 31


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cluster_reductions_gb300 as rr
    rr.load()
    return rr


@pytest.fixture(autouse=True)
def _free():
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _f32(rows, cols, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn((rows, cols), generator=g, device="cuda")


def _check_rows(oracle_mod, x, got, rows_idx, op):
    xh = to_np(x[rows_idx])
    ref = oracle_mod.reduce_rows(xh, op)
    g = to_np(got[rows_idx])
    if op == "sum":
        assert_sum_close(g, ref, xh)
    else:
        assert_bits_equal(g, ref)


@pytest.mark.parametrize("rows,cols", [(70000, 32768), (70 << 20, 32), (300 << 20, 8), (2, 1200 << 20)],
                         ids=["block", "warp", "tiled", "splitk"])
def test_reduce_past_2_31(rr, oracle_mod, rows, cols):
    assert rows * cols > BIG
    x = _f32(rows, cols, 9001)
    tail = [0, 1, rows - 2, rows - 1] if rows > 2 else [0, 1]
    for op in ("sum", "max"):
        got = rr.reduce(x, op)
        _check_rows(oracle_mod, x, got, tail, op)
    if rows == 2:
        ws = torch.empty(2 * 1024, dtype=torch.int32, device="cuda")
        got = rr.reduce_splitk_multi(x, "sum", workspace=ws)
        _check_rows(oracle_mod, x, got, [0, 1], "sum")


def test_reduce_axis_past_2_31(rr, oracle_mod):
    outer, axis, inner = 1, 70000, 32768
    x = _f32(outer * axis, inner, 9002).view(outer, axis, inner)
    got = to_np(rr.reduce_axis(x, "max", 1))
    cols = [0, 5, inner - 1]
    sub = np.ascontiguousarray(to_np(x[:, :, cols]))
    assert_bits_equal(got[:, cols].reshape(-1), oracle_mod.reduce_axis(sub, "max").reshape(-1))
    x2 = _f32(300 << 20, 8, 9003).view(3 << 20, 100, 8)        # tiled / warp tier, 2.4 G elements
    got2 = to_np(rr.reduce_axis(x2, "sum", 1))
    idx = [0, (3 << 20) - 1]
    sub2 = np.ascontiguousarray(to_np(x2[idx]))
    ref2 = oracle_mod.reduce_axis(sub2, "sum")
    lines = np.ascontiguousarray(sub2.transpose(0, 2, 1)).reshape(-1, 100)
    assert_sum_close(got2[idx].reshape(-1), ref2.reshape(-1), lines)


def test_rowwise_past_2_31(rr, oracle_mod):
    rows, cols = 270000, 8192
    assert rows * cols > BIG
    xb = _f32(rows, cols, 9004).to(torch.bfloat16)
    tail = [0, rows - 2, rows - 1]
    y = rr.softmax(xb)
    xh = to_np(xb[tail])
    assert_rel_close(to_np(y[tail]), oracle_mod.softmax(xh), 1e-5, floor=1e-30, what="softmax")
    del y
    from cluster_reductions_gb300 import inputs
    g, b = inputs.layernorm_params(cols, 9005, "cuda")
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    yb = rr.layernorm(xb, g, b, 1e-5, mean=mean, rstd=rstd)
    y64, y16, m64, r64 = oracle_mod.layernorm(xh, to_np(g), to_np(b), 1e-5)
    xf = xb[tail].to(torch.float64).cpu().numpy()
    assert_layernorm_close(to_np(yb[tail]), y64, y16, xf, to_np(g), to_np(b), m64, r64,
                           to_np(mean[tail]), to_np(rstd[tail]))
    assert_rel_close(to_np(rstd[tail]), r64, 1e-5, what="layernorm rstd")


def test_combine_past_2_31(rr, oracle_mod):
    from cluster_reductions_gb300 import inputs
    P, rows, D = 8, (2 << 20) + 4096, 128
    assert P * rows * D > BIG
    O, m, l, s = inputs.combine_partials(P, rows, D, 9006, "cuda")
    out = rr.splitk_combine(O, m, l, s)
    tail = [0, rows - 3, rows - 1]
    Oh = np.ascontiguousarray(to_np(O[:, tail]))
    mh, lh = np.ascontiguousarray(to_np(m[:, tail])), np.ascontiguousarray(to_np(l[:, tail]))
    ref64, ref = oracle_mod.splitk_combine(Oh, mh, lh, s)
    assert_combine_close(to_np(out[tail]), ref64, ref, Oh, mh, lh, s)


def test_rowwise_warp_past_2_31(rr, oracle_mod):
    # the warp tier of the row ops: 2,098,152 rows of 1024 bf16 (2.1 G elements)
    rows, cols = (BIG >> 10) + 1000, 1024
    xb = _f32(rows, cols, 9007).to(torch.bfloat16)
    tail = [0, rows - 2, rows - 1]
    xh = to_np(xb[tail])
    y = rr.softmax(xb)
    assert rr.last_tier()[0] == "warp"
    assert_rel_close(to_np(y[tail]), oracle_mod.softmax(xh), 1e-5, floor=1e-30, what="softmax warp")
    del y
    from cluster_reductions_gb300 import inputs
    g, b = inputs.layernorm_params(cols, 9008, "cuda")
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    yb = rr.layernorm(xb, g, b, 1e-5, mean=mean, rstd=rstd)
    assert rr.last_tier()[0] == "warp"
    y64, y16, m64, r64 = oracle_mod.layernorm(xh, to_np(g), to_np(b), 1e-5)
    xf = xb[tail].to(torch.float64).cpu().numpy()
    assert_layernorm_close(to_np(yb[tail]), y64, y16, xf, to_np(g), to_np(b), m64, r64,
                           to_np(mean[tail]), to_np(rstd[tail]))
    assert_rel_close(to_np(rstd[tail]), r64, 1e-5, what="layernorm rstd warp")
