"""GPU parity of rr_softmax and rr_layernorm_stats against the fp64 oracle.

Bars: softmax per element within relative 1e-5 (elements >= 1e-30); each
row's sum within 1e-5 of 1; layernorm mean within 1e-5 * max(|mean|,
||x_row||_2 / N), rstd within relative 1e-5."""
import numpy as np
import pytest
import torch

from _util import assert_bits_equal, assert_rel_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cluster_reductions_gb300 as rr
    rr.load()
    return rr


def _x(rows, cols, dtype, seed, std, offset=0):
    from cluster_reductions_gb300 import inputs
    base = inputs.normal_f32(1, rows * cols + offset, seed, "cuda", std).to(dtype)
    return base.view(-1)[offset:].view(rows, cols)


def check_softmax(rr, oracle_mod, x):
    y = to_np(rr.softmax(x))
    ref = oracle_mod.softmax(to_np(x))
    assert_rel_close(y, ref, 1e-5, floor=1e-30, what="softmax")
    np.testing.assert_allclose(y.astype(np.float64).sum(axis=1), 1.0, rtol=0, atol=1e-5)


def check_lnstats(rr, oracle_mod, x, eps=1e-5):
    mean, rstd = rr.layernorm_stats(x, eps)
    xh = to_np(x)
    rm, rv, rr_ = oracle_mod.layernorm_stats(xh, eps)
    xf = x.to(torch.float64).cpu().numpy()
    n = xf.shape[1]
    bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / n)
    err = np.abs(to_np(mean).astype(np.float64) - rm)
    assert (err <= bound).all(), f"mean: max err {err.max()} bound {bound[err.argmax()]}"
    assert_rel_close(to_np(rstd), rr_, 1e-5, what="rstd")


SHAPES = [(1, 1), (3, 7), (5, 8), (4, 64), (7, 100), (3, 1000), (2, 4096), (9, 4104),
          (2, 16384), (2, 20000), (1, 70001)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_softmax_small(rr, oracle_mod, dtype):
    for i, (rows, cols) in enumerate(SHAPES):
        for offset in (0, 1):
            check_softmax(rr, oracle_mod, _x(rows, cols, dtype, 200 + i, 3.0, offset))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_layernorm_small(rr, oracle_mod, dtype):
    for i, (rows, cols) in enumerate(SHAPES):
        for offset in (0, 3):
            check_lnstats(rr, oracle_mod, _x(rows, cols, dtype, 300 + i, 1.0, offset))


def test_special_rows(rr, oracle_mod):
    x = torch.full((2, 4096), 3.25, dtype=torch.bfloat16, device="cuda")
    y = to_np(rr.softmax(x))
    np.testing.assert_allclose(y, 1.0 / 4096, rtol=1e-6)
    a = 1.75
    x = torch.tensor([a, -a] * 4096, dtype=torch.bfloat16, device="cuda").view(1, -1)
    mean, rstd = rr.layernorm_stats(x, 1e-5)
    assert abs(float(mean[0])) <= 1e-6
    assert abs(float(rstd[0]) - 1.0 / np.sqrt(a * a + 1e-5)) <= 1e-5 / a
    x = torch.full((1, 8192), 2.5, dtype=torch.bfloat16, device="cuda")
    mean, rstd = rr.layernorm_stats(x, 1e-5)
    assert float(mean[0]) == 2.5
    assert abs(float(rstd[0]) - 1.0 / np.sqrt(1e-5)) <= 1e-5 / np.sqrt(1e-5)


def test_softmax_workload_full_size(rr, oracle_mod):
    # 32768 x 4096 bf16 = bf16_rn(3 * N(0,1)); sampled rows against the oracle,
    # every row's sum against 1
    from cluster_reductions_gb300 import inputs
    x = inputs.normal_bf16(32768, 4096, inputs.seed_for(3, 0), "cuda", 3.0)
    y = rr.softmax(x)
    idx = torch.tensor(np.r_[np.arange(0, 32768, 256), 32767], device="cuda")
    ref = oracle_mod.softmax(to_np(x[idx]))
    assert_rel_close(to_np(y[idx]), ref, 1e-5, floor=1e-30, what="softmax")
    s = y.to(torch.float64).sum(dim=1).cpu().numpy()
    np.testing.assert_allclose(s, 1.0, rtol=0, atol=1e-5)


def test_layernorm_workload_full_size(rr, oracle_mod):
    from cluster_reductions_gb300 import inputs
    x = inputs.normal_bf16(16384, 8192, inputs.seed_for(3, 1), "cuda")
    mean, rstd = rr.layernorm_stats(x, 1e-5)
    idx = np.r_[np.arange(0, 16384, 128), 16383]
    xs = x[torch.from_numpy(idx).cuda()]
    rm, rv, rr_ = oracle_mod.layernorm_stats(to_np(xs), 1e-5)
    xf = xs.to(torch.float64).cpu().numpy()
    bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / 8192)
    assert (np.abs(to_np(mean)[idx] - rm) <= bound).all()
    assert_rel_close(to_np(rstd)[idx], rr_, 1e-5, what="rstd")


SPLITK_SHAPES = [(1, 1000), (3, 16387), (2, 20000), (1, 65536), (4, 100003)]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("C", [1, 2, 4, 8, 16])
def test_softmax_splitk_forced(rr, oracle_mod, dtype, C):
    for i, (rows, cols) in enumerate(SPLITK_SHAPES):
        for offset in (0, 1):
            x = _x(rows, cols, dtype, 500 + i, 3.0, offset)
            try:
                y = to_np(rr.softmax(x, tier="splitk", cluster_size=C))
            except rr.RRError as e:
                if C == 16 and e.status == 2:
                    pytest.skip("cluster of 16 not schedulable")
                raise
            assert rr.last_tier() == ("splitk", C)
            ref = oracle_mod.softmax(to_np(x))
            assert_rel_close(y, ref, 1e-5, floor=1e-30, what=f"softmax splitk {rows}x{cols}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("C", [1, 2, 4, 8, 16])
def test_layernorm_splitk_forced(rr, oracle_mod, dtype, C):
    for i, (rows, cols) in enumerate(SPLITK_SHAPES):
        for offset in (0, 3):
            x = _x(rows, cols, dtype, 600 + i, 1.0, offset)
            try:
                check_lnstats_tier(rr, oracle_mod, x, C)
            except rr.RRError as e:
                if C == 16 and e.status == 2:
                    pytest.skip("cluster of 16 not schedulable")
                raise


def check_lnstats_tier(rr, oracle_mod, x, C, eps=1e-5):
    mean, rstd = rr.layernorm_stats(x, eps, tier="splitk", cluster_size=C)
    assert rr.last_tier() == ("splitk", C)
    rm, rv, rr_ = oracle_mod.layernorm_stats(to_np(x), eps)
    xf = x.to(torch.float64).cpu().numpy()
    n = xf.shape[1]
    bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / n)
    err = np.abs(to_np(mean).astype(np.float64) - rm)
    assert (err <= bound).all(), f"mean: max err {err.max()}"
    assert_rel_close(to_np(rstd), rr_, 1e-5, what="rstd splitk")


def test_splitk_rowwise_long_rows_auto(rr, oracle_mod):
    # a few very long rows: the automatic choice is split-K; every row is
    # checked against the oracle and repeated runs give the same bits
    from cluster_reductions_gb300 import inputs
    x = inputs.normal_bf16(16, 1 << 20, 4242, "cuda", 3.0)
    y = rr.softmax(x)
    assert rr.last_tier()[0] == "splitk"
    ref = oracle_mod.softmax(to_np(x))
    assert_rel_close(to_np(y), ref, 1e-5, floor=1e-30, what="softmax 16x1M")
    y2 = rr.softmax(x)
    assert torch.equal(y.view(torch.int32), y2.view(torch.int32))
    xl = inputs.normal_bf16(16, 1 << 20, 4243, "cuda", 1.0)
    mean, rstd = rr.layernorm_stats(xl, 1e-5)
    assert rr.last_tier()[0] == "splitk"
    rm, _, rr_ = oracle_mod.layernorm_stats(to_np(xl), 1e-5)
    xf = xl.to(torch.float64).cpu().numpy()
    bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / xf.shape[1])
    assert (np.abs(to_np(mean) - rm) <= bound).all()
    assert_rel_close(to_np(rstd), rr_, 1e-5, what="rstd 16x1M")
    # fp32 rows too long to stage on chip: the slice is streamed twice
    xf32 = inputs.normal_f32(4, 1 << 21, 4244, "cuda", 2.0)
    yf = rr.softmax(xf32, tier="splitk", cluster_size=2)
    assert_rel_close(to_np(yf), oracle_mod.softmax(to_np(xf32)), 1e-5, floor=1e-30,
                     what="softmax fp32 unstaged")


def check_layernorm(rr, oracle_mod, x, gamma, beta, **kw):
    from _util import assert_layernorm_close
    rows = x.shape[0]
    mean = torch.empty(rows, device="cuda")
    rstd = torch.empty(rows, device="cuda")
    y = rr.layernorm(x, gamma, beta, 1e-5, mean=mean, rstd=rstd, **kw)
    xh = to_np(x)
    y64, y16, rm, rr_ = oracle_mod.layernorm(xh, to_np(gamma), to_np(beta), 1e-5)
    xf = x.to(torch.float64).cpu().numpy()
    assert_layernorm_close(to_np(y), y64, y16, xf, to_np(gamma), to_np(beta), rm, rr_,
                           to_np(mean), to_np(rstd))
    assert_rel_close(to_np(rstd), rr_, 1e-5, what="layernorm rstd")
    return y, mean, rstd


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_layernorm_rewrite_small(rr, oracle_mod, dtype):
    from cluster_reductions_gb300 import inputs
    for i, (rows, cols) in enumerate(SHAPES):
        gamma, beta = inputs.layernorm_params(cols, 700 + i, "cuda")
        for offset in (0, 1):
            check_layernorm(rr, oracle_mod, _x(rows, cols, dtype, 710 + i, 1.0, offset), gamma, beta)


@pytest.mark.parametrize("C", [1, 2, 4, 8, 16])
def test_layernorm_rewrite_splitk(rr, oracle_mod, C):
    from cluster_reductions_gb300 import inputs
    for i, (rows, cols) in enumerate(SPLITK_SHAPES):
        gamma, beta = inputs.layernorm_params(cols, 800 + i, "cuda")
        x = _x(rows, cols, torch.bfloat16, 810 + i, 1.0, i % 2)
        try:
            check_layernorm(rr, oracle_mod, x, gamma, beta, tier="splitk", cluster_size=C)
        except rr.RRError as e:
            if C == 16 and e.status == 2:
                pytest.skip("cluster of 16 not schedulable")
            raise
        assert rr.last_tier() == ("splitk", C)


def test_layernorm_rewrite_workload_and_stats_agree(rr, oracle_mod):
    # 16384 x 8192 bf16 with gamma = 1 + 0.1 N, beta = 0.1 N: sampled rows
    # against the oracle; the fused kernel's mean / rstd are the statistics
    # kernel's, bit for bit
    from cluster_reductions_gb300 import inputs
    from _util import assert_layernorm_close
    x = inputs.normal_bf16(16384, 8192, inputs.seed_for(3, 2), "cuda")
    gamma, beta = inputs.layernorm_params(8192, inputs.seed_for(3, 3), "cuda")
    mean, rstd = torch.empty(16384, device="cuda"), torch.empty(16384, device="cuda")
    y = rr.layernorm(x, gamma, beta, 1e-5, mean=mean, rstd=rstd)
    m2, r2 = rr.layernorm_stats(x, 1e-5)
    assert torch.equal(mean.view(torch.int32), m2.view(torch.int32))
    assert torch.equal(rstd.view(torch.int32), r2.view(torch.int32))
    idx = torch.arange(0, 16384, 509, device="cuda")
    xs = x[idx]
    y64, y16, rm, rr_ = oracle_mod.layernorm(to_np(xs), to_np(gamma), to_np(beta), 1e-5)
    assert_layernorm_close(to_np(y[idx]), y64, y16, xs.to(torch.float64).cpu().numpy(),
                           to_np(gamma), to_np(beta), rm, rr_, to_np(mean[idx]), to_np(rstd[idx]))


def test_argument_errors(rr):
    with pytest.raises(rr.RRError):
        rr.softmax(torch.zeros((3, 0), device="cuda"))
    with pytest.raises(rr.RRError):
        rr.layernorm_stats(torch.zeros((3, 0), device="cuda"))
    with pytest.raises(rr.RRError):
        rr.layernorm_stats(torch.zeros((3, 4), device="cuda"), eps=-1.0)


# ---------------------------------------------------------------------------
# Warp tier: a segment of L lanes per row, up to 8 16-byte vectors per lane.
# Widths cover one vector, fewer vectors than lanes (idle lanes), ragged
# multiples of L and the largest row a segment holds; row counts cover a
# partial segment group, a partial CTA and, for one width per L, more rows
# than the persistent grid takes in one pass (the prefetch path).
# ---------------------------------------------------------------------------
def _warp_widths(L, epv):
    nv = sorted({1, max(1, L - 1), L, L + 1, 3 * L - 1, 8 * L - 1, 8 * L})
    return [n * epv for n in nv if n <= 8 * L]


def _warp_rows(L, cols, elt):
    # one more pass than a full grid needs at 2 CTAs per SM (the fewest any
    # variant gets), capped at 64 MiB of input
    many = min(152 * 2 * 8 * (32 // L) * 2 + 37, (64 << 20) // (cols * elt))
    return [1, 7, 300, many]


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("L", [1, 2, 4, 8, 16, 32])
def test_softmax_warp_forced(rr, oracle_mod, dtype, L):
    epv = 8 if dtype == torch.bfloat16 else 4
    elt = 2 if dtype == torch.bfloat16 else 4
    for i, cols in enumerate(_warp_widths(L, epv)):
        for rows in (_warp_rows(L, cols, elt) if i == len(_warp_widths(L, epv)) - 2 else [7, 300]):
            x = _x(rows, cols, dtype, 1000 + 10 * L + i, 3.0)
            y = to_np(rr.softmax(x, tier="warp", lanes_per_row=L))
            assert rr.last_tier() == ("warp", L)
            idx = np.r_[0:min(rows, 64), max(rows - 64, 0):rows]
            ref = oracle_mod.softmax(to_np(x[torch.from_numpy(idx).cuda()]))
            assert_rel_close(y[idx], ref, 1e-5, floor=1e-30, what=f"softmax warp L={L} {rows}x{cols}")
            np.testing.assert_allclose(y.astype(np.float64).sum(axis=1), 1.0, rtol=0, atol=1e-5)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("L", [1, 2, 4, 8, 16, 32])
def test_layernorm_warp_forced(rr, oracle_mod, dtype, L):
    from cluster_reductions_gb300 import inputs
    from _util import assert_layernorm_close
    epv = 8 if dtype == torch.bfloat16 else 4
    elt = 2 if dtype == torch.bfloat16 else 4
    widths = _warp_widths(L, epv)
    for i, cols in enumerate(widths):
        gamma, beta = inputs.layernorm_params(cols, 1100 + i, "cuda")
        for rows in (_warp_rows(L, cols, elt) if i == len(widths) - 1 else [7, 300]):
            x = _x(rows, cols, dtype, 1200 + 10 * L + i, 1.0)
            mean, rstd = torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda")
            y = rr.layernorm(x, gamma, beta, 1e-5, mean=mean, rstd=rstd, tier="warp",
                             lanes_per_row=L)
            assert rr.last_tier() == ("warp", L)
            m2, r2 = rr.layernorm_stats(x, 1e-5, tier="warp", lanes_per_row=L)
            assert torch.equal(mean.view(torch.int32), m2.view(torch.int32))
            assert torch.equal(rstd.view(torch.int32), r2.view(torch.int32))
            idx = np.r_[0:min(rows, 48), max(rows - 48, 0):rows]
            xs = x[torch.from_numpy(idx).cuda()]
            y64, y16, rm, rr_ = oracle_mod.layernorm(to_np(xs), to_np(gamma), to_np(beta), 1e-5)
            xf = xs.to(torch.float64).cpu().numpy()
            assert_layernorm_close(to_np(y)[idx], y64, y16, xf, to_np(gamma), to_np(beta), rm, rr_,
                                   to_np(mean)[idx], to_np(rstd)[idx])
            bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / cols)
            assert (np.abs(to_np(mean)[idx].astype(np.float64) - rm) <= bound).all()
            assert_rel_close(to_np(rstd)[idx], rr_, 1e-5, what=f"rstd warp L={L} {rows}x{cols}")


# Warp tier for rows that are not aligned 16-byte vectors (widths that are no
# vector multiple, misaligned bases): the chunked form (a row's whole
# 16-byte chunks over the lanes, head and tail elements apart) and the
# element-wise form (lane `sub` holding elements k * L + sub).  x at offset
# 0 gives outputs that share its offset within a chunk (chunked softmax and
# rewrite), offsets 1 and 3 outputs that do not (element-wise softmax and
# rewrite); the statistics are chunked throughout.  Widths: 1, ragged ones,
# the most an L-lane segment holds (4 L below 32 lanes; 1024 at 32 lanes),
# one width per L with more rows than the persistent grid takes in one pass.
def _el_widths(L):
    top = 4 * L if L < 32 else 1024
    w = {1, 3, top - 1, top} if L < 32 else {4 * 16 + 1, 127, 250, 513, 1000, 1023, 1024}
    return sorted(c for c in w if c <= top)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("L", [1, 2, 4, 8, 16, 32])
def test_rowwise_warp_elementwise_forced(rr, oracle_mod, dtype, L):
    elt = 2 if dtype == torch.bfloat16 else 4
    widths = _el_widths(L)
    for i, cols in enumerate(widths):
        for off in (0, 1, 3):
            rows_list = (_warp_rows(L, cols, elt) if (i == len(widths) - 2 and off < 2)
                         else [7, 300])
            for rows in rows_list:
                x = _x(rows, cols, dtype, 2400 + 10 * L + i, 2.0, off)
                idx = np.r_[0:min(rows, 24), max(rows - 24, 0):rows]
                _check_all_row_ops(rr, oracle_mod, x, np.unique(idx),
                                   expect_tier=(("warp", L), False), stats_bitwise=False,
                                   tier="warp", lanes_per_row=L)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_rowwise_warp_misaligned_operand_offsets(rr, oracle_mod, dtype):
    # outputs, gamma and beta each at their own offset within a 16-byte
    # chunk, matching x's or not (vector or element stores; shifted or
    # element loads of gamma / beta); x at every element offset
    from _util import assert_layernorm_close
    from cluster_reductions_gb300 import inputs
    epv = 8 if dtype == torch.bfloat16 else 4
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows = 8 * sms + 5
    for i, (cols, xo) in enumerate([(250, 1), (301, 2), (97, epv - 1), (1001, 0), (40, 3)]):
        x = _x(rows, cols, dtype, 2600 + i, 2.0, xo % epv)
        idx = np.r_[0:6, rows // 2, rows - 6:rows]
        xs = x[torch.from_numpy(idx).cuda()]
        ref = oracle_mod.softmax(to_np(xs))
        for yo in (0, 1, 2, 3):
            y = torch.empty(rows * cols + yo, device="cuda")[yo:].view(rows, cols)
            rr.softmax(x, out=y)
            assert rr.last_tier()[0] == "warp", (cols, xo, rr.last_tier())
            assert_rel_close(to_np(y)[idx], ref, 1e-5, floor=1e-30, what=f"softmax {cols} x+{xo} y+{yo}")
        g0, b0 = inputs.layernorm_params(cols + 8, 2650 + i, "cuda")
        for go, bo, oo in ((0, 0, 0), (1, 3, 1), (2, 1, 5), (3, 2, 7)):
            g, b = g0[go:go + cols], b0[bo:bo + cols]
            yb = torch.empty(rows * cols + oo, dtype=torch.bfloat16, device="cuda")[oo:].view(rows, cols)
            mean, rstd = torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda")
            rr.layernorm(x, g, b, 1e-5, out=yb, mean=mean, rstd=rstd)
            assert rr.last_tier()[0] == "warp"
            y64, y16, rm, rr_ = oracle_mod.layernorm(to_np(xs), to_np(g), to_np(b), 1e-5)
            xf = xs.to(torch.float64).cpu().numpy()
            assert_layernorm_close(to_np(yb)[idx], y64, y16, xf, to_np(g), to_np(b), rm, rr_,
                                   to_np(mean)[idx], to_np(rstd)[idx])
            bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / cols)
            assert (np.abs(to_np(mean)[idx].astype(np.float64) - rm) <= bound).all()
            assert_rel_close(to_np(rstd)[idx], rr_, 1e-5, what=f"rstd {cols} x+{xo} out+{oo}")


def test_rowwise_warp_elementwise_special(rr, oracle_mod):
    # -inf over whole lanes (elements sub, sub + L, ... of a segment), over a
    # row's first half and over a whole row; constant rows
    for L, cols in ((16, 60), (32, 250), (32, 1023)):
        x = _x(9, cols, torch.bfloat16, 2500 + cols, 3.0, 1)
        x[:, 3::L] = float("-inf")
        x[1, : cols // 2] = float("-inf")
        x[3, :] = float("-inf")
        y = to_np(rr.softmax(x, tier="warp", lanes_per_row=L))
        assert rr.last_tier() == ("warp", L)
        ref = oracle_mod.softmax(to_np(x))
        live = [r for r in range(9) if r != 3]
        assert_rel_close(y[live], ref[live], 1e-5, floor=1e-30, what=f"softmax -inf el L={L}")
        assert (y[:, 3::L] == 0).all() and (y[1, : cols // 2] == 0).all()
        assert np.isnan(ref[3]).all() and (y[3] == 0).all()
        c = torch.full((5, cols), -2.5, dtype=torch.bfloat16, device="cuda")
        np.testing.assert_allclose(to_np(rr.softmax(c, tier="warp", lanes_per_row=L)), 1.0 / cols,
                                   rtol=1e-6)
        mean, rstd = rr.layernorm_stats(c, 1e-5, tier="warp", lanes_per_row=L)
        assert (to_np(mean) == -2.5).all()
        np.testing.assert_allclose(to_np(rstd), 1.0 / np.sqrt(1e-5), rtol=1e-5)


def test_warp_rowwise_special_rows(rr, oracle_mod):
    # constant rows, alternating +-a, and -inf over whole lanes of a segment
    x = torch.full((5, 512), 3.25, dtype=torch.bfloat16, device="cuda")
    y = to_np(rr.softmax(x, tier="warp"))
    np.testing.assert_allclose(y, 1.0 / 512, rtol=1e-6)
    mean, rstd = rr.layernorm_stats(x, 1e-5, tier="warp")
    assert (to_np(mean) == 3.25).all()
    np.testing.assert_allclose(to_np(rstd), 1.0 / np.sqrt(1e-5), rtol=1e-5)
    a = 1.75
    x = torch.tensor([a, -a] * 256, dtype=torch.bfloat16, device="cuda").view(1, -1).repeat(3, 1)
    mean, rstd = rr.layernorm_stats(x, 1e-5, tier="warp", lanes_per_row=8)
    assert (np.abs(to_np(mean)) <= 1e-6).all()
    assert (np.abs(to_np(rstd) - 1.0 / np.sqrt(a * a + 1e-5)) <= 1e-5 / a).all()
    for L in (4, 8, 32):                      # L = 4 holds the 32 vectors at 8 per lane
        x = _x(9, 256, torch.bfloat16, 1300 + L, 3.0)
        x[:, :128] = float("-inf")
        x[3, :] = float("-inf")
        x[4, 255] = float("-inf")
        y = to_np(rr.softmax(x, tier="warp", lanes_per_row=L))
        ref = oracle_mod.softmax(to_np(x))
        live = [r for r in range(9) if r != 3]
        assert_rel_close(y[live], ref[live], 1e-5, floor=1e-30, what=f"softmax -inf L={L}")
        assert (y[:, :128] == 0).all()
        # an all -inf row is 0/0: the oracle's fp64 exp(-inf - -inf) is NaN, the
        # kernels write 0 (the combine's convention for a row with no mass)
        assert np.isnan(ref[3]).all() and (y[3] == 0).all()


def test_warp_rowwise_auto_and_unsupported(rr, oracle_mod):
    # AUTO takes the warp tier for many short aligned rows, with about 4
    # vectors per lane (2 for rows of up to 8 vectors); misaligned or
    # over-long rows cannot be forced onto it
    x = _x(4096, 512, torch.bfloat16, 1400, 3.0)
    rr.softmax(x)
    assert rr.last_tier() == ("warp", 16)
    rr.layernorm_stats(x[:, :64].contiguous())
    assert rr.last_tier() == ("warp", 4)
    rr.layernorm_stats(x[:, :16].contiguous())
    assert rr.last_tier() == ("warp", 1)
    from cluster_reductions_gb300 import inputs
    g, b = inputs.layernorm_params(512, 1406, "cuda")
    rr.layernorm(x, g, b, 1e-5)                                 # the rewrite: ~2 vectors per lane
    assert rr.last_tier() == ("warp", 32)
    rr.layernorm(x[:1000], g, b, 1e-5)                          # < 8 rows per SM
    assert rr.last_tier() == ("block", 1)
    xf = _x(4096, 1024, torch.float32, 1401, 1.0)
    rr.layernorm_stats(xf)
    assert rr.last_tier() == ("warp", 32)
    check_lnstats(rr, oracle_mod, xf[:200].contiguous())
    rr.softmax(x[:8])
    assert rr.last_tier() == ("block", 1)
    # rows that are not aligned vectors take the chunked or element-wise
    # form: with 16-byte aligned bases the lanes the host plan gives many
    # such rows, with x misaligned (the output then not sharing its offset)
    # the element-wise form's
    for ok in (_x(8, 100, torch.bfloat16, 1403, 1.0), _x(8, 30, torch.float32, 1407, 1.0),
               _x(8, 3, torch.bfloat16, 1410, 1.0)):
        rr.softmax(ok, tier="warp")
        assert rr.last_tier() == rr.plan_rowwise(1 << 20, ok.shape[1], "softmax", 152, 16,
                                                 dtype=ok.dtype, aligned=False)
    for ok, lanes in ((_x(8, 512, torch.bfloat16, 1402, 1.0, 1), 32),   # x not 16-byte aligned
                      (_x(8, 30, torch.float32, 1407, 1.0, 1), 8)):
        rr.softmax(ok, tier="warp")
        assert rr.last_tier() == ("warp", lanes)
    for bad in (_x(8, 4000, torch.bfloat16, 1408, 1.0, 1),     # 501 chunks > 8 per lane
                _x(8, 4096, torch.bfloat16, 1404, 1.0)):       # 512 vectors > 8 per lane
        with pytest.raises(rr.RRError) as e:
            rr.softmax(bad, tier="warp")
        assert e.value.status == 2
    with pytest.raises(rr.RRError) as e:                        # 14 chunks > 8 x 1
        rr.softmax(_x(8, 100, torch.bfloat16, 1409, 1.0), tier="warp", lanes_per_row=1)
    assert e.value.status == 2
    with pytest.raises(rr.RRError) as e:
        rr.softmax(_x(8, 1024, torch.bfloat16, 1405, 1.0), tier="warp", lanes_per_row=8)
    assert e.value.status == 2                                  # 128 vectors > 8 x 8
    for bad_l in (3, 64):
        with pytest.raises(rr.RRError) as e:
            rr.softmax(x, tier="warp", lanes_per_row=bad_l)
        assert e.value.status == 1


@pytest.mark.parametrize("tier", ["block", "splitk"])
def test_softmax_neg_inf_spans(rr, oracle_mod, tier):
    # -inf over whole threads' (or CTAs') share of a row: those elements are
    # exactly 0, the rest match the oracle; an all -inf row (0/0, NaN in the
    # oracle) is written as 0
    for cols in (4096, 20000, 65536):
        x = _x(4, cols, torch.bfloat16, 1500 + cols % 97, 3.0)
        x[:, : cols // 2] = float("-inf")
        x[2, :] = float("-inf")
        y = to_np(rr.softmax(x, tier=tier))
        ref = oracle_mod.softmax(to_np(x))
        live = [0, 1, 3]
        assert_rel_close(y[live], ref[live], 1e-5, floor=1e-30, what=f"softmax -inf {tier} {cols}")
        assert (y[:, : cols // 2] == 0).all()
        assert np.isnan(ref[2]).all() and (y[2] == 0).all()


def test_rowwise_launch_matches_host_plan(rr):
    # the tier a call takes on this device is the one rr_plan_rowwise reports
    from cluster_reductions_gb300 import inputs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for rows, cols, dt in [(4 * sms, 256, torch.bfloat16), (4 * sms - 1, 256, torch.bfloat16),
                           (8 * sms, 1024, torch.float32), (3000, 2048, torch.bfloat16),
                           (2000, 4096, torch.bfloat16), (40000, 16, torch.bfloat16),
                           (40000, 100, torch.bfloat16), (40000, 21, torch.float32),
                           (4 * sms, 1001, torch.bfloat16), (4 * sms - 1, 250, torch.bfloat16),
                           (20000, 1025, torch.float32)]:
        x = _x(rows, cols, dt, 1600 + cols, 1.0)
        g, b = inputs.layernorm_params(cols, 1601, "cuda")
        for op, call in (("softmax", lambda: rr.softmax(x)),
                         ("lnstats", lambda: rr.layernorm_stats(x)),
                         ("layernorm", lambda: rr.layernorm(x, g, b))):
            call()
            assert rr.last_tier() == rr.plan_rowwise(rows, cols, op, sms, 16, dtype=dt), (rows, cols, op)


# ---------------------------------------------------------------------------
# Staged rows: the row (or each CTA's slice of it) copied into shared memory,
# persistent clusters with two stage buffers.  Row counts above the
# persistent grid make clusters take several rows (both buffers, the
# prefetch); widths give a CTA per row, clusters of 2 and 4, ragged last
# slices and, for fp32, 4-element tails.
# ---------------------------------------------------------------------------
def _check_all_row_ops(rr, oracle_mod, x, idx, expect_tier=None, stats_bitwise=True, **kw):
    from cluster_reductions_gb300 import inputs
    from _util import assert_layernorm_close
    rows, cols = x.shape
    xs = x[torch.from_numpy(idx).cuda()]
    xh = to_np(xs)
    y = to_np(rr.softmax(x, **kw))
    # expect_tier: (tier, staged flag) or (tier, form string)
    got = (rr.last_tier(), rr.last_staged())
    if expect_tier is not None and isinstance(expect_tier[1], str):
        got = (rr.last_tier(), rr.last_form())
    if expect_tier is not None:
        assert got == expect_tier, (rows, cols, got)
    ref = oracle_mod.softmax(xh)
    assert_rel_close(y[idx], ref, 1e-5, floor=1e-30, what=f"softmax {rows}x{cols} {got}")
    np.testing.assert_allclose(y[idx].astype(np.float64).sum(axis=1), 1.0, rtol=0, atol=1e-5)
    del y
    g, b = inputs.layernorm_params(cols, 1700 + cols % 13, "cuda")
    mean, rstd = torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda")
    yb = rr.layernorm(x, g, b, 1e-5, mean=mean, rstd=rstd, **kw)
    form_rw = (rr.last_tier(), rr.last_form())
    m2, r2 = rr.layernorm_stats(x, 1e-5, **kw)
    # the two calls' statistics agree bit for bit when they take the same
    # form (the statistics alone stream long rows through the ring, where
    # the rewrite may stage them)
    if stats_bitwise and form_rw == (rr.last_tier(), rr.last_form()):
        assert torch.equal(mean.view(torch.int32), m2.view(torch.int32))
        assert torch.equal(rstd.view(torch.int32), r2.view(torch.int32))
    y64, y16, rm, rr_ = oracle_mod.layernorm(xh, to_np(g), to_np(b), 1e-5)
    xf = xs.to(torch.float64).cpu().numpy()
    assert_layernorm_close(to_np(yb)[idx], y64, y16, xf, to_np(g), to_np(b), rm, rr_,
                           to_np(mean)[idx], to_np(rstd)[idx])
    bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / cols)
    assert (np.abs(to_np(mean)[idx].astype(np.float64) - rm) <= bound).all()
    assert_rel_close(to_np(rstd)[idx], rr_, 1e-5, what=f"rstd {rows}x{cols}")
    assert (np.abs(to_np(m2)[idx].astype(np.float64) - rm) <= bound).all()
    assert_rel_close(to_np(r2)[idx], rr_, 1e-5, what=f"stats rstd {rows}x{cols}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_staged_rows_block(rr, oracle_mod, dtype):
    # a forced block tier on rows beyond the register form stages each row
    widths = [16392, 20000, 32768, 49152] if dtype == torch.bfloat16 else [8196, 10004, 24576]
    for i, cols in enumerate(widths):
        x = _x(7, cols, dtype, 1800 + i, 2.0)
        _check_all_row_ops(rr, oracle_mod, x, np.arange(7), (("block", 1), True), tier="block")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_staged_rows_auto(rr, oracle_mod, dtype):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    elt = 2 if dtype == torch.bfloat16 else 4
    cases = ([(3 * sms + 5, 20000), (sms + 9, 65544), (sms + 3, 100008)] if elt == 2 else
             [(3 * sms + 5, 10004), (sms + 9, 40004), (sms + 3, 50000)])
    for i, (rows, cols) in enumerate(cases):
        x = _x(rows, cols, dtype, 1900 + i, 2.0)
        plan = rr.plan_rowwise(rows, cols, "softmax", sms, 16, dtype=dtype, form=True)
        assert plan[2] in ("staged", "ring"), plan
        idx = np.r_[0:6, rows // 2:rows // 2 + 3, rows - 6:rows]
        # the ring's cluster width may shrink at launch; the staged form keeps it
        exp = ((plan[0], plan[1]), plan[2]) if plan[2] == "staged" else None
        _check_all_row_ops(rr, oracle_mod, x, idx, exp)


def test_staged_rows_special(rr, oracle_mod):
    # constant rows, and -inf over whole slices of a clustered row
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows, cols = sms + 1, 65544
    x = torch.full((rows, cols), 1.5, dtype=torch.bfloat16, device="cuda")
    y = rr.softmax(x)
    assert rr.last_form() in ("staged", "ring") and rr.last_tier()[0] == "splitk"
    np.testing.assert_allclose(to_np(y[:4]), 1.0 / cols, rtol=2e-6)
    mean, rstd = rr.layernorm_stats(x, 1e-5)
    assert (to_np(mean) == 1.5).all()
    x = _x(rows, cols, torch.bfloat16, 1950, 3.0)
    x[:, : cols // 2 + 100] = float("-inf")
    x[1, :] = float("-inf")
    y = to_np(rr.softmax(x)[:4])
    assert rr.last_form() in ("staged", "ring")
    ref = oracle_mod.softmax(to_np(x[:4]))
    live = [0, 2, 3]
    assert_rel_close(y[live], ref[live], 1e-5, floor=1e-30, what="staged softmax -inf")
    assert (y[:, : cols // 2 + 100] == 0).all()
    assert np.isnan(ref[1]).all() and (y[1] == 0).all()


def test_long_rows_split_fallback(rr, oracle_mod):
    # long rows too long to stage take split-K over global memory
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows, cols = sms + 2, 1 << 20
    x = _x(rows, cols, torch.bfloat16, 2000, 2.0)
    plan = rr.plan_rowwise(rows, cols, "softmax", sms, 16)
    assert plan[0] == "splitk"
    _check_all_row_ops(rr, oracle_mod, x, np.r_[0:3, rows - 3:rows], expect_tier=(plan, False))
    # (the statistics alone stream such rows through the ring, a CTA per row)
    assert rr.last_form() == "ring" and rr.last_tier() == ("block", 1)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_staged_misaligned_rows(rr, oracle_mod, dtype):
    # rows that do not start 16-byte aligned (a width that is not a vector
    # multiple, or a misaligned base): staged with their partial first and
    # last 16-byte chunks loaded element by element; a CTA per row and
    # clusters, every slice offset, outputs vector-aligned or not
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    epv = 8 if dtype == torch.bfloat16 else 4
    cases = ([(sms + 5, 20001, 0), (sms + 5, 32768, 1), (sms + 3, 50257, 0), (sms + 3, 65536, 3),
              (sms + 2, 100003, 5)] if epv == 8 else
             [(sms + 5, 10001, 0), (sms + 5, 16384, 1), (sms + 3, 25002, 0), (sms + 2, 40003, 2)])
    for i, (rows, cols, off) in enumerate(cases):
        x = _x(rows, cols, dtype, 2200 + i, 2.0, off)
        idx = np.r_[0:4, rows // 2, rows - 4:rows]
        _check_all_row_ops(rr, oracle_mod, x, idx)
        assert rr.last_staged(), (rows, cols, off, rr.last_tier())


# ---------------------------------------------------------------------------
# Chunked rows at a CTA per row (rowwise.cu, k_lnstats_ck, k_layernorm_ck):
# the statistics and the rewrite of rows that are not 16-byte aligned --
# odd widths, misaligned bases -- held as head + 16-byte vectors + tail up
# to 1024 vectors (beyond, the statistics stage and the rewrite takes the
# scalar form).  Widths from one vector to the 512-thread geometry, every
# head length, outputs and gamma / beta at their own offsets; where both
# are chunked the rewrite's mean / rstd are the statistics' bits.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_chunked_rows_statistics_and_rewrite(rr, oracle_mod, dtype):
    from _util import assert_layernorm_close
    from cluster_reductions_gb300 import inputs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    epv = 8 if dtype == torch.bfloat16 else 4
    widths = ([4099, 2057, 8191, 12289, 16383, 9] if epv == 8 else
              [2051, 1029, 4095, 6145, 8191, 5])
    for i, cols in enumerate(widths):
        rows = sms + 3 if cols > 64 else 5
        for xo in (0, 1):
            x = _x(rows, cols, dtype, 4000 + 2 * i + xo, 2.0, xo)
            idx = np.unique(np.r_[0:4, rows // 2, rows - 4:rows])
            xs = x[torch.from_numpy(idx).cuda()]
            mean, rstd = rr.layernorm_stats(x, 1e-5)
            # the statistics stage rows of more than 1024 vectors
            chunked = cols * (16 // epv) // 16 <= 1024
            assert rr.last_tier() == ("block", 1), (cols, xo)
            assert rr.last_form() == ("chunked" if chunked else "staged"), (cols, xo)
            rm, _, rr_ = oracle_mod.layernorm_stats(to_np(xs), 1e-5)
            xf = xs.to(torch.float64).cpu().numpy()
            bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / cols)
            assert (np.abs(to_np(mean)[idx].astype(np.float64) - rm) <= bound).all(), (cols, xo)
            assert_rel_close(to_np(rstd)[idx], rr_, 1e-5, what=f"chunk rstd {cols} x+{xo}")
            g0, b0 = inputs.layernorm_params(cols + 8, 4100 + i, "cuda")
            for go, bo, oo in ((0, 0, xo), (1, 3, 0), (4, 4, 3)):
                g, b = g0[go:go + cols], b0[bo:bo + cols]
                yb = torch.empty(rows * cols + oo, dtype=torch.bfloat16,
                                 device="cuda")[oo:].view(rows, cols)
                m2, r2 = torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda")
                rr.layernorm(x, g, b, 1e-5, out=yb, mean=m2, rstd=r2)
                assert rr.last_tier() == ("block", 1), (cols, xo, go, oo)
                assert rr.last_form() == ("chunked" if chunked else "direct"), (cols, xo, go, oo)
                if chunked:
                    assert_bits_equal(to_np(m2), to_np(mean))
                    assert_bits_equal(to_np(r2), to_np(rstd))
                y64, y16, rm2, rr2 = oracle_mod.layernorm(to_np(xs), to_np(g), to_np(b), 1e-5)
                assert_layernorm_close(to_np(yb)[idx], y64, y16, xf, to_np(g), to_np(b), rm2, rr2,
                                       to_np(m2)[idx], to_np(r2)[idx])


def test_chunked_rows_forced_block_and_special(rr, oracle_mod):
    # a forced block tier on a misaligned width takes the chunked form;
    # constant rows (variance 0) and rows with a large common offset
    x = _x(7, 5001, torch.bfloat16, 4200, 1.0, 3)
    _check_all_row_ops(rr, oracle_mod, x, np.arange(7), tier="block")
    c = torch.full((4, 3001), 1.25, dtype=torch.bfloat16, device="cuda")
    mean, rstd = rr.layernorm_stats(c, 1e-5)
    assert (to_np(mean) == 1.25).all()
    np.testing.assert_allclose(to_np(rstd), 1 / np.sqrt(1e-5), rtol=1e-6)
    o = (_x(4, 3001, torch.float32, 4201, 1.0, 1) + 1000.0)
    mean, rstd = rr.layernorm_stats(o, 1e-5)
    rm, _, rr_ = oracle_mod.layernorm_stats(to_np(o), 1e-5)
    of = o.to(torch.float64).cpu().numpy()
    bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((of ** 2).sum(axis=1)) / 3001)
    assert (np.abs(to_np(mean).astype(np.float64) - rm) <= bound).all()
    assert_rel_close(to_np(rstd), rr_, 1e-5, what="chunk rstd offset rows")
    # the rewrite of constant rows: (x - mean) * rstd = 0, so y = beta
    from cluster_reductions_gb300 import inputs
    g, b = inputs.layernorm_params(3001, 4202, "cuda")
    yc = rr.layernorm(c, g, b, 1e-5)
    assert rr.last_form() == "chunked"
    assert_bits_equal(to_np(yc), np.broadcast_to(to_np(b.to(torch.bfloat16)), (4, 3001)))


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_chunked_softmax_rows(rr, oracle_mod, dtype):
    # softmax of rows that are not 16-byte aligned, up to 4096 elements, at
    # a CTA per row (k_softmax_ck): odd widths, x at offsets 0 and 1, the
    # output at x's offset within a 16-byte chunk (32- and 16-byte stores);
    # an output off that offset takes another form; rows of -inf, whole and
    # within one thread's vectors; more rows than the persistent grid holds
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    epv = 8 if dtype == torch.bfloat16 else 4
    widths = [4099, 2057, 513, 4103] if epv == 8 else [4095, 2051, 1029, 4099]
    for i, cols in enumerate(widths):
        rows = 3 * sms + 7
        for xo in (0, 1):
            x = _x(rows, cols, dtype, 4300 + 2 * i + xo, 3.0, xo)
            if i == 0:
                x[1] = float("-inf")                      # a whole row
                x[2, : cols // 3] = float("-inf")         # the first third
                x[3, 5:12] = float("-inf")
            idx = np.unique(np.r_[0:6, rows // 2, rows - 4:rows])
            # the output at x's offset: elements of 4 bytes, x's of 2 or 4
            yo = xo
            y = torch.empty(rows * cols + yo, device="cuda")[yo:].view(rows, cols)
            rr.softmax(x, out=y)
            assert rr.last_tier() == ("block", 1) and rr.last_form() == "chunked", (cols, xo)
            ref = oracle_mod.softmax(to_np(x[torch.from_numpy(idx).cuda()]))
            got = to_np(y)[idx]
            # an all -inf row (0/0, NaN in the oracle) is written as 0
            live = [r for r in range(len(idx)) if not (i == 0 and idx[r] == 1)]
            assert_rel_close(got[live], ref[live], 1e-5, floor=1e-30,
                             what=f"chunked softmax {cols} x+{xo}")
            np.testing.assert_allclose(got[live].astype(np.float64).sum(axis=1), 1.0, rtol=0,
                                       atol=1e-5)
            if i == 0:
                assert np.isnan(ref[1]).all() and (got[1] == 0).all()
                assert (got[2, : cols // 3] == 0).all() and (got[3, 5:12] == 0).all()
        # an output one element off x's offset: not the chunked form
        x = _x(rows, cols, dtype, 4320 + i, 3.0, 0)
        y = torch.empty(rows * cols + 1, device="cuda")[1:].view(rows, cols)
        rr.softmax(x, out=y)
        assert rr.last_form() != "chunked", cols
        idx = np.r_[0:3, rows - 3:rows]
        assert_rel_close(to_np(y)[idx], oracle_mod.softmax(to_np(x[torch.from_numpy(idx).cuda()])),
                         1e-5, floor=1e-30, what=f"softmax {cols} y+1")


def test_chunked_rewrite_many_rows(rr, oracle_mod):
    # more rows than the persistent grid holds, so that each CTA takes
    # several rows, every head length among them (4099 = 3 mod 8), the next
    # row's vectors loaded while the current one is rewritten
    from _util import assert_layernorm_close
    from cluster_reductions_gb300 import inputs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    rows, cols = 8 * sms + 5, 4099
    x = _x(rows, cols, torch.bfloat16, 4210, 2.0, 0)
    g, b = inputs.layernorm_params(cols, 4211, "cuda")
    mean, rstd = rr.layernorm_stats(x, 1e-5)
    y = torch.empty((rows, cols), dtype=torch.bfloat16, device="cuda")
    m2, r2 = torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda")
    rr.layernorm(x, g, b, 1e-5, out=y, mean=m2, rstd=r2)
    assert rr.last_form() == "chunked"
    assert_bits_equal(to_np(m2), to_np(mean))
    assert_bits_equal(to_np(r2), to_np(rstd))
    idx = np.unique(np.r_[0:9, rows // 3:rows // 3 + 8, rows - 9:rows])
    xs = x[torch.from_numpy(idx).cuda()]
    y64, y16, rm2, rr2 = oracle_mod.layernorm(to_np(xs), to_np(g), to_np(b), 1e-5)
    assert_layernorm_close(to_np(y)[idx], y64, y16, xs.to(torch.float64).cpu().numpy(), to_np(g),
                           to_np(b), rm2, rr2, to_np(m2)[idx], to_np(r2)[idx])


# ---------------------------------------------------------------------------
# Streamed ring form (rowring.cu): slices bulk-copied piece by piece through
# a shared-memory ring, one combine per row (softmax: the (max, sum) pair;
# layernorm: the (count, mean, M2) monoid).  Shapes give empty slices
# (fewer units than CTAs), ragged last pieces and slices, several pieces
# and rows per CTA, cluster sizes that are not powers of two, and rows of
# more than 2^24 elements.
# ---------------------------------------------------------------------------
def _ring_all_ops(rr, oracle_mod, x, idx, **kw):
    _check_all_row_ops(rr, oracle_mod, x, idx, **kw)
    assert rr.last_form() == "ring", (x.shape, rr.last_tier(), rr.last_form())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("C", [1, 2, 4, 8, 16])
def test_ring_forced_splitk(rr, oracle_mod, dtype, C):
    shapes = [(1, 8), (2, 64), (3, 2056), (2, 16392), (5, 40000), (1, 131080)]
    for i, (rows, cols) in enumerate(shapes):
        x = _x(rows, cols, dtype, 2400 + i, 2.0)
        try:
            _ring_all_ops(rr, oracle_mod, x, np.arange(rows), tier="splitk", cluster_size=C)
        except rr.RRError as e:
            if C == 16 and e.status == 2:
                pytest.skip("cluster of 16 not schedulable")
            raise
        assert rr.last_tier() == ("splitk", C)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_ring_auto_few_rows(rr, oracle_mod, dtype):
    # a few long rows: clusters of about SMs / rows CTAs, one CTA per SM
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for i, (rows, cols) in enumerate([(16, 65536), (10, 100000), (3, 1 << 20), (sms - 1, 16384),
                                      (sms // 2, 24576)]):
        x = _x(rows, cols, dtype, 2500 + i, 3.0)
        idx = np.unique(np.r_[0:3, rows - 3:rows]) if rows > 6 else np.arange(rows)
        _ring_all_ops(rr, oracle_mod, x, idx, workspace=False)  # (with one: the grid form)
        t, c = rr.last_tier()
        plan = rr.plan_rowwise(rows, cols, "lnstats", sms, 16, dtype=dtype, form=True)
        assert plan[2] == "ring" and t == plan[0], (rows, cols, plan, t, c)
        if t == "splitk":  # the launch may take a smaller cluster that the device co-schedules
            assert 2 <= c <= plan[1], (rows, cols, plan, c)
        else:
            assert c == 1


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_ring_long_row_statistics(rr, oracle_mod, dtype):
    # rows beyond the register form, many of them: a CTA per row, several
    # rows per CTA, the ring running ahead across rows
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cols = 65544 if dtype == torch.bfloat16 else 32776   # rows of 128 KiB and more
    rows = 3 * sms + 7
    x = _x(rows, cols, dtype, 2600, 2.0)
    mean, rstd = rr.layernorm_stats(x, 1e-5)
    assert rr.last_form() == "ring" and rr.last_tier() == ("block", 1)
    idx = np.r_[0:5, rows // 2, rows - 5:rows]
    xs = x[torch.from_numpy(idx).cuda()]
    rm, _, rr_ = oracle_mod.layernorm_stats(to_np(xs), 1e-5)
    xf = xs.to(torch.float64).cpu().numpy()
    bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / cols)
    assert (np.abs(to_np(mean)[idx].astype(np.float64) - rm) <= bound).all()
    assert_rel_close(to_np(rstd)[idx], rr_, 1e-5, what="ring rstd")
    m2, r2 = rr.layernorm_stats(x, 1e-5)
    assert torch.equal(mean.view(torch.int32), m2.view(torch.int32))
    assert torch.equal(rstd.view(torch.int32), r2.view(torch.int32))


def test_ring_special_rows(rr, oracle_mod):
    # constant rows (variance 0), a large common offset (the (count, mean,
    # M2) merge must not cancel), one outlier, -inf over whole slices and
    # an all -inf row; 16 rows of 65536 take the automatic split-K ring
    rows, cols = 16, 65536
    x = _x(rows, cols, torch.bfloat16, 2700, 1.0)
    x[0] = 1.5
    x[1] = (x[1].float() + 1000.0).to(torch.bfloat16)
    x[2] = 0.0
    x[2, cols - 1] = 1.0e4
    x[3, : cols // 2 + 77] = float("-inf")
    x[4] = float("-inf")
    y = to_np(rr.softmax(x, workspace=False))
    assert rr.last_form() == "ring"
    ref = oracle_mod.softmax(to_np(x))
    live = [i for i in range(rows) if i != 4]
    assert_rel_close(y[live], ref[live], 1e-5, floor=1e-30, what="ring softmax special")
    assert (y[3, : cols // 2 + 77] == 0).all()
    assert np.isnan(ref[4]).all() and (y[4] == 0).all()
    xs = x[torch.tensor([0, 1, 2] + list(range(5, rows)), device="cuda")]
    mean, rstd = rr.layernorm_stats(xs, 1e-5, workspace=False)
    assert rr.last_form() == "ring"
    assert float(mean[0]) == 1.5 and float(rstd[0]) == pytest.approx(1 / np.sqrt(1e-5), rel=1e-6)
    rm, _, rr_ = oracle_mod.layernorm_stats(to_np(xs), 1e-5)
    xf = xs.to(torch.float64).cpu().numpy()
    bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / cols)
    assert (np.abs(to_np(mean).astype(np.float64) - rm) <= bound).all()
    assert_rel_close(to_np(rstd), rr_, 1e-5, what="ring rstd special")


def test_ring_repeatable_and_huge_rows(rr, oracle_mod):
    # the same call gives the same bits; a row of 2^25 elements (counts past
    # 2^24) matches the oracle
    x = _x(16, 1 << 20, torch.bfloat16, 2800, 3.0)
    y1, y2 = rr.softmax(x, workspace=False), rr.softmax(x, workspace=False)
    assert rr.last_form() == "ring"
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    from cluster_reductions_gb300 import inputs
    g, b = inputs.layernorm_params(1 << 20, 2801, "cuda")
    z1, z2 = rr.layernorm(x, g, b, workspace=False), rr.layernorm(x, g, b, workspace=False)
    assert torch.equal(z1.view(torch.int16), z2.view(torch.int16))
    xh = _x(1, 1 << 25, torch.bfloat16, 2802, 2.0)
    mean, rstd = rr.layernorm_stats(xh, 1e-5, workspace=False)
    assert rr.last_form() == "ring"
    rm, _, rr_ = oracle_mod.layernorm_stats(to_np(xh), 1e-5)
    xf = xh.to(torch.float64).cpu().numpy()
    bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / (1 << 25))
    assert (np.abs(to_np(mean).astype(np.float64) - rm) <= bound).all()
    assert_rel_close(to_np(rstd), rr_, 1e-5, what="ring rstd 2^25")


# ---------------------------------------------------------------------------
# Grid form (rowgrid.cu): G CTAs per row of a plain grid, the slices' states
# through a workspace, a second kernel folding them in one fixed order.
# Shapes give empty slices (more CTAs than 8-element units), ragged last
# slices, one slice, several units a thread, G past 32 (lanes fold several
# states each) and past 255 (the width's high byte in rr_last_tier).
# ---------------------------------------------------------------------------
def _grid_all_ops(rr, oracle_mod, x, idx, **kw):
    _check_all_row_ops(rr, oracle_mod, x, idx, **kw)
    assert rr.last_form() == "grid", (x.shape, rr.last_tier(), rr.last_form())


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
@pytest.mark.parametrize("G", [1, 3, 32, 77, 300])
def test_grid_forced_splits(rr, oracle_mod, dtype, G):
    shapes = [(1, 8), (2, 64), (3, 2056), (2, 16392), (5, 40000), (1, 131080)]
    for i, (rows, cols) in enumerate(shapes):
        x = _x(rows, cols, dtype, 3000 + i, 2.0)
        _grid_all_ops(rr, oracle_mod, x, np.arange(rows), tier="splitk", splits=G)
        assert rr.last_tier() == ("splitk", G)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_grid_auto_few_rows(rr, oracle_mod, dtype):
    # the automatic plan with the workspace the binding allocates
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for i, (rows, cols) in enumerate([(16, 65536), (10, 100000), (3, 1 << 20), (sms - 1, 16384),
                                      (sms // 2, 24576), (1, 40008)]):
        x = _x(rows, cols, dtype, 3100 + i, 3.0)
        idx = np.unique(np.r_[0:3, rows - 3:rows]) if rows > 6 else np.arange(rows)
        _grid_all_ops(rr, oracle_mod, x, idx)
        plan = rr.plan_rowwise(rows, cols, "lnstats", sms, 16, dtype=dtype, form=True,
                               with_workspace=True)
        assert plan[2] == "grid" and rr.last_tier() == plan[:2], (rows, cols, plan)


def test_grid_special_rows(rr, oracle_mod):
    # constant rows, a large common offset, one outlier, -inf over whole
    # slices and an all -inf row
    rows, cols = 16, 65536
    x = _x(rows, cols, torch.bfloat16, 3200, 1.0)
    x[0] = 1.5
    x[1] = (x[1].float() + 1000.0).to(torch.bfloat16)
    x[2] = 0.0
    x[2, cols - 1] = 1.0e4
    x[3, : cols // 2 + 77] = float("-inf")
    x[4] = float("-inf")
    y = to_np(rr.softmax(x))
    assert rr.last_form() == "grid"
    ref = oracle_mod.softmax(to_np(x))
    live = [i for i in range(rows) if i != 4]
    assert_rel_close(y[live], ref[live], 1e-5, floor=1e-30, what="grid softmax special")
    assert (y[3, : cols // 2 + 77] == 0).all()
    assert np.isnan(ref[4]).all() and (y[4] == 0).all()
    xs = x[torch.tensor([0, 1, 2] + list(range(5, rows)), device="cuda")]
    mean, rstd = rr.layernorm_stats(xs, 1e-5)
    assert rr.last_form() == "grid"
    assert float(mean[0]) == 1.5 and float(rstd[0]) == pytest.approx(1 / np.sqrt(1e-5), rel=1e-6)
    rm, _, rr_ = oracle_mod.layernorm_stats(to_np(xs), 1e-5)
    xf = xs.to(torch.float64).cpu().numpy()
    bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / cols)
    assert (np.abs(to_np(mean).astype(np.float64) - rm) <= bound).all()
    assert_rel_close(to_np(rstd), rr_, 1e-5, what="grid rstd special")


def test_grid_repeatable_and_huge_rows(rr, oracle_mod):
    # the same call gives the same bits; the statistics of the rewrite and of
    # layernorm_stats agree bit for bit; a row of 2^25 elements (counts past
    # 2^24) matches the oracle
    from cluster_reductions_gb300 import inputs
    x = _x(16, 1 << 20, torch.bfloat16, 3300, 3.0)
    y1, y2 = rr.softmax(x), rr.softmax(x)
    assert rr.last_form() == "grid"
    assert torch.equal(y1.view(torch.int32), y2.view(torch.int32))
    g, b = inputs.layernorm_params(1 << 20, 3301, "cuda")
    mu, rs = torch.empty(16, device="cuda"), torch.empty(16, device="cuda")
    z1, z2 = rr.layernorm(x, g, b, mean=mu, rstd=rs), rr.layernorm(x, g, b)
    assert rr.last_form() == "grid"
    assert torch.equal(z1.view(torch.int16), z2.view(torch.int16))
    m2, r2 = rr.layernorm_stats(x, 1e-5)
    assert rr.last_form() == "grid"
    assert torch.equal(mu.view(torch.int32), m2.view(torch.int32))
    assert torch.equal(rs.view(torch.int32), r2.view(torch.int32))
    xh = _x(1, 1 << 25, torch.bfloat16, 3302, 2.0)
    mean, rstd = rr.layernorm_stats(xh, 1e-5)
    assert rr.last_form() == "grid" and rr.last_tier()[1] > 255
    rm, _, rr_ = oracle_mod.layernorm_stats(to_np(xh), 1e-5)
    xf = xh.to(torch.float64).cpu().numpy()
    bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / (1 << 25))
    assert (np.abs(to_np(mean).astype(np.float64) - rm) <= bound).all()
    assert_rel_close(to_np(rstd), rr_, 1e-5, what="grid rstd 2^25")


def test_grid_workspace_handling(rr, oracle_mod):
    # a workspace too small for a forced G is refused; too small for the
    # automatic plan, the call plans without it; rows the form cannot take
    # (x not 16-byte aligned) refuse a forced G
    x = _x(4, 65536, torch.bfloat16, 3400, 2.0)
    small = torch.empty(4, dtype=torch.int32, device="cuda")
    with pytest.raises(rr.RRError) as e:
        rr.softmax(x, tier="splitk", splits=8, workspace=small)
    assert e.value.status == 1
    y = rr.softmax(x, workspace=small)
    assert rr.last_form() != "grid"
    assert_rel_close(to_np(y), oracle_mod.softmax(to_np(x)), 1e-5, floor=1e-30, what="no grid")
    xm = _x(4, 65536, torch.bfloat16, 3401, 2.0, offset=4)
    with pytest.raises(rr.RRError) as e:
        rr.softmax(xm, tier="splitk", splits=8)
    assert e.value.status == 2
    big = torch.empty(4 * 8 * 4, dtype=torch.int32, device="cuda")  # a state per CTA
    y = rr.softmax(x, tier="splitk", splits=8, workspace=big)
    assert rr.last_tier() == ("splitk", 8) and rr.last_form() == "grid"
    assert_rel_close(to_np(y), oracle_mod.softmax(to_np(x)), 1e-5, floor=1e-30, what="G=8")


@pytest.mark.parametrize("dtype,shape", [(torch.bfloat16, (160, 131072)), (torch.float32, (152, 65536))],
                         ids=["bf16", "f32"])
def test_twopass_rewrite(rr, oracle_mod, dtype, shape):
    # at least as many rows as SMs, rows of 256 KiB, a workspace: the
    # statistics through the ring, then the rewrite pass; its mean / rstd
    # are the statistics' bits whether they go to the caller or to the
    # workspace; a constant row gives y = beta; without a workspace (or with
    # one too small) another form
    from _util import assert_layernorm_close
    from cluster_reductions_gb300 import inputs
    rows, cols = shape
    x = _x(rows, cols, dtype, 3700, 2.0)
    x[5] = 0.75
    g, b = inputs.layernorm_params(cols, 3701, "cuda")
    mean, rstd = rr.layernorm_stats(x, 1e-5)
    assert rr.last_form() == "ring"
    m1, r1 = torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda")
    y1 = rr.layernorm(x, g, b, 1e-5, mean=m1, rstd=r1)
    assert rr.last_tier() == ("block", 1) and rr.last_form() == "twopass"
    assert_bits_equal(to_np(m1), to_np(mean))
    assert_bits_equal(to_np(r1), to_np(rstd))
    y2 = rr.layernorm(x, g, b, 1e-5)                        # statistics in the workspace
    assert rr.last_form() == "twopass"
    assert_bits_equal(to_np(y2), to_np(y1))
    m3 = torch.full((rows,), -1.0, device="cuda")
    y3 = rr.layernorm(x, g, b, 1e-5, mean=m3)               # only the mean asked for
    assert_bits_equal(to_np(m3), to_np(mean))
    assert_bits_equal(to_np(y3), to_np(y1))
    assert_bits_equal(to_np(y1)[5], to_np(b.to(torch.bfloat16)))
    idx = np.r_[0:8, rows // 2, rows - 3:rows]
    xs = x[torch.from_numpy(idx).cuda()]
    y64, y16, rm, rr_ = oracle_mod.layernorm(to_np(xs), to_np(g), to_np(b), 1e-5)
    assert_layernorm_close(to_np(y1)[idx], y64, y16, xs.to(torch.float64).cpu().numpy(), to_np(g),
                           to_np(b), rm, rr_, to_np(m1)[idx], to_np(r1)[idx])
    for ws in (False, torch.empty(4, dtype=torch.int32, device="cuda")):
        m4, r4 = torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda")
        y4 = rr.layernorm(x, g, b, 1e-5, mean=m4, rstd=r4, workspace=ws)
        assert rr.last_form() != "twopass"
        assert_layernorm_close(to_np(y4)[idx], y64, y16, xs.to(torch.float64).cpu().numpy(),
                               to_np(g), to_np(b), rm, rr_, to_np(m4)[idx], to_np(r4)[idx])


def test_grid_workspace_reused_across_shapes(rr, oracle_mod):
    # one workspace, its contents scratch, through calls of different
    # shapes, G and operations
    from cluster_reductions_gb300 import inputs
    ws = torch.full((1 << 16,), -1, dtype=torch.int32, device="cuda")
    calls = [(2, 16384, "softmax"), (2, 16384, "lnstats"), (16, 65536, "softmax"),
             (16, 65536, "lnstats"), (5, 40000, "layernorm"), (16, 65536, "layernorm"),
             (3, 1 << 20, "lnstats"), (16, 65536, "softmax")]
    for i, (rows, cols, op) in enumerate(calls):
        x = _x(rows, cols, torch.bfloat16, 3500 + i, 2.0)
        xh = to_np(x)
        if op == "softmax":
            y = rr.softmax(x, workspace=ws)
            assert_rel_close(to_np(y), oracle_mod.softmax(xh), 1e-5, floor=1e-30, what=op)
        else:
            if op == "lnstats":
                mean, rstd = rr.layernorm_stats(x, 1e-5, workspace=ws)
            else:
                g, b = inputs.layernorm_params(cols, 3600 + i, "cuda")
                mean, rstd = torch.empty(rows, device="cuda"), torch.empty(rows, device="cuda")
                rr.layernorm(x, g, b, 1e-5, mean=mean, rstd=rstd, workspace=ws)
            rm, _, rr_ = oracle_mod.layernorm_stats(xh, 1e-5)
            xf = x.to(torch.float64).cpu().numpy()
            bound = 1e-5 * np.maximum(np.abs(rm), np.sqrt((xf ** 2).sum(axis=1)) / cols)
            assert (np.abs(to_np(mean).astype(np.float64) - rm) <= bound).all(), (rows, cols, op)
            assert_rel_close(to_np(rstd), rr_, 1e-5, what=op)
        assert rr.last_form() == "grid", (rows, cols, op)


# ---------------------------------------------------------------------------
# Rows whose base is 8-byte but not 16-byte aligned (4k bf16 / 2k fp32
# columns that are not 8k / 4k, or x 8 bytes past a 16-byte boundary): the
# block tier's register form read as 8-byte vectors.  Widths give a thread
# fewer vectors than threads, 1-8 vectors a thread, the 512-thread layernorm
# geometry past 1024 vectors; more rows than one persistent wave.
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_half_vector_rows(rr, oracle_mod, dtype):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    epv = 8 if dtype == torch.bfloat16 else 4
    half = epv // 2
    rows = 3 * sms + 5
    widths = ([4100, 1028, 2052, 6148, 8188] if epv == 8 else [2050, 514, 1026, 3074, 4094])
    for i, cols in enumerate(widths):
        x = _x(rows, cols, dtype, 2900 + i, 2.0)
        idx = np.r_[0:4, rows // 2, rows - 4:rows]
        # softmax keeps 8-byte vectors in registers up to 1024 of them, then
        # holds 16-byte vectors with head and tail apart (chunked) up to 4096
        # elements and stages longer rows; the statistics and the rewrite
        # keep 8-byte vectors up to 2048
        sm_form = ("direct" if cols // half <= 1024 else
                   "chunked" if cols // epv <= (512 if epv == 8 else 1024) else "staged")
        assert rr.plan_rowwise(rows, cols, "softmax", sms, 16, dtype=dtype,
                               form=True) == ("block", 1, sm_form)
        _check_all_row_ops(rr, oracle_mod, x, idx, expect_tier=(("block", 1), sm_form))
        assert rr.last_form() == "direct"
    # an aligned width with x one 8-byte half-vector past a 16-byte boundary
    cols = 2048 if epv == 8 else 1024
    x = _x(rows, cols, dtype, 2950, 2.0, offset=half)
    _check_all_row_ops(rr, oracle_mod, x, np.r_[0:3, rows - 3:rows], expect_tier=(("block", 1), False))
