"""GPU parity of rr_reduce in every tier against the CPU oracle.

Bars: int32 sum and every max / min bit-exact; fp32 sum within
1e-5 * max(|ref|, ||x_row||_2) of the fp64 oracle.  Small shapes span several
tiles, ragged tails and misaligned rows; the full workload sizes are checked
on every row the oracle can afford (all rows for the warp, tiled and split-K
workloads, sampled rows for 8192 x 8192)."""
import numpy as np
import pytest
import torch

from _util import assert_bits_equal, assert_sum_close, to_np

pytestmark = pytest.mark.gpu

TIERS = ["warp", "tiled", "block", "splitk"]


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cluster_reductions_gb300 as rr
    rr.load()
    return rr


def check(rr, oracle_mod, x: torch.Tensor, op: str, **kw):
    got = to_np(rr.reduce(x, op, **kw))
    xh = to_np(x)
    ref = oracle_mod.reduce_rows(xh, op)
    if op == "sum" and xh.dtype == np.float32:
        assert_sum_close(got, ref, xh)
    else:
        assert_bits_equal(got, ref.astype(xh.dtype) if xh.dtype == np.int32 else ref)


def gen(rows, cols, dtype, seed, offset=0):
    """Seeded input; `offset` elements of padding in front make the rows
    start off 16-byte boundaries."""
    from cluster_reductions_gb300 import inputs
    if dtype == torch.int32:
        base = inputs.uniform_i32(1, rows * cols + offset, seed, "cuda")
    else:
        base = inputs.normal_f32(1, rows * cols + offset, seed, "cuda")
    return base.view(-1)[offset:].view(rows, cols)


SHAPES = [(1, 1), (3, 3), (5, 4), (7, 5), (9, 8), (4, 13), (6, 16), (5, 17), (7, 20), (9, 24),
          (5, 28), (33, 31), (65, 32), (3, 33), (2, 100), (9, 1000), (4, 4099), (3, 8192)]


@pytest.mark.parametrize("tier", TIERS)
@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.int32], ids=["f32", "i32"])
def test_forced_tiers_small(rr, oracle_mod, tier, op, dtype):
    for i, (rows, cols) in enumerate(SHAPES):
        for offset in (0, 1, 3):
            x = gen(rows, cols, dtype, 100 + i, offset)
            kw = {"tier": tier}
            if tier == "splitk":
                for C in (1, 2, 4):
                    check(rr, oracle_mod, x, op, tier=tier, cluster_size=C)
                continue
            if tier == "tiled":
                for e in (1, 2, 4):
                    check(rr, oracle_mod, x, op, tier=tier, emit_tile_width=e)
                continue
            check(rr, oracle_mod, x, op, **kw)


@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.int32], ids=["f32", "i32"])
def test_block_long_rows(rr, oracle_mod, op, dtype):
    # rows of >= 32768 elements take the block kernel with 16 loads per
    # thread: exactly one and two passes of them, ragged tails, misaligned
    # bases, and a few-rows-per-SM count
    for i, (rows, cols) in enumerate([(3, 32768), (2, 32769), (4, 65536 + 4 * 256 + 3),
                                      (5, 100003), (160, 40000)]):
        for offset in (0, 1, 3):
            check(rr, oracle_mod, gen(rows, cols, dtype, 150 + i, offset), op, tier="block")


@pytest.mark.parametrize("op", ["sum", "max", "min"])
def test_auto_tier_and_empty(rr, oracle_mod, op):
    for rows, cols in [(0, 5), (4, 0), (1, 0)]:
        x = torch.zeros((rows, cols), device="cuda")
        got = to_np(rr.reduce(x, op))
        ref = oracle_mod.reduce_rows(to_np(x), op)
        assert_bits_equal(got, ref)
    for rows, cols in [(1000, 7), (1000, 24), (300, 2000), (3, 70000)]:
        check(rr, oracle_mod, gen(rows, cols, torch.float32, 7), op)


def test_signed_zero_nan_all_tiers(rr, oracle_mod):
    rows = [[0.0, -0.0, -0.0, 0.0], [-0.0, -0.0, -0.0, -0.0], [0.0, 0.0, 0.0, 0.0],
            [1.0, float("nan"), 2.0, -3.0], [-1.0, -2.0, -0.0, float("nan")]]
    x = torch.tensor(rows, dtype=torch.float32, device="cuda")
    for tier in TIERS:
        for op in ("max", "min"):
            got = to_np(rr.reduce(x, op, tier=tier,
                                  **({"cluster_size": 2} if tier == "splitk" else {})))
            ref = oracle_mod.reduce_rows(to_np(x), op)
            assert_bits_equal(got[:3], ref[:3])
            assert np.isnan(got[3:]).all()
            assert (to_np(torch.from_numpy(got[3:]).view(torch.int32)) == 0x7fc00000).all()


def test_small_splitk_workload(rr, oracle_mod):
    # 64 x 4096, x ~ U[-1, 1], sum / max / min, plus int32 sum; cluster 1 and 2
    from cluster_reductions_gb300 import inputs
    for oi, op in enumerate(["sum", "max", "min"]):
        x = inputs.uniform_f32(64, 4096, inputs.seed_for(0, oi), "cuda")
        for C in (1, 2):
            check(rr, oracle_mod, x, op, tier="splitk", cluster_size=C)
        check(rr, oracle_mod, x, op)
        assert rr.last_tier()[0] == "splitk"
    xi = inputs.uniform_i32(64, 4096, inputs.seed_for(0, 3), "cuda")
    for C in (1, 2):
        check(rr, oracle_mod, xi, "sum", tier="splitk", cluster_size=C)


def test_block_workload_full_size(rr, oracle_mod):
    # 8192 x 8192; the kernel runs on the whole matrix, the oracle checks
    # every 64th row plus the last one
    from cluster_reductions_gb300 import inputs
    idx = np.r_[np.arange(0, 8192, 64), 8191]
    for oi, op in enumerate(["sum", "max", "min"]):
        x = inputs.normal_f32(8192, 8192, inputs.seed_for(1, oi), "cuda")
        got = to_np(rr.reduce(x, op))
        assert rr.last_tier() == ("block", 1)
        xs = to_np(x[torch.from_numpy(idx).cuda()])
        ref = oracle_mod.reduce_rows(xs, op)
        if op == "sum":
            assert_sum_close(got[idx], ref, xs)
        else:
            assert_bits_equal(got[idx], ref)
        del x
    xi = inputs.uniform_i32(8192, 8192, inputs.seed_for(1, 3), "cuda")
    got = to_np(rr.reduce(xi, "sum"))
    # every row: int64 sums of |x| <= 2^15 over 8192 columns cannot wrap
    assert_bits_equal(got, xi.to(torch.int64).sum(dim=1).to(torch.int32).cpu().numpy())
    xs = to_np(xi[torch.from_numpy(idx).cuda()])
    assert_bits_equal(got[idx], oracle_mod.reduce_rows(xs, "sum"))


@pytest.mark.parametrize("cols,tier", [(32, "warp"), (8, "tiled")])
def test_narrow_workloads_full_size(rr, oracle_mod, cols, tier):
    from cluster_reductions_gb300 import inputs
    rows = 1 << 20
    for oi, op in enumerate(["sum", "max", "min"]):
        x = inputs.normal_f32(rows, cols, inputs.seed_for(1, 4 + oi), "cuda")
        got = to_np(rr.reduce(x, op))
        assert rr.last_tier() == (tier, 1)
        xh = to_np(x)
        ref = oracle_mod.reduce_rows(xh, op)
        if op == "sum":
            assert_sum_close(got, ref, xh)
        else:
            assert_bits_equal(got, ref)


def test_splitk_workload_full_size(rr, oracle_mod):
    # 16 x 16,777,216 fp32, sum and max, cluster 2 / 4 / 8 / 16; all 16 rows
    # against the oracle, every rank's copy bit-identical
    from cluster_reductions_gb300 import inputs
    rows, cols = 16, 1 << 24
    x = inputs.normal_f32(rows, cols, inputs.seed_for(2, 0), "cuda")
    xh = to_np(x)
    for op in ("sum", "max"):
        ref = oracle_mod.reduce_rows(xh, op)
        for C in (2, 4, 8, 16):
            rank_out = torch.empty(rows * C, dtype=torch.float32, device="cuda")
            try:
                got = to_np(rr.reduce(x, op, tier="splitk", cluster_size=C, rank_out=rank_out))
            except rr.RRError as e:
                if C == 16 and e.status == 2:
                    continue   # cluster of 16 not schedulable on this device
                raise
            if op == "sum":
                assert_sum_close(got, ref, xh)
            else:
                assert_bits_equal(got, ref)
            ro = to_np(rank_out).reshape(rows, C)
            assert (ro.view(np.uint32) == got.view(np.uint32)[:, None]).all()
    got = rr.reduce(x, "sum")
    assert rr.last_tier()[0] == "splitk"


def test_splitk_bit_identical_100_runs(rr):
    from cluster_reductions_gb300 import inputs
    x = inputs.normal_f32(16, 1 << 22, inputs.seed_for(2, 1), "cuda")
    for C in (2, 8):
        first = rr.reduce(x, "sum", tier="splitk", cluster_size=C).clone()
        outs = torch.empty((100, 16), dtype=torch.float32, device="cuda")
        for i in range(100):
            rr.reduce(x, "sum", tier="splitk", cluster_size=C, out=outs[i])
        assert (outs.view(torch.int32) == first.view(torch.int32)).all()


@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.int32], ids=["f32", "i32"])
def test_splitk_multi_small(rr, oracle_mod, op, dtype):
    for i, (rows, cols) in enumerate([(1, 1), (2, 100), (3, 4099), (1, 70000), (2, 33333)]):
        for C, G in ((1, 1), (2, 3), (4, 0), (16, 7), (0, 0)):
            x = gen(rows, cols, dtype, 900 + i, i % 3)
            try:
                got = to_np(rr.reduce_splitk_multi(x, op, cluster_size=C, clusters_per_row=G))
            except rr.RRError as e:
                if C == 16 and e.status == 2:
                    continue
                raise
            xh = to_np(x)
            ref = oracle_mod.reduce_rows(xh, op)
            if op == "sum" and dtype == torch.float32:
                assert_sum_close(got, ref, xh)
            else:
                assert_bits_equal(got, ref.astype(xh.dtype) if dtype == torch.int32 else ref)


def test_splitk_multi_long_rows(rr, oracle_mod):
    # two rows of 64M fp32: one 16-CTA cluster per row would use 32 SMs; the
    # automatic G spreads each row over enough clusters to cover the GPU
    from cluster_reductions_gb300 import inputs
    x = inputs.normal_f32(2, 1 << 26, inputs.seed_for(2, 5), "cuda")
    xh = to_np(x)
    for op in ("sum", "max"):
        got = rr.reduce_splitk_multi(x, op)
        ref = oracle_mod.reduce_rows(xh, op)
        if op == "sum":
            assert_sum_close(to_np(got), ref, xh)
        else:
            assert_bits_equal(to_np(got), ref)
        for _ in range(10):   # the same bits every run
            assert torch.equal(rr.reduce_splitk_multi(x, op).view(torch.int32), got.view(torch.int32))
    # one cluster per row gives the single-cluster split-K tier's bits
    a = rr.reduce_splitk_multi(x, "sum", cluster_size=8, clusters_per_row=1)
    b = rr.reduce(x, "sum", tier="splitk", cluster_size=8)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_argument_errors(rr):
    x = torch.zeros((4, 8), device="cuda")
    with pytest.raises(rr.RRError) as e:
        rr.reduce(x, "sum", tier="warp", out=None, emit_tile_width=3)
    assert e.value.status == 1
    with pytest.raises(rr.RRError):
        rr.reduce(torch.zeros((4, 64), device="cuda"), "sum", tier="splitk", cluster_size=3)
    with pytest.raises(rr.RRError):
        rr.reduce(x, "sum", out=x.view(-1)[:4])   # out overlaps x
    with pytest.raises(TypeError):
        rr.reduce(torch.zeros((4, 8), device="cuda", dtype=torch.float64), "sum")


@pytest.mark.parametrize("rows,cols,offset", [(1 << 20, 64, 0), (65536, 1024, 0), (262144, 256, 1),
                                              (671088, 100, 0), (2033601, 33, 0)])
def test_medium_width_rows(rr, oracle_mod, rows, cols, offset):
    """Rows of 33 to 4095 elements and at least an SM's count of them take the
    warp tier (a warp segment per row): all ops against the oracle on every
    row of a sampled set, vector and scalar paths."""
    x = gen(rows, cols, torch.float32, 300 + cols, offset)
    idx = np.r_[np.arange(0, rows, max(1, rows // 4096)), rows - 1]
    xs = to_np(x[torch.from_numpy(idx).cuda()])
    for op in ("sum", "max", "min"):
        got = to_np(rr.reduce(x, op))
        assert rr.last_tier() == ("warp", 1)
        ref = oracle_mod.reduce_rows(xs, op)
        if op == "sum":
            assert_sum_close(got[idx], ref, xs)
        else:
            assert_bits_equal(got[idx], ref)
    xi = gen(rows, cols, torch.int32, 400 + cols, offset)
    got = to_np(rr.reduce(xi, "sum"))
    assert_bits_equal(got[idx], oracle_mod.reduce_rows(to_np(xi[torch.from_numpy(idx).cuda()]), "sum"))
