"""GPU parity of rr_reduce_axis (reduction over a non-last axis, the "reduce"
page's row_coords / ctx.axis) in every tier against the CPU oracle.

Bars, as for the last-axis reduction: int32 sum and every max / min
bit-exact; fp32 sum within 1e-5 * max(|ref|, ||x[o,:,i]||_2) of the fp64
oracle.  Small shapes span several tiles and ragged tails in every dimension,
aligned and misaligned bases; the three 256 MiB workloads are checked in full."""
import numpy as np
import pytest
import torch

from _util import assert_bits_equal, assert_sum_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cluster_reductions_gb300 as rr
    rr.load()
    return rr


def gen(shape, dtype, seed, offset=0):
    """Seeded [outer, axis, inner] input; `offset` elements of padding in
    front move the base off 16-byte alignment."""
    from cluster_reductions_gb300 import inputs
    n = int(np.prod(shape))
    if dtype == torch.int32:
        base = inputs.uniform_i32(1, n + offset, seed, "cuda")
    else:
        base = inputs.normal_f32(1, n + offset, seed, "cuda")
    return base.view(-1)[offset:].view(*shape)


def check(rr, oracle_mod, x: torch.Tensor, op: str, **kw):
    got = to_np(rr.reduce_axis(x, op, 1, **kw))
    xh = to_np(x)
    ref = oracle_mod.reduce_axis(xh, op)
    outer, axis, inner = xh.shape
    if op == "sum" and xh.dtype == np.float32:
        lines = np.ascontiguousarray(xh.transpose(0, 2, 1)).reshape(outer * inner, axis)
        assert_sum_close(got.reshape(-1), ref.reshape(-1), lines)
    else:
        r = ref.astype(xh.dtype) if xh.dtype == np.int32 else ref
        assert_bits_equal(got.reshape(-1), r.reshape(-1))


SHAPES = [(1, 1, 2), (3, 50, 7), (2, 300, 129), (5, 1000, 64), (1, 4097, 1000), (7, 33, 2),
          (4, 64, 1), (2, 513, 8), (9, 17, 12), (1, 3000, 4), (3, 7, 260), (2, 1, 33)]
# (tier, cluster_size, emit_tile_width, tile_rows, splits)
TIER_CASES = [("tiled", 0, 1, 0, 0), ("tiled", 0, 2, 0, 0), ("tiled", 0, 4, 0, 0),
              ("warp", 0, 0, 0, 0), ("warp", 0, 0, 4, 0), ("block", 0, 0, 0, 0),
              ("block", 0, 0, 8, 0), ("block", 0, 0, 0, 3), ("splitk", 2, 0, 0, 0),
              ("splitk", 4, 0, 0, 0), ("splitk", 16, 0, 0, 0), ("splitk", 4, 0, 16, 5),
              ("auto", 0, 0, 0, 0)]


def allowed(shape, offset, tier, ewt, tile_rows, splits):
    inner = shape[2]
    if inner == 1:        # the last-axis reduction: no tiles or splits
        return not tile_rows and splits <= 1
    V = 4 if (inner % 4 == 0 and offset % 4 == 0) else 1
    if tile_rows and (tile_rows % V or tile_rows // V > 32):
        return False
    if tier != "tiled":
        return True
    if ewt == 4:
        return inner % 4 == 0 and offset % 4 == 0
    if ewt == 2:
        return inner % 2 == 0 and offset % 2 == 0
    return True


@pytest.mark.parametrize("tier,C,ewt,tr,G", TIER_CASES,
                         ids=[f"{t}{c or ''}e{e}t{tr}g{g}" for t, c, e, tr, g in TIER_CASES])
@pytest.mark.parametrize("op", ["sum", "max", "min"])
@pytest.mark.parametrize("dtype", [torch.float32, torch.int32], ids=["f32", "i32"])
def test_forced_tiers_small(rr, oracle_mod, tier, C, ewt, tr, G, op, dtype):
    for i, shape in enumerate(SHAPES):
        for offset in (0, 1, 2):
            x = gen(shape, dtype, 7000 + 10 * i + offset, offset)
            kw = dict(tier=None if tier == "auto" else tier, cluster_size=C, emit_tile_width=ewt,
                      tile_rows=tr, splits=G)
            if not allowed(shape, offset, tier, ewt, tr, G):
                with pytest.raises(RuntimeError, match="invalid"):
                    rr.reduce_axis(x, op, 1, **kw)
                continue
            check(rr, oracle_mod, x, op, **kw)


def test_split_workspace_rules(rr, oracle_mod):
    """splits > 1 needs a workspace of splits * outer * inner elements; the
    automatic plan splits the axis of a shape with a single tile."""
    x = gen((2, 5000, 12), torch.float32, 7201)
    small = torch.empty(2 * 12 * 3 - 1, dtype=torch.int32, device="cuda")
    with pytest.raises(RuntimeError, match="invalid"):
        rr.reduce_axis(x, "sum", 1, tier="block", splits=3, workspace=small)
    ok = torch.empty(2 * 12 * 3, dtype=torch.int32, device="cuda")
    check(rr, oracle_mod, x, "sum", tier="block", splits=3, workspace=ok)
    with pytest.raises(RuntimeError, match="invalid"):
        rr.reduce_axis(x, "sum", 1, tier="warp", splits=2)
    y = gen((1, 1 << 20, 16), torch.float32, 7202)
    plan = rr.plan_reduce_axis(1, 1 << 20, 16, torch.cuda.get_device_properties(0).multi_processor_count, 16)
    assert plan["splits"] > 1
    for op in ("sum", "max", "min"):
        check(rr, oracle_mod, y, op)


def test_any_dim_and_empty(rr, oracle_mod):
    x = gen((4, 6, 10, 12), torch.float32, 7301)
    xh = to_np(x).astype(np.float64)
    for dim in range(4):
        got = to_np(rr.reduce_axis(x, "max", dim))
        assert_bits_equal(got.reshape(-1), xh.max(axis=dim).astype(np.float32).reshape(-1))
    # axis of length 0 writes the identity
    e = torch.empty((3, 0, 5), dtype=torch.float32, device="cuda")
    assert (to_np(rr.reduce_axis(e, "sum", 1)) == 0).all()
    assert np.isneginf(to_np(rr.reduce_axis(e, "max", 1))).all()
    ei = torch.empty((3, 0, 5), dtype=torch.int32, device="cuda")
    assert (to_np(rr.reduce_axis(ei, "min", 1)) == 2**31 - 1).all()
    # outer or inner of length 0: nothing to do
    assert rr.reduce_axis(torch.empty((0, 4, 5), device="cuda"), "sum", 1).shape == (0, 5)
    assert rr.reduce_axis(torch.empty((2, 4, 0), device="cuda"), "sum", 1).shape == (2, 0)


def test_signed_zero_and_nan(rr, oracle_mod):
    x = torch.zeros((2, 40, 64), dtype=torch.float32, device="cuda")
    x[0, :, :] = -0.0
    x[0, 17, 3] = 0.0            # max over {-0, +0} is +0, min is -0
    x[1, 5, 9] = float("nan")    # NaN propagates
    x[1, 39, 63] = float("inf")
    for tier, C in (("tiled", 0), ("warp", 0), ("block", 0), ("splitk", 4)):
        for op in ("max", "min"):
            check(rr, oracle_mod, x, op, tier=tier, cluster_size=C)


def test_splitk_deterministic(rr):
    x = gen((1, 8192, 1024), torch.float32, 7401)
    first = to_np(rr.reduce_axis(x, "sum", 1, tier="splitk", cluster_size=16))
    for _ in range(20):
        assert_bits_equal(to_np(rr.reduce_axis(x, "sum", 1, tier="splitk", cluster_size=16)), first)


WORKLOADS = [(1, 8192, 8192), (256, 1024, 256), (32768, 256, 8), (1, 1 << 22, 16)]


@pytest.mark.parametrize("shape", WORKLOADS, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("op", ["sum", "max", "min"])
def test_workloads_full_size(rr, oracle_mod, shape, op):
    x = gen(shape, torch.float32, 7500 + WORKLOADS.index(shape))
    check(rr, oracle_mod, x, op)
    if op == "sum":
        xi = gen(shape, torch.int32, 7510 + WORKLOADS.index(shape))
        check(rr, oracle_mod, xi, "sum")


@pytest.mark.parametrize("inner", [2, 3, 5, 6, 7])
@pytest.mark.parametrize("dtype", [torch.float32, torch.int32], ids=["f32", "i32"])
def test_slab_form(rr, oracle_mod, inner, dtype):
    # narrow inner widths that are not a multiple of 4: the contiguous slabs
    # x[o, :, :] with 16-byte loads, a warp per slab from 16 slabs per SM, a
    # CTA per slab from 2; axis lengths give a single group of 4 positions,
    # a 1-3 position tail and more than one fold chunk
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cases = [(16 * sms + 5, 4, "warp"), (16 * sms + 5, 1020, "warp"), (16 * sms + 5, 1023, "warp"),
             (2 * sms + 3, 5000, "block"), (2 * sms + 3, 4099, "block"), (2 * sms + 3, 20000, "block")]
    for outer, axis, tier in cases:
        if (axis * inner) % 4:
            continue
        x = gen((outer, axis, inner), dtype, 3000 + inner * 7 + axis % 97)
        p = rr.plan_reduce_axis(outer, axis, inner, sms, 16)
        assert (p["tier"], p["tile_rows"]) == (tier, inner), p
        for op in (("sum", "max", "min") if dtype == torch.float32 else ("sum", "max")):
            check(rr, oracle_mod, x, op)
            assert rr.last_tier()[0] == tier
