"""GPU parity of rr_splitk_combine against the fp64 oracle: every output
within 1 bf16 ulp of the oracle's correctly rounded bf16 value, except where
sum_p w_p O_p cancels far below its summands; there the bound is one ulp
plus the fp32 rounding bound of the weighted sum (see _util.combine_fp32_bound),
and such outputs must stay rare."""
import numpy as np
import pytest
import torch

from _util import assert_bf16_ulp, assert_combine_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cluster_reductions_gb300 as rr
    rr.load()
    return rr


def shape_supported(P, D, mode):
    """Whether a combine variant takes (P, D) for aligned operands, as
    rr_splitk_combine_ex documents: pull needs P a power of two and
    D % 4P == 0; push P a power of two, D % 4 == 0 and D <= 256; direct P a
    power of two, D % 4 == 0 and 2 P D 4 bytes <= 96 KiB; generic and the
    automatic choice take every P <= 16 and D <= 1024."""
    pow2 = P in (1, 2, 4, 8, 16)
    if mode == "pull":
        return pow2 and D % (4 * P) == 0
    if mode == "push":
        return pow2 and D % 4 == 0 and D <= 256
    if mode == "direct":
        return pow2 and D % 4 == 0 and 2 * P * D * 4 <= 96 * 1024
    return P <= 16 and D <= 1024


def run(rr, oracle_mod, P, rows, D, seed, mode=None):
    from cluster_reductions_gb300 import inputs
    O, m, l, s = inputs.combine_partials(P, rows, D, seed, "cuda")
    if not shape_supported(P, D, mode):
        # a variant that does not take the shape must say so, not run
        with pytest.raises(rr.RRError) as ei:
            rr.splitk_combine(O, m, l, s, mode=mode)
        assert ei.value.status == 2
        pytest.skip(f"variant {mode} does not take P={P}, D={D}")
    out = rr.splitk_combine(O, m, l, s, mode=mode)
    Oh, mh, lh = to_np(O), to_np(m), to_np(l)
    ref64, ref = oracle_mod.splitk_combine(Oh, mh, lh, s)
    assert_combine_close(to_np(out), ref64, ref, Oh, mh, lh, s)


MODES = [None, "pull", "push", "generic", "direct"]


@pytest.mark.parametrize("mode", MODES, ids=lambda m: m or "auto")
@pytest.mark.parametrize("P", [1, 2, 3, 4, 8, 16])
@pytest.mark.parametrize("D", [256, 128, 64, 16, 12, 7, 3])
def test_combine_small(rr, oracle_mod, P, D, mode):
    # 132 and 260 rows: multiples of 4, so (m, l) ride the copy engine in the
    # direct variant, with a short last tile
    for rows in (1, 5, 33, 130, 132, 257, 260):
        run(rr, oracle_mod, P, rows, D, 400 + P * 7 + D + rows, mode)


def test_combine_modes_agree_bitwise(rr):
    # every variant folds in rank order with the same fp32 operations per
    # output, so they agree bit for bit
    from cluster_reductions_gb300 import inputs
    for P, rows, D in ((2, 1000, 128), (8, 517, 128), (4, 64, 64), (16, 96, 128)):
        O, m, l, s = inputs.combine_partials(P, rows, D, 77 + P, "cuda")
        outs = {}
        for mode in ("pull", "push", "direct", "generic"):
            assert shape_supported(P, D, mode), (P, D, mode)
            outs[mode] = rr.splitk_combine(O, m, l, s, mode=mode).view(torch.int16)
        ref = outs.pop("generic")
        for mode, o in outs.items():
            assert torch.equal(o, ref), (P, rows, D, mode)


@pytest.mark.parametrize("mode", [None, "pull", "push", "direct"], ids=lambda m: m or "auto")
@pytest.mark.parametrize("P", [2, 4, 8])
def test_combine_workload_full_size(rr, oracle_mod, P, mode):
    # rows = 32 batch x 32 heads x 128 queries = 131072, D = 128; the oracle
    # checks a strided sample of rows
    from cluster_reductions_gb300 import inputs
    rows, D = 131072, 128
    O, m, l, s = inputs.combine_partials(P, rows, D, inputs.seed_for(4, P), "cuda")
    out = rr.splitk_combine(O, m, l, s, mode=mode)
    idx = torch.arange(0, rows, 97, device="cuda")
    Oh, mh, lh = to_np(O[:, idx]), to_np(m[:, idx]), to_np(l[:, idx])
    ref64, ref = oracle_mod.splitk_combine(Oh, mh, lh, s)
    assert_combine_close(to_np(out[idx]), ref64, ref, Oh, mh, lh, s)


def test_combine_special_cases(rr, oracle_mod):
    P, rows, D = 4, 40, 128
    from cluster_reductions_gb300 import inputs
    O, m, l, s = inputs.combine_partials(P, rows, D, 9, "cuda")
    m[:, 0] = float("-inf")            # every partition empty -> 0
    l[:, 1] = 0.0                      # zero mass -> 0
    m[2, 2] += 1000.0                  # one dominant partition -> its O / l
    m[:, 3] = m[0, 3]                  # equal maxima -> sum O / sum l
    out = rr.splitk_combine(O, m, l, s)
    got = to_np(out)
    assert (got[0] == 0).all() and (got[1] == 0).all()
    Oh, mh, lh = to_np(O), to_np(m), to_np(l)
    ref64, ref = oracle_mod.splitk_combine(Oh, mh, lh, s)
    assert_combine_close(got, ref64, ref, Oh, mh, lh, s)
    # P = 1: O / l, one fp32 division: within 1 ulp everywhere
    out1 = rr.splitk_combine(O[:1].contiguous(), m[:1].contiguous(), l[:1].contiguous(), s)
    _, ref1 = oracle_mod.splitk_combine(Oh[:1], mh[:1], lh[:1], s)
    assert_bf16_ulp(to_np(out1)[2:], ref1[2:])


def test_combine_deterministic(rr):
    from cluster_reductions_gb300 import inputs
    O, m, l, s = inputs.combine_partials(8, 4096, 128, 11, "cuda")
    a = rr.splitk_combine(O, m, l, s).clone()
    for _ in range(20):
        assert torch.equal(rr.splitk_combine(O, m, l, s).view(torch.int16), a.view(torch.int16))


def test_combine_argument_errors(rr):
    O = torch.zeros((2, 4, 8), device="cuda")
    m = torch.zeros((2, 4), device="cuda")
    with pytest.raises(rr.RRError):
        rr.splitk_combine(torch.zeros((17, 4, 8), device="cuda"), torch.zeros((17, 4), device="cuda"),
                          torch.zeros((17, 4), device="cuda"), 1.0)
    with pytest.raises(rr.RRError):
        rr.splitk_combine(O, m, m.clone(), float("nan"))
