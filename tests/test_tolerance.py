"""CPU checks of the layernorm-rewrite tolerance (tests/_util.py): an fp32
emulation of the kernels' evaluation order passes it, and outputs with a
planted mistake (a wrong statistic, a dropped beta, an extra ulp, gamma read
at the wrong index) fail it."""
import numpy as np
import pytest
import torch

from _util import assert_layernorm_close, bf16_ord, layernorm_rewrite_bound


def _bf16_bits_of_f32(f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(f32, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _emulate_kernel(xb_bits, gamma, beta, eps):
    """fp32 statistics (pairwise numpy sum; any fp32 order within the 1e-5
    statistics tolerance), then y = bf16(fmaf(fl(fl(x - mu) * rs), g, b)).
    The fused multiply-add is emulated exactly: fl(x - mu) * rs is rounded
    to fp32, its product with gamma is exact in fp64 (24 + 24 bits) and the
    fp64 sum with beta is rounded to fp32 (a double rounding that is off by
    at most 2^-53 relative, inside the bound's slack in practice)."""
    x = (xb_bits.astype(np.uint32) << 16).view(np.float32)
    n = x.shape[1]
    mu = (x.sum(axis=1, dtype=np.float32) / np.float32(n)).astype(np.float32)
    d = (x - mu[:, None]).astype(np.float32)
    var = ((d * d).sum(axis=1, dtype=np.float32) / np.float32(n)).astype(np.float32)
    rs = (np.float32(1.0) / np.sqrt(var + np.float32(eps))).astype(np.float32)
    t2 = (d * rs[:, None]).astype(np.float32)
    f = (t2.astype(np.float64) * gamma.astype(np.float64)[None, :] +
         beta.astype(np.float64)[None, :]).astype(np.float32)
    return x.astype(np.float64), mu, rs, f


def _case(oracle_mod, rows=24, cols=1000, seed=5):
    g = torch.Generator().manual_seed(seed)
    xb = torch.randn(rows, cols, generator=g).to(torch.bfloat16)
    xb_bits = xb.view(torch.int16).numpy().view(np.uint16)
    gamma = (1.0 + 0.1 * torch.randn(cols, generator=g)).numpy().astype(np.float32)
    beta = (0.1 * torch.randn(cols, generator=g)).numpy().astype(np.float32)
    xf, mu, rs, f = _emulate_kernel(xb_bits, gamma, beta, 1e-5)
    y64, y16, rm, rr_ = oracle_mod.layernorm(xb_bits, gamma, beta, 1e-5)
    return xf, gamma, beta, mu, rs, f, y64, y16, rm, rr_


def test_emulated_kernel_passes(oracle_mod):
    xf, gamma, beta, mu, rs, f, y64, y16, rm, rr_ = _case(oracle_mod)
    n = assert_layernorm_close(_bf16_bits_of_f32(f), y64, y16, xf, gamma, beta, rm, rr_, mu, rs)
    assert n <= 2


def test_step2_bound_covers_the_fp32_evaluation(oracle_mod):
    # |f - z| <= e for the emulated fp32 value itself, before the bf16 rounding
    xf, gamma, beta, mu, rs, f, *_ = _case(oracle_mod, seed=6)
    z, e = layernorm_rewrite_bound(xf, gamma, beta, mu, rs)
    assert (np.abs(f.astype(np.float64) - z) <= e).all()
    # and the bound is not vacuous: well under a bf16 ulp of the outputs
    assert np.median(e / np.maximum(np.abs(z), 1e-30)) < 2.0 ** -20


@pytest.mark.parametrize("plant", ["mean", "rstd", "beta", "ulp", "gamma_index"])
def test_planted_mistakes_fail(oracle_mod, plant):
    xf, gamma, beta, mu, rs, f, y64, y16, rm, rr_ = _case(oracle_mod, seed=7)
    km, kr, y = mu.copy(), rs.copy(), f.copy()
    if plant == "mean":          # a mean off by far more than 1e-5 of the row scale
        km = (km + np.float32(1e-3)).astype(np.float32)
    elif plant == "rstd":
        kr = (kr * np.float32(1.001)).astype(np.float32)
    elif plant == "beta":        # the rewrite drops beta
        y = (f - beta[None, :]).astype(np.float32)
    elif plant == "gamma_index":  # gamma read one element off
        t = (f - beta[None, :]) / gamma[None, :]
        y = (t * np.roll(gamma, 1)[None, :] + beta[None, :]).astype(np.float32)
    bits = _bf16_bits_of_f32(y)
    if plant == "ulp":            # one output moved by two bf16 ulps
        o = bf16_ord(bits[3:4, 10:11])[0, 0] + 2
        bits = bits.copy()
        bits[3, 10] = o if o >= 0 else (0x8000 | -o)
    with pytest.raises(AssertionError):
        assert_layernorm_close(bits, y64, y16, xf, gamma, beta, rm, rr_, km, kr)


def test_splitmix64_published_outputs():
    # the first three outputs of the generator started from state 0, as
    # printed with its reference implementation
    from _util import splitmix64
    g = 0x9E3779B97F4A7C15
    with np.errstate(over="ignore"):
        got = splitmix64(np.array([0, g, (2 * g) % (1 << 64)], dtype=np.uint64))
    assert [int(v) for v in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
