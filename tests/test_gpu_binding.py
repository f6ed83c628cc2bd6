"""The Python binding's host-buffer paths: CPU tensors in (pageable or
pinned) and CPU `out` tensors are staged through device memory and give the
same bits as the device call; a mis-shaped or mistyped `out` is refused
before anything is launched."""
import pytest
import torch

from _util import assert_bits_equal, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cluster_reductions_gb300 as rr
    rr.load()
    return rr


def _host(t, pinned):
    h = t.cpu()
    return h.pin_memory() if pinned else h


@pytest.mark.parametrize("pinned", [False, True], ids=["pageable", "pinned"])
def test_host_buffers_match_device(rr, pinned):
    from cluster_reductions_gb300 import inputs
    x = inputs.normal_f32(300, 700, 8301, "cuda")
    ref = to_np(rr.reduce(x, "sum"))
    xh = _host(x, pinned)
    got = rr.reduce(xh, "sum")
    torch.cuda.synchronize()
    assert not got.is_cuda
    assert_bits_equal(to_np(got), ref)
    oh = _host(torch.empty(300), pinned)
    assert rr.reduce(xh, "sum", out=oh) is oh
    torch.cuda.synchronize()
    assert_bits_equal(to_np(oh), ref)

    xa = inputs.normal_f32(8, 300 * 40, 8302, "cuda").view(8, 300, 40)
    ref_a = to_np(rr.reduce_axis(xa, "max", 1))
    oa = _host(torch.empty(8, 40), pinned)
    rr.reduce_axis(_host(xa, pinned), "max", 1, out=oa)
    torch.cuda.synchronize()
    assert_bits_equal(to_np(oa).reshape(-1), ref_a.reshape(-1))

    b = inputs.normal_bf16(64, 1000, 8303, "cuda", 3.0)
    ref_s = to_np(rr.softmax(b))
    os_ = _host(torch.empty(64, 1000), pinned)
    rr.softmax(_host(b, pinned), out=os_)
    m_d, r_d = rr.layernorm_stats(b)
    mh, rh = _host(torch.empty(64), pinned), _host(torch.empty(64), pinned)
    rr.layernorm_stats(_host(b, pinned), mean=mh, rstd=rh)
    g, be = inputs.layernorm_params(1000, 8304, "cuda")
    y_d = rr.layernorm(b, g, be)
    yh = _host(torch.empty(64, 1000, dtype=torch.bfloat16), pinned)
    mh2 = _host(torch.empty(64), pinned)
    rr.layernorm(_host(b, pinned), g.cpu(), be.cpu(), out=yh, mean=mh2)
    O, m, l, sc = inputs.combine_partials(4, 96, 128, 8305, "cuda")
    c_d = rr.splitk_combine(O, m, l, sc)
    ch = _host(torch.empty(96, 128, dtype=torch.bfloat16), pinned)
    rr.splitk_combine(_host(O, pinned), _host(m, pinned), _host(l, pinned), sc, out=ch)
    torch.cuda.synchronize()
    assert_bits_equal(to_np(os_).reshape(-1), ref_s.reshape(-1))
    assert_bits_equal(to_np(mh), to_np(m_d))
    assert_bits_equal(to_np(rh), to_np(r_d))
    assert (to_np(yh) == to_np(y_d)).all()
    assert_bits_equal(to_np(mh2), to_np(m_d))
    assert (to_np(ch) == to_np(c_d)).all()


def test_bad_out_refused(rr):
    x = torch.randn(16, 64, device="cuda")
    with pytest.raises(ValueError, match="shape"):
        rr.reduce(x, "sum", out=torch.empty(15, device="cuda"))
    with pytest.raises(ValueError, match="shape"):
        rr.reduce(x, "sum", out=torch.empty(16, dtype=torch.int32, device="cuda"))
    with pytest.raises(ValueError, match="shape"):
        rr.softmax(x, out=torch.empty(16, 63, device="cuda"))
    with pytest.raises(ValueError, match="shape"):
        rr.reduce_axis(x.view(4, 4, 64), "sum", 1, out=torch.empty(4, 65, device="cuda"))
    with pytest.raises(ValueError, match="shape"):
        rr.layernorm_stats(x, mean=torch.empty(17, device="cuda"))
    with pytest.raises(ValueError, match="contiguous"):
        rr.reduce(x, "sum", out=torch.empty(32, device="cuda")[::2])
