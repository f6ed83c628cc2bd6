"""Failure paths on the GPU without faulting it: an injected runtime error
surfaces as RRError and leaves the library usable; a cluster-size cap
(RR_MAX_CLUSTER) makes the co-schedulability query report larger clusters
as unavailable, so forced sizes fail with RR_ERR_UNSUPPORTED and automatic
plans shrink, with results still matching the oracle."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from _util import assert_bits_equal, assert_sum_close, to_np

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def rr():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cluster_reductions_gb300 as rr
    rr.load()
    return rr


def test_injected_error_then_recovery(rr, oracle_mod):
    from cluster_reductions_gb300 import inputs
    x = inputs.normal_f32(64, 4096, 8101, "cuda")
    rr.test_inject_error(2)
    for _ in range(2):
        with pytest.raises(rr.RRError, match="CUDA runtime error") as e:
            rr.reduce(x, "max")
        assert e.value.status == rr._lib.RR_ERR_CUDA
    got = to_np(rr.reduce(x, "max"))                       # the next call runs
    assert_bits_equal(got, oracle_mod.reduce_rows(to_np(x), "max"))
    rr.test_inject_error(5)
    rr.test_inject_error(0)                                # cleared
    rr.softmax(inputs.normal_bf16(4, 64, 8102, "cuda"))
    # validation still comes first: an invalid call reports INVALID and does
    # not consume the injected failure
    rr.test_inject_error(1)
    with pytest.raises(rr.RRError, match="invalid"):
        rr.reduce(x, "max", tier="tiled", emit_tile_width=3)  # no such tile width
    with pytest.raises(rr.RRError, match="CUDA runtime error"):
        rr.reduce(x, "sum")
    assert rr.device_status() == 0
    with pytest.raises(rr.RRError, match="invalid"):
        rr.test_inject_error(-1)


CAPPED = r"""
import json, sys, os
sys.path.insert(0, sys.argv[1])
import numpy as np
import torch
import cluster_reductions_gb300 as rr
from cluster_reductions_gb300 import inputs
rr.load()
out = {}
x = inputs.normal_f32(16, 1 << 16, 8201, "cuda")
def status_of(fn):
    try:
        fn()
        return 0
    except rr.RRError as e:
        return e.status
out["forced_c8"] = status_of(lambda: rr.reduce(x, "sum", tier="splitk", cluster_size=8))
out["sum"] = rr.reduce(x, "sum").cpu().tolist()
np.save(os.path.join(sys.argv[2], "x.npy"), x.cpu().numpy())
out["auto_tier"] = rr.last_tier()
xb = inputs.normal_bf16(16, 1 << 16, 8202, "cuda", 3.0)
y = rr.softmax(xb)
out["softmax_grid"] = [rr.last_tier(), rr.last_form()]
out["softmax_grid_rowsum_err"] = float((y.double().sum(1) - 1).abs().max())
y = rr.softmax(xb, workspace=False)
out["softmax_tier"] = rr.last_tier()
out["softmax_rowsum_err"] = float((y.double().sum(1) - 1).abs().max())
xa = inputs.normal_f32(1, 1 << 20, 8203, "cuda").view(1, 1 << 16, 16)
out["axis_max"] = rr.reduce_axis(xa, "max", 1).cpu().tolist()
np.save(os.path.join(sys.argv[2], "xa.npy"), xa.cpu().numpy())
out["axis_tier"] = rr.last_tier()
out["selftest_c8"] = status_of(lambda: rr.cluster_allreduce_selftest(8, iters=4))
out["selftest_c4"] = rr.cluster_allreduce_selftest(4, iters=64)
O, m, l, s = inputs.combine_partials(8, 256, 128, 8204, "cuda")
out["combine_pull_p8"] = status_of(lambda: rr.splitk_combine(O, m, l, s, mode="pull"))
out["combine_auto_p8"] = status_of(lambda: rr.splitk_combine(O, m, l, s))
out["status"] = rr.device_status()
print(json.dumps(out))
"""


def test_cluster_cap(oracle_mod, tmp_path):
    env = dict(os.environ, RR_MAX_CLUSTER="4")
    r = subprocess.run([sys.executable, "-c", CAPPED, ROOT, str(tmp_path)], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    UNSUPPORTED = 2
    assert out["forced_c8"] == UNSUPPORTED
    assert out["auto_tier"][0] == "splitk" and out["auto_tier"][1] <= 4
    xh = np.load(tmp_path / "x.npy")
    assert_sum_close(np.array(out["sum"], np.float32), oracle_mod.reduce_rows(xh, "sum"), xh)
    # with a workspace the few long rows take the grid form (no clusters);
    # without one, split-K clusters within the cap
    assert out["softmax_grid"][1] == "grid" and out["softmax_grid_rowsum_err"] < 1e-4
    assert out["softmax_tier"][0] == "splitk" and out["softmax_tier"][1] <= 4
    assert out["softmax_rowsum_err"] < 1e-4
    assert out["axis_tier"][1] <= 4
    xa = np.load(tmp_path / "xa.npy")
    assert_bits_equal(np.array(out["axis_max"], np.float32).reshape(-1),
                      oracle_mod.reduce_axis(xa, "max").reshape(-1))
    assert out["selftest_c8"] == UNSUPPORTED
    assert out["selftest_c4"] == 0
    assert out["combine_pull_p8"] == UNSUPPORTED
    assert out["combine_auto_p8"] == 0
    assert out["status"] == 0
