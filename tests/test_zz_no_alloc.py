"""GPU test of rr_cluster_allreduce_selftest_noalloc, the self-test variant
for callers that cannot allocate device memory (a process whose memory pool
already holds the whole GPU, or one that must not risk the implicit device
synchronisation of cudaMalloc / cudaFree).  It must give the same result as
rr_cluster_allreduce_selftest, call after call, while running out of the
library's fixed device array.

This file is collected last on purpose, so that a run stopping at the first
failure has run every other test before it; it also passes on its own in a
fresh process."""
import ctypes
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import cluster_reductions_gb300 as rr
    return rr.load()


def _call(fn, *args):
    n = ctypes.c_int64(-7)
    stream = torch.cuda.current_stream().cuda_stream
    st = fn(*args, stream, ctypes.byref(n))
    return st, n.value


@pytest.mark.parametrize("C,width,op,dtype,two_slot", [
    (2, 1, 0, 0, 1), (4, 2, 0, 0, 1), (8, 4, 1, 0, 0), (4, 8, 0, 1, 0), (2, 2, 2, 1, 1)])
def test_noalloc_matches_allocating_selftest_twice(lib, C, width, op, dtype, two_slot):
    iters = 512
    for call in range(2):                     # two calls in a row share the array
        seed = 100 + call
        ref_st, ref_n = _call(lib.rr_cluster_allreduce_selftest, C, width, op, dtype, iters,
                              two_slot, seed)
        st, n = _call(lib.rr_cluster_allreduce_selftest_noalloc, C, width, op, dtype, iters,
                      two_slot, seed)
        assert (st, n) == (ref_st, ref_n)
        assert (st, n) == (0, 0)


def test_noalloc_rejects_more_than_its_scratch(lib):
    # 2 clusters * 16 CTAs * 8 values * 1025 iterations > 2^18 values
    st, n = _call(lib.rr_cluster_allreduce_selftest_noalloc, 16, 8, 0, 0, 1025, 1, 1)
    assert st == 1 and n == -7               # RR_ERR_INVALID, output untouched
    st, n = _call(lib.rr_cluster_allreduce_selftest_noalloc, 16, 8, 0, 0, 1024, 1, 1)
    if st == 2:
        pytest.skip("cluster of 16 not schedulable")
    assert (st, n) == (0, 0)                 # exactly at the limit is accepted


def test_noalloc_from_two_host_threads(lib):
    """Calls from several host threads share the one scratch array; the
    library runs them one after another, so every call still checks out."""
    import threading
    import torch
    import cluster_reductions_gb300 as rr
    results, errors = [], []

    def worker(C, width, seed):
        try:
            torch.cuda.set_device(0)
            s = torch.cuda.Stream()
            with torch.cuda.stream(s):
                for i in range(20):
                    results.append(rr.cluster_allreduce_selftest_noalloc(
                        C, width=width, op="sum", iters=256, seed=seed + i))
        except Exception as e:  # reported below
            errors.append(e)

    ts = [threading.Thread(target=worker, args=(4, 8, 100)),
          threading.Thread(target=worker, args=(8, 4, 900))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    assert results == [0] * 40


@pytest.mark.parametrize("C,width,op,dtype", [
    (2, 1, "sum", torch.float32), (4, 8, "max", torch.int32), (8, 2, "sum", torch.int32),
    (4, 4, "min", torch.float32)])
def test_noalloc_results_checked_on_host(lib, oracle_mod, C, width, op, dtype):
    """The inputs and every rank's results, copied out of the fixed array:
    the inputs equal the documented seeded generator recomputed here, and each
    result equals the oracle's rank-order fold of its inputs.  This does not
    rest on the kernel's own re-fold, which shares its operator with the
    all-reduce."""
    import cluster_reductions_gb300 as rr
    from _util import selftest_values
    iters = 400
    for seed in (5, 6):                           # two calls in a row
        n, vals, res = rr.cluster_allreduce_selftest_dump(C, width, op, dtype, iters,
                                                         True, seed, noalloc=True)
        assert n == 0
        np_dt = np.float32 if dtype == torch.float32 else np.int32
        want = selftest_values(vals.size, seed, np_dt).reshape(vals.shape)
        assert (vals.view(np.uint32) == want.view(np.uint32)).all()
        for t in range(iters):
            for c in range(2):
                ref = oracle_mod.cluster_fold(vals[t, c], op).view(np.uint32)
                assert (res[t, c].view(np.uint32) == ref[None, :]).all(), (seed, t, c)


def test_noalloc_leaves_device_memory_alone(lib):
    """Once the library's modules are loaded (a first call), a call changes
    neither the device's free memory nor torch's allocator."""
    st, n = _call(lib.rr_cluster_allreduce_selftest_noalloc, 4, 2, 0, 0, 256, 1, 11)
    assert (st, n) == (0, 0)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    reserved0 = torch.cuda.memory_reserved()
    for seed in (12, 13, 14):
        st, n = _call(lib.rr_cluster_allreduce_selftest_noalloc, 4, 2, 0, 0, 256, 1, seed)
        assert (st, n) == (0, 0)
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert torch.cuda.memory_reserved() == reserved0


FAIL_THEN_PASS = r"""
import json, sys, threading
sys.path.insert(0, sys.argv[1])
import torch
import cluster_reductions_gb300 as rr
rr.load()
out = {}

def failing():
    torch.cuda.set_device(0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        try:
            rr.cluster_allreduce_selftest_noalloc(8, width=8, op="sum", iters=2048, seed=1)
            out["first"] = 0
        except rr.RRError as e:
            out["first"] = e.status

def passing():
    torch.cuda.set_device(0)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out["second"] = [rr.cluster_allreduce_selftest_noalloc(4, width=8, op="sum", iters=4096,
                                                               seed=2 + i) for i in range(5)]

for fn in (failing, passing):
    t = threading.Thread(target=fn)
    t.start()
    t.join()
out["status"] = rr.device_status()
print(json.dumps(out))
"""


def test_noalloc_failed_call_then_good_call(lib):
    """A call refused after it has queued work on the shared array (a cluster
    of 8 above a cap of 4: the fill is queued, the all-reduce launch is
    refused) waits for its stream before it returns, so the next call, from
    another thread on another stream, still checks out."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RR_MAX_CLUSTER="4")
    r = subprocess.run([sys.executable, "-c", FAIL_THEN_PASS, root], env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["first"] == 2                 # RR_ERR_UNSUPPORTED
    assert out["second"] == [0] * 5
    assert out["status"] == 0
