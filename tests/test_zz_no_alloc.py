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
