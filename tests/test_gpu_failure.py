"""Failure detection on the device, tested without faulting or hanging the GPU.

The strip kernels wait on mbarriers for their tile copies with a bounded
number of polls; a wait that gives up sets the filter's sticky timeout status,
the kernel returns, and the host learns of it from sbf_get_status.  The test
hook sbf_test_wait_timeout makes one thread wait, with a small bound, on an
mbarrier that nothing completes (no copy attached), so the give-up path runs
for real while nothing is in flight.
"""
import numpy as np
import pytest

from minimizer_sharded_bloom_gb300 import synth
from _gpu_helpers import MAIN, assert_images_equal, assert_words_equal, gpu_insert, gpu_query, need_gpu, \
    oracle_answers, oracle_image

pytestmark = pytest.mark.gpu


def test_bounded_wait_timeout_is_reported_and_cleared():
    torch = need_gpu()
    from minimizer_sharded_bloom_gb300 import SuperBloomFilter, _native as N
    L = N.load()
    sbf = SuperBloomFilter(1 << 20, seed=3, **MAIN)
    assert sbf.specialized
    for polls in (1, 64, 4096):
        assert L.sbf_test_wait_timeout(sbf.handle, polls, None) == N.SBF_OK, N.last_error()
        rc = N.sbf_get_status(sbf.handle, 0)
        assert rc == N.SBF_ERR_CUDA, rc
        assert "timed out" in N.last_error()
        # reported once, then cleared
        assert N.sbf_get_status(sbf.handle, 0) == N.SBF_OK
    # the context and the filter are fine: an insert and a query match the oracle
    rng = np.random.default_rng(31)
    wl = synth.random_records(rng, 6, 100, 20_000, n_prob=0.001)
    gpu_insert(torch, sbf, wl.seq, wl.offsets)
    assert sbf.status() == 0
    F = oracle_image(wl.seq, wl.offsets, MAIN, 1 << 20, 3)
    assert_images_equal(sbf.to_numpy(), F)
    got = gpu_query(torch, sbf, wl.seq, wl.offsets)
    assert_words_equal(got, oracle_answers(F, wl.seq, wl.offsets, MAIN, 3), wl.offsets)
    sbf.close()


def test_wait_timeout_hook_rejects_filters_without_bounded_waits():
    need_gpu()
    from minimizer_sharded_bloom_gb300 import _native as N
    L = N.load()
    f = N.sbf_create(1 << 16, 7, 3, 5, 3, 1)  # runtime-parameter kernels: no mbarrier waits
    try:
        assert L.sbf_test_wait_timeout(f, 10, None) == N.SBF_ERR_INVALID_ARG
        assert L.sbf_test_wait_timeout(f, 0, None) == N.SBF_ERR_INVALID_ARG
        assert N.sbf_get_status(f, 0) == N.SBF_OK
    finally:
        N.sbf_destroy(f)
