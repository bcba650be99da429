"""sbf_query_host_noalloc: the host-facing query for callers that cannot
allocate device memory at call time (an allocator that owns the whole device,
or loops that cannot accept cudaMalloc's implicit synchronisation).  It stages
through a fixed device array instead of allocating; its answers must equal the
allocating sbf_query_host's, bit for bit, call after call.

Collected last on purpose (file name), so that a run stopping at the first
failure has already run every other test; it also passes alone in a fresh
process."""
import ctypes

import numpy as np
import pytest

from minimizer_sharded_bloom_gb300 import synth
from _gpu_helpers import MAIN, need_gpu

pytestmark = pytest.mark.gpu


def _words(offsets):
    return (int(offsets[-1]) + 31) // 32 + 1


def test_noalloc_query_matches_host_query_twice_in_a_row():
    need_gpu()
    from minimizer_sharded_bloom_gb300 import _native as N
    L = N.load()
    rng = np.random.default_rng(4242)
    ins = synth.random_records(rng, 40, 200, 6000, n_prob=0.002, lower_prob=0.05)
    f = N.sbf_create(1 << 18, MAIN["k"], MAIN["m"], MAIN["s"], MAIN["H"], 99)
    try:
        N.sbf_insert_host(f, ins.seq.ctypes.data, ins.offsets.ctypes.data, ins.n_records)
        # two different batches back to back: the second one is shorter and
        # starts at a non-zero, non-aligned offset, so stale staging contents
        # from the first call would show
        q1 = synth.Workload(np.concatenate([ins.seq, synth.uniform_bases(rng, 30_000)]),
                            np.concatenate([ins.offsets, [ins.offsets[-1] + 30_000]]))
        pad = 77
        tail = synth.random_records(rng, 25, 0, 400, n_prob=0.01)
        q2 = synth.Workload(np.concatenate([np.full(pad, ord("N"), np.uint8), ins.seq[:9000], tail.seq]),
                            np.concatenate([[pad], pad + np.array([3000, 9000]),
                                            pad + 9000 + tail.offsets[1:]]))
        for q in (q1, q2):
            got = np.full(_words(q.offsets), 0xDEADBEEF, dtype=np.uint32)
            want = np.full(_words(q.offsets), 0xDEADBEEF, dtype=np.uint32)
            rc = L.sbf_query_host_noalloc(f, q.seq.ctypes.data, q.offsets.ctypes.data, q.n_records,
                                          got.ctypes.data, None)
            assert rc == N.SBF_OK, N.last_error()
            N.sbf_query_host(f, q.seq.ctypes.data, q.offsets.ctypes.data, q.n_records, want.ctypes.data)
            lo, hi = int(q.offsets[0]) >> 5, (int(q.offsets[-1]) + 31) >> 5
            assert np.array_equal(got[lo:hi], want[lo:hi])
            assert got[lo:hi].any()
        assert N.sbf_get_status(f, 0) == N.SBF_OK
    finally:
        N.sbf_destroy(f)


def test_noalloc_query_rejects_batches_beyond_its_limit():
    need_gpu()
    from minimizer_sharded_bloom_gb300 import _native as N
    L = N.load()
    f = N.sbf_create(1 << 16, 31, 16, 28, 4, 1)
    try:
        big = (1 << 24) + 1
        seq = np.full(big, ord("A"), dtype=np.uint8)
        off = np.array([0, big], dtype=np.int64)
        out = np.zeros(_words(off), dtype=np.uint32)
        rc = L.sbf_query_host_noalloc(f, seq.ctypes.data, off.ctypes.data, 1, out.ctypes.data, None)
        assert rc == N.SBF_ERR_INVALID_ARG
        assert "maximum" in N.last_error()
        many = np.arange((1 << 20) + 2, dtype=np.int64)
        rc = L.sbf_query_host_noalloc(f, seq.ctypes.data, many.ctypes.data, many.size - 1,
                                      out.ctypes.data, None)
        assert rc == N.SBF_ERR_INVALID_ARG
        assert not out.any()
    finally:
        N.sbf_destroy(f)


def test_noalloc_query_reports_a_pending_bad_offsets_status():
    """A device-facing query with decreasing offsets sets the filter's sticky
    status and nobody reads it.  The next no-alloc call must not hand back the
    staging array's stale words as answers: the query kernel skips its work
    while the status is set, so the call reports SBF_ERR_BAD_OFFSETS (and
    clears the status); the call after it answers normally."""
    torch = need_gpu()
    from minimizer_sharded_bloom_gb300 import _native as N
    L = N.load()
    rng = np.random.default_rng(777)
    ins = synth.random_records(rng, 20, 100, 3000, n_prob=0.002)
    f = N.sbf_create(1 << 18, MAIN["k"], MAIN["m"], MAIN["s"], MAIN["H"], 5)
    try:
        N.sbf_insert_host(f, ins.seq.ctypes.data, ins.offsets.ctypes.data, ins.n_records)
        # a good no-alloc call first, so the staging array holds real answers
        first = np.zeros(_words(ins.offsets), dtype=np.uint32)
        assert L.sbf_query_host_noalloc(f, ins.seq.ctypes.data, ins.offsets.ctypes.data, ins.n_records,
                                        first.ctypes.data, None) == N.SBF_OK, N.last_error()
        assert first.any()
        # device-facing query with decreasing offsets; its status is left unread
        dseq = torch.from_numpy(ins.seq.copy()).cuda()
        bad = torch.tensor([0, 500, 200, 900], dtype=torch.int64, device="cuda")
        dout = torch.zeros(64, dtype=torch.int32, device="cuda")
        N.sbf_query(f, dseq.data_ptr(), bad.data_ptr(), 3, dout.data_ptr())
        torch.cuda.synchronize()
        # the same batch again through the no-alloc call: the error, not answers
        stale = np.zeros(_words(ins.offsets), dtype=np.uint32)
        rc = L.sbf_query_host_noalloc(f, ins.seq.ctypes.data, ins.offsets.ctypes.data, ins.n_records,
                                      stale.ctypes.data, None)
        assert rc == N.SBF_ERR_BAD_OFFSETS, (rc, N.last_error())
        # the status was cleared: the next call matches the allocating query
        got = np.zeros(_words(ins.offsets), dtype=np.uint32)
        want = np.zeros(_words(ins.offsets), dtype=np.uint32)
        assert L.sbf_query_host_noalloc(f, ins.seq.ctypes.data, ins.offsets.ctypes.data, ins.n_records,
                                        got.ctypes.data, None) == N.SBF_OK, N.last_error()
        N.sbf_query_host(f, ins.seq.ctypes.data, ins.offsets.ctypes.data, ins.n_records, want.ctypes.data)
        lo, hi = int(ins.offsets[0]) >> 5, (int(ins.offsets[-1]) + 31) >> 5
        assert np.array_equal(got[lo:hi], want[lo:hi])
        assert np.array_equal(got[lo:hi], first[lo:hi])
    finally:
        N.sbf_destroy(f)
