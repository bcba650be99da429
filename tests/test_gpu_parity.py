"""Parity of the CUDA path (through the C ABI) with the CPU oracle: bit-exact
filter images and answer bits, on seeded inputs that span several tiles with a
ragged tail, over the specialised and the runtime-parameter kernels, and on the
edge cases of the contract."""
import numpy as np
import pytest

import oracle
from minimizer_sharded_bloom_gb300 import synth
from _gpu_helpers import (MAIN, assert_images_equal, assert_words_equal, gpu_insert, gpu_query,
                          need_gpu, oracle_answers, oracle_image, to_dev, answer_bits)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _filter(num_bits, params, seed):
    from minimizer_sharded_bloom_gb300 import SuperBloomFilter
    return SuperBloomFilter(num_bits, seed=seed, **params)


def _roundtrip(torch, ins, qry, params, num_bits, seed, pad_front=0, expect_specialized=None):
    sbf = _filter(num_bits, params, seed)
    if expect_specialized is not None:
        assert sbf.specialized == expect_specialized
    gpu_insert(torch, sbf, ins.seq, ins.offsets, pad_front)
    F = oracle_image(ins.seq, ins.offsets, params, num_bits, seed)
    assert_images_equal(sbf.to_numpy(), F)
    got = gpu_query(torch, sbf, qry.seq, qry.offsets, pad_front)
    want = oracle_answers(F, qry.seq, qry.offsets, params, seed)
    assert_words_equal(got, want, qry.offsets)
    sbf.close()
    return F, got


def test_tiny_config(torch):
    """tiny: 100 kbp into 2^20 bits; the inserted record answers all-positive,
    the independent one measures the false-positive rate."""
    ins, qry = synth.tiny()
    F, got = _roundtrip(torch, ins, qry, MAIN, 1 << 20, seed=1, expect_specialized=True)
    first = np.arange(0, 100_000 - 31 + 1)
    assert answer_bits(got, first).all()
    second = np.arange(100_000, 200_000 - 31 + 1)
    fpr = answer_bits(got, second).mean()
    assert fpr < 0.05


@pytest.mark.parametrize("case", range(10))
def test_main_config_mixed_records(torch, case):
    """k=31,m=16,s=28,H=4 (specialised kernel) on mixed records: N runs,
    lowercase, junk bytes, empty and short records, several tiles, ragged
    tail, and an unaligned sequence pointer for odd cases."""
    rng = np.random.default_rng(500 + case)
    ins = synth.random_records(rng, int(rng.integers(1, 60)), 0, int(rng.integers(40, 20000)),
                               n_prob=0.002 * (case % 3), lower_prob=0.05 * (case % 2),
                               junk_prob=0.0005 * (case % 4 == 3))
    qry = synth.random_records(rng, int(rng.integers(1, 200)), 0, 400, n_prob=0.001)
    qry = synth.Workload(np.concatenate([ins.seq, qry.seq]),
                         np.concatenate([ins.offsets, ins.offsets[-1] + qry.offsets[1:]]))
    bits = int(1 << int(rng.integers(10, 22)))
    _roundtrip(torch, ins, qry, MAIN, bits, seed=int(rng.integers(0, 2**62)),
               pad_front=(case * 5) % 16, expect_specialized=True)


GRID = [(m, s, H) for m in (12, 14, 16, 18, 21) for s in (20, 24, 28, 31) for H in (1, 2, 4, 6, 8)]


@pytest.mark.parametrize("m,s,H", GRID)
def test_sweep_grid_specialisations(torch, m, s, H):
    """Every (s, m, H) of the k = 31 sweep grid runs its own specialised
    kernel; each must match the oracle bit for bit."""
    rng = np.random.default_rng(1000 + 100 * m + 10 * s + H)
    params = dict(k=31, m=m, s=s, H=H)
    ins = synth.random_records(rng, 3, 10_000, 25_000, n_prob=0.0005)
    q_rand = synth.Workload(synth.uniform_bases(rng, 3000 * 31), synth.csr(np.full(3000, 31)))
    qry = synth.Workload(np.concatenate([ins.seq, q_rand.seq]),
                         np.concatenate([ins.offsets, ins.offsets[-1] + q_rand.offsets[1:]]))
    _roundtrip(torch, ins, qry, params, 1 << 16, seed=77 + H, expect_specialized=True)


@pytest.mark.parametrize("case", range(12))
def test_runtime_parameter_kernel(torch, case):
    """(k, m, s, H) outside the specialised grid run the runtime-parameter
    kernel, which must match the oracle too."""
    rng = np.random.default_rng(2000 + case)
    while True:
        k = int(rng.integers(1, 33))
        m = int(rng.integers(1, k + 1))
        s = int(rng.integers(1, k + 1))
        H = int(rng.integers(1, 11)) if case % 3 else int(rng.integers(11, 33))
        if not (k == 31 and m in (12, 14, 16, 18, 21) and s in (20, 24, 28, 31) and H in (1, 2, 4, 6, 8)):
            break
    params = dict(k=k, m=m, s=s, H=H)
    ins = synth.random_records(rng, int(rng.integers(1, 30)), 0, 3000, n_prob=0.01, lower_prob=0.1)
    qry = synth.random_records(rng, int(rng.integers(1, 30)), 0, 300, n_prob=0.01)
    qry = synth.Workload(np.concatenate([ins.seq, qry.seq]),
                         np.concatenate([ins.offsets, ins.offsets[-1] + qry.offsets[1:]]))
    _roundtrip(torch, ins, qry, params, 1 << int(rng.integers(8, 16)), seed=case * 977,
               pad_front=case % 7, expect_specialized=False)


@pytest.mark.parametrize("H", [12, 16])
def test_large_h_specialisations(torch, H):
    """H = 12, 16 at (31, 16, 28) run specialised kernels with the salted
    multiply (Sec. IV-G) and match the oracle."""
    rng = np.random.default_rng(3000 + H)
    params = dict(k=31, m=16, s=28, H=H)
    ins = synth.random_records(rng, 4, 5_000, 30_000, n_prob=0.0005)
    q = synth.Workload(synth.uniform_bases(rng, 2000 * 31), synth.csr(np.full(2000, 31)))
    qry = synth.Workload(np.concatenate([ins.seq, q.seq]),
                         np.concatenate([ins.offsets, ins.offsets[-1] + q.offsets[1:]]))
    _roundtrip(torch, ins, qry, params, 1 << 15, seed=H, expect_specialized=True)


def test_edge_cases(torch):
    """Records of length 0, k-1, k, k+1 and 31 + 32 j; an all-N record; a
    first record that does not start at 0; a single base."""
    k = 31
    texts = ["", "A" * (k - 1), "ACGT" * 7 + "ACG", "C" * (k + 1), "N" * 100, "G"]
    rng = np.random.default_rng(3)
    texts += ["".join(rng.choice(list("ACGT"), size=31 + 32 * j)) for j in range(1, 5)]
    seq = np.frombuffer("".join(texts).encode(), dtype=np.uint8).copy()
    off = synth.csr([len(t) for t in texts])
    ins = synth.Workload(seq, off)
    _roundtrip(torch, ins, ins, MAIN, 1 << 12, seed=5)
    # the same records shifted so that offsets[0] = 37 (bytes before it unused)
    seq2 = np.concatenate([np.full(37, ord("T"), dtype=np.uint8), seq])
    ins2 = synth.Workload(seq2, off + 37)
    _roundtrip(torch, ins2, ins2, MAIN, 1 << 12, seed=5)


def test_empty_batch_is_a_noop(torch):
    sbf = _filter(1 << 12, MAIN, 1)
    seq, off = to_dev(torch, np.zeros(0, np.uint8), np.zeros(1, np.int64))
    sbf.insert(seq, off)
    out = torch.full((4,), 7, dtype=torch.int32, device="cuda")
    sbf.query(seq, off, out=out)
    torch.cuda.synchronize()
    assert (out.cpu().numpy() == 7).all()
    assert not sbf.to_numpy().any()
    assert sbf.status() == 0


def test_query_writes_exactly_the_contract_words(torch):
    """Words in [offsets[0] >> 5, (offsets[n] + 31) >> 5) are written, the
    rest are left alone."""
    rng = np.random.default_rng(9)
    body = synth.uniform_bases(rng, 5000)
    seq = np.concatenate([np.full(100, ord("A"), np.uint8), body])
    off = np.array([100, 2100, 5100], dtype=np.int64)
    sbf = _filter(1 << 14, MAIN, 4)
    gpu_insert(torch, sbf, seq, off)
    got = gpu_query(torch, sbf, seq, off, sentinel=-1)
    lo, hi = 100 >> 5, (5100 + 31) >> 5
    assert (got[:lo] == 0xFFFFFFFF).all() and (got[hi:] == 0xFFFFFFFF).all()
    F = oracle_image(seq, off, MAIN, 1 << 14, 4)
    assert_words_equal(got, oracle_answers(F, seq, off, MAIN, 4), off)


def test_bad_offsets_set_the_status(torch):
    """Decreasing offsets: the device check sets the sticky status, the
    kernels skip the work, sbf_get_status reports and clears it."""
    from minimizer_sharded_bloom_gb300 import _native as N
    rng = np.random.default_rng(10)
    seq = synth.uniform_bases(rng, 4000)
    good = np.array([0, 2000, 4000], dtype=np.int64)
    bad = np.array([0, 3000, 2000, 4000], dtype=np.int64)
    sbf = _filter(1 << 14, MAIN, 4)
    dseq, doff = to_dev(torch, seq, bad)
    sbf.insert(dseq, doff)
    assert sbf.status() == N.SBF_ERR_BAD_OFFSETS
    assert not sbf.to_numpy().any()
    assert sbf.status() == 0
    gpu_insert(torch, sbf, seq, good)
    assert sbf.status() == 0
    assert_images_equal(sbf.to_numpy(), oracle_image(seq, good, MAIN, 1 << 14, 4))


@pytest.mark.parametrize("mode", [0, 1, 2])
def test_host_calls_report_bad_offsets(torch, mode):
    """Host-facing insert/query with decreasing offsets fail with
    SBF_ERR_BAD_OFFSETS (found by the device check, on the offsets read in
    place, before any chunk runs), change nothing, leave the status clear,
    and the next good call works."""
    from minimizer_sharded_bloom_gb300 import _native as N
    rng = np.random.default_rng(14)
    seq = synth.uniform_bases(rng, 4000)
    good = np.array([0, 2000, 4000], dtype=np.int64)
    bad = np.array([0, 3000, 2000, 4000], dtype=np.int64)
    sbf = _filter(1 << 14, MAIN, 4)
    N.sbf_set_host_mode(sbf.handle, mode)
    with pytest.raises(N.SBFError) as err:
        sbf.insert_host(seq, bad)
    assert err.value.code == N.SBF_ERR_BAD_OFFSETS
    assert not sbf.to_numpy().any()
    assert sbf.status() == 0
    out = np.full(4000 // 32 + 2, 0xDEADBEEF, dtype=np.uint32)
    with pytest.raises(N.SBFError) as err:
        sbf.query_host(seq, bad, out=out)
    assert err.value.code == N.SBF_ERR_BAD_OFFSETS
    assert sbf.status() == 0
    # page-locked buffers (staged in mode 0): nothing written
    pseq = torch.from_numpy(seq).pin_memory()
    pbad = torch.from_numpy(bad).pin_memory()
    pout = torch.full((4000 // 32 + 2,), -1, dtype=torch.int32).pin_memory()
    with pytest.raises(N.SBFError) as err:
        N.sbf_query_host(sbf.handle, pseq.data_ptr(), pbad.data_ptr(), 3, pout.data_ptr(), 0)
    assert err.value.code == N.SBF_ERR_BAD_OFFSETS
    assert (pout.numpy() == -1).all()
    assert sbf.status() == 0
    sbf.insert_host(seq, good)
    F = oracle_image(seq, good, MAIN, 1 << 14, 4)
    assert_images_equal(sbf.to_numpy(), F)
    assert_words_equal(sbf.query_host(seq, good), oracle_answers(F, seq, good, MAIN, 4), good)


@pytest.mark.parametrize("R,n,params", [
    (31, 300, MAIN), (50, 129, MAIN), (120, 1000, MAIN), (150, 777, MAIN), (160, 128, MAIN),
    (150, 1, MAIN), (30, 200, MAIN), (161, 300, MAIN), (400, 90, MAIN),
    (150, 500, dict(k=25, m=11, s=20, H=3)), (100, 64, dict(k=31, m=16, s=28, H=12))])
def test_dense_query_equals_csr_and_oracle(torch, R, n, params):
    """sbf_query_dense on n fixed-length records of R bytes (N runs, lowercase;
    partial last tile; an unaligned pointer for odd n) equals the oracle on
    the same records as CSR offsets and the CSR query, word for word: the
    dense strip kernel (R <= 160 at the operating point) and the
    runtime-parameter fallback (shorter than k, longer than 160, other
    parameters)."""
    from minimizer_sharded_bloom_gb300 import _native as N
    rng = np.random.default_rng(900 + R + n)
    ins = synth.random_records(rng, 60, 500, 8000, n_prob=0.002)
    reads = synth.random_records(rng, n, R, R, n_prob=0.003, lower_prob=0.05)
    half = reads.seq.reshape(n, R)[: n // 2]
    take = min(ins.seq.size, half.size) // R * R
    src = ins.seq[:take].reshape(-1, R)
    half[: src.shape[0]] = src  # up to half the reads copied from the inserted records
    seq = reads.seq
    off = synth.csr(np.full(n, R))
    sbf = _filter(1 << 18, params, 61)
    gpu_insert(torch, sbf, ins.seq, ins.offsets)
    F = oracle_image(ins.seq, ins.offsets, params, 1 << 18, 61)
    pad = n % 2 * 3
    dseq, _ = to_dev(torch, seq, off, pad)
    words = (n * R + 31) // 32
    out = torch.full((words + 2,), -1, dtype=torch.int32, device="cuda")
    sbf.query_dense(dseq[: n * R], R, out=out)
    torch.cuda.synchronize()
    got = out.cpu().numpy().view(np.uint32)
    assert (got[words:] == 0xFFFFFFFF).all()  # nothing past the answer range
    want = oracle_answers(F, seq, off, params, 61)
    assert_words_equal(got, want, off)
    assert_words_equal(got, gpu_query(torch, sbf, seq, off), off)


def _uniform_case(rng, n, R, offset0=0, tail=None):
    """n reads of R bytes (half copied from inserted records) at CSR offsets
    starting at offset0; `tail` replaces the last read's length."""
    ins = synth.random_records(rng, 60, 500, 8000, n_prob=0.002)
    lens = np.full(n, R)
    if tail is not None:
        lens[-1] = tail
    reads = synth.random_records(rng, n, R, R, n_prob=0.003, lower_prob=0.05)
    body = rng.integers(0, 4, size=offset0 + int(lens.sum()), dtype=np.uint8)
    seq = np.frombuffer(b"ACGT", dtype=np.uint8)[body]
    seq[offset0: offset0 + min(n * R, int(lens.sum()))] = reads.seq[: min(n * R, int(lens.sum()))]
    take = min(ins.seq.size, n * R // 2)
    seq[offset0: offset0 + take] = ins.seq[:take]
    off = offset0 + synth.csr(lens)
    return ins, seq, off


@pytest.mark.parametrize("R,n,offset0,tail", [
    (150, 777, 0, None), (31, 300, 0, None), (160, 129, 0, None), (97, 1, 0, None),
    (150, 500, 64, None), (150, 500, 7, None), (150, 500, 0, 149), (150, 500, 0, 151),
    (30, 400, 0, None), (161, 300, 0, None)])
def test_csr_query_of_uniform_batches(torch, R, n, offset0, tail):
    """The operating point's CSR query runs a batch whose records are all one
    length (k <= R <= 160, starting at offset 0) with the one-read-per-strip
    geometry, and every other batch (a nonzero first offset, one record of
    another length, records shorter than k or longer than 160) with the CSR
    one: the answers equal the oracle's either way, and no word outside the
    answer range is written."""
    rng = np.random.default_rng(3100 + R + n + offset0)
    ins, seq, off = _uniform_case(rng, n, R, offset0, tail)
    sbf = _filter(1 << 18, MAIN, 62)
    gpu_insert(torch, sbf, ins.seq, ins.offsets)
    F = oracle_image(ins.seq, ins.offsets, MAIN, 1 << 18, 62)
    want = oracle_answers(F, seq, off, MAIN, 62)
    got = gpu_query(torch, sbf, seq, off, sentinel=-1)
    assert_words_equal(got, want, off)
    lo, hi = int(off[0]) >> 5, (int(off[-1]) + 31) >> 5
    assert (got[:lo] == 0xFFFFFFFF).all() and (got[hi:] == 0xFFFFFFFF).all()
    # the host-facing calls: in place (pageable or pinned), staged, no-alloc
    from minimizer_sharded_bloom_gb300 import _native as N
    for mode in (0, 1):
        N.sbf_set_host_mode(sbf.handle, mode)
        assert_words_equal(sbf.query_host(seq, off), want, off)
    N.sbf_set_host_mode(sbf.handle, 0)
    pseq = torch.from_numpy(seq).pin_memory()
    poff = torch.from_numpy(off.astype(np.int64)).pin_memory()
    pout = torch.zeros((int(off[-1]) + 31) // 32 + 1, dtype=torch.int32).pin_memory()
    N.sbf_query_host(sbf.handle, pseq.data_ptr(), poff.data_ptr(), n, pout.data_ptr(), 0)
    assert_words_equal(pout.numpy().view(np.uint32), want, off)
    out = np.zeros((int(off[-1]) + 31) // 32 + 1, dtype=np.uint32)
    N.sbf_query_host_noalloc(sbf.handle, seq.ctypes.data, off.ctypes.data, n, out.ctypes.data, 0)
    assert_words_equal(out, want, off)
    sbf.close()


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("pinned", [False, True])
@pytest.mark.parametrize("case", ["reads", "long", "mixed"])
def test_host_query_chunk_edges(torch, case, pinned, mode):
    """Host-facing queries cut into chunks of 4096 positions: a batch of
    150 bp reads (every chunk ends at a read that starts on a 32-position
    boundary and runs dense), records longer than a chunk (chunks cut inside
    records: each leaves the answer words from its cut on to the next), and a
    mix with empty records.  Answers equal the oracle's, and no word outside
    the answer range is written."""
    from minimizer_sharded_bloom_gb300 import _native as N
    rng = np.random.default_rng({"reads": 3300, "long": 3301, "mixed": 3302}[case])
    ins = synth.random_records(rng, 40, 500, 6000, n_prob=0.002)
    if case == "reads":
        q = synth.random_records(rng, 400, 150, 150, n_prob=0.003)
    elif case == "long":
        q = synth.random_records(rng, 6, 5000, 13000, n_prob=0.002)
    else:
        q = synth.random_records(rng, 120, 0, 3000, n_prob=0.002)
    seq = q.seq.copy()
    take = min(ins.seq.size, seq.size // 2)
    seq[:take] = ins.seq[:take]
    off = q.offsets.copy()
    sbf = _filter(1 << 16, MAIN, 64)
    gpu_insert(torch, sbf, ins.seq, ins.offsets)
    F = oracle_image(ins.seq, ins.offsets, MAIN, 1 << 16, 64)
    want = oracle_answers(F, seq, off, MAIN, 64)
    N.sbf_set_host_chunk(sbf.handle, 4096)
    N.sbf_set_host_mode(sbf.handle, mode)
    words = (int(off[-1]) + 31) // 32
    if pinned:
        ks = torch.from_numpy(seq).pin_memory()
        ko = torch.from_numpy(off).pin_memory()
        kt = torch.full((words + 3,), -1, dtype=torch.int32).pin_memory()
        N.sbf_query_host(sbf.handle, ks.data_ptr(), ko.data_ptr(), q.n_records, kt.data_ptr(), 0)
        got = kt.numpy().view(np.uint32)
    else:
        got = np.full(words + 3, 0xFFFFFFFF, dtype=np.uint32)
        N.sbf_query_host(sbf.handle, seq.ctypes.data, off.ctypes.data, q.n_records, got.ctypes.data, 0)
    assert_words_equal(got, want, off)
    assert (got[words:] == 0xFFFFFFFF).all()
    assert sbf.status() == 0
    sbf.close()


def test_concurrent_uniform_and_ragged_queries(torch):
    """Two streams query one filter at once, one with a uniform batch and one
    with a ragged batch, many times over: each call's uniformity flag is its
    own, so both keep answering like the oracle."""
    rng = np.random.default_rng(3200)
    ins, useq, uoff = _uniform_case(rng, 3000, 150)
    rag = synth.random_records(rng, 2000, 60, 240, n_prob=0.003)
    sbf = _filter(1 << 20, MAIN, 63)
    gpu_insert(torch, sbf, ins.seq, ins.offsets)
    F = oracle_image(ins.seq, ins.offsets, MAIN, 1 << 20, 63)
    want_u = oracle_answers(F, useq, uoff, MAIN, 63)
    want_r = oracle_answers(F, rag.seq, rag.offsets, MAIN, 63)
    du, dou = to_dev(torch, useq, uoff)
    dr, dor = to_dev(torch, rag.seq, rag.offsets)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    outs_u, outs_r = [], []
    torch.cuda.synchronize()
    for _ in range(20):
        ou = torch.zeros((int(uoff[-1]) + 31) // 32 + 1, dtype=torch.int32, device="cuda")
        orr = torch.zeros((int(rag.offsets[-1]) + 31) // 32 + 1, dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        sbf.query(du, dou, out=ou, stream=s1)
        sbf.query(dr, dor, out=orr, stream=s2)
        outs_u.append(ou)
        outs_r.append(orr)
    torch.cuda.synchronize()
    for ou, orr in zip(outs_u, outs_r):
        assert_words_equal(ou.cpu().numpy().view(np.uint32), want_u, uoff)
        assert_words_equal(orr.cpu().numpy().view(np.uint32), want_r, rag.offsets)
    assert sbf.status() == 0
    sbf.close()


def test_filter_algebra_on_gpu(torch):
    """Order independence, split inserts, idempotence and union, on the GPU
    image (OR is commutative and idempotent)."""
    rng = np.random.default_rng(11)
    a = synth.random_records(rng, 40, 100, 3000, n_prob=0.001)
    b = synth.random_records(rng, 40, 100, 3000, n_prob=0.001)
    both = synth.Workload(np.concatenate([b.seq, a.seq]),
                          np.concatenate([b.offsets, b.offsets[-1] + a.offsets[1:]]))
    bits = 1 << 16
    fa = gpu_insert(torch, _filter(bits, MAIN, 8), a.seq, a.offsets).to_numpy()
    fb = gpu_insert(torch, _filter(bits, MAIN, 8), b.seq, b.offsets).to_numpy()
    s = _filter(bits, MAIN, 8)
    gpu_insert(torch, s, both.seq, both.offsets)
    fab = s.to_numpy()
    assert np.array_equal(fab, fa | fb)
    gpu_insert(torch, s, a.seq, a.offsets)
    assert np.array_equal(s.to_numpy(), fab)


def test_copy_load_clear(torch):
    rng = np.random.default_rng(12)
    a = synth.random_records(rng, 10, 1000, 5000)
    s1 = gpu_insert(torch, _filter(1 << 15, MAIN, 3), a.seq, a.offsets)
    img = s1.to_numpy()
    s2 = _filter(1 << 15, MAIN, 3)
    s2.load(img)
    assert np.array_equal(s2.to_numpy(), img)
    assert np.array_equal(gpu_query(torch, s1, a.seq, a.offsets), gpu_query(torch, s2, a.seq, a.offsets))
    dev = s1.to_tensor()
    s3 = _filter(1 << 15, MAIN, 3)
    s3.load(dev)
    torch.cuda.synchronize()
    assert np.array_equal(s3.to_numpy(), img)
    s2.clear()
    torch.cuda.synchronize()
    assert not s2.to_numpy().any()


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("pinned", [False, True])
@pytest.mark.parametrize("params", [MAIN, dict(k=25, m=11, s=20, H=3)])
def test_host_entry_points(torch, pinned, params, mode):
    """sbf_insert_host / sbf_query_host, reading the host buffers in place
    (mode 2, and mode 0 for pageable buffers) or staged in chunks of 4096
    positions so that chunks end at records or cut them (mode 1, and mode 0
    for pinned buffers), with pageable and pinned host buffers, equal the
    oracle."""
    from minimizer_sharded_bloom_gb300 import _native as N
    rng = np.random.default_rng(13)
    ins = synth.random_records(rng, 30, 0, 2500, n_prob=0.002)
    qry = synth.random_records(rng, 50, 0, 900, n_prob=0.002)
    qry = synth.Workload(np.concatenate([ins.seq, qry.seq]),
                         np.concatenate([ins.offsets, ins.offsets[-1] + qry.offsets[1:]]))
    sbf = _filter(1 << 14, params, 21)
    N.sbf_set_host_chunk(sbf.handle, 4096)
    N.sbf_set_host_mode(sbf.handle, mode)
    if pinned:
        def pin(a):
            t = torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
            return t, t.numpy()
        _ks, s_ins = pin(ins.seq)
        _ko, o_ins = pin(ins.offsets)
        _kq, s_q = pin(qry.seq)
        _kqo, o_q = pin(qry.offsets)
        out_t = torch.zeros((int(qry.offsets[-1]) + 31) // 32 + 1, dtype=torch.int32).pin_memory()
        out = out_t.numpy().view(np.uint32)
    else:
        s_ins, o_ins, s_q, o_q = ins.seq, ins.offsets, qry.seq, qry.offsets
        out = np.zeros((int(qry.offsets[-1]) + 31) // 32 + 1, dtype=np.uint32)
    sbf.insert_host(s_ins, o_ins)
    F = oracle_image(ins.seq, ins.offsets, params, 1 << 14, 21)
    assert_images_equal(sbf.to_numpy(), F)
    sbf.query_host(s_q, o_q, out=out)
    assert_words_equal(out, oracle_answers(F, qry.seq, qry.offsets, params, 21), qry.offsets)


@pytest.mark.parametrize("params", [dict(k=31, m=16, s=28, H=4), dict(k=31, m=12, s=20, H=8),
                                    dict(k=31, m=21, s=31, H=1), dict(k=31, m=16, s=28, H=16)])
def test_runtime_kernels_flag_matches_strip_kernels(params):
    """SBF_FLAG_RUNTIME_KERNELS runs a specialised point on the runtime-
    parameter kernels: the images and answers equal the strip kernels'."""
    torch = need_gpu()
    from minimizer_sharded_bloom_gb300 import SuperBloomFilter
    rng = np.random.default_rng(sum(params.values()))
    ins = synth.random_records(rng, 10, 200, 40_000, n_prob=0.001, lower_prob=0.01)
    qry = synth.random_records(rng, 400, 20, 300, n_prob=0.002)
    qseq = np.concatenate([ins.seq, qry.seq])
    qoff = np.concatenate([ins.offsets, ins.offsets[-1] + qry.offsets[1:]])
    res = []
    for rt in (False, True):
        sbf = SuperBloomFilter(1 << 22, seed=9, runtime_kernels=rt, **params)
        assert sbf.specialized == (not rt)
        gpu_insert(torch, sbf, ins.seq, ins.offsets)
        res.append((sbf.to_numpy(), gpu_query(torch, sbf, qseq, qoff)))
        assert sbf.status() == 0
        sbf.close()
    assert_images_equal(res[1][0], res[0][0])
    assert_words_equal(res[1][1], res[0][1], qoff)


def test_queued_insert_on_a_filter_far_larger_than_l2():
    """Filters several times larger than L2 insert with the warp run-queue
    flush.  A 2^34-bit (2 GiB) filter takes it; the image must equal the
    oracle's, with inputs that flush many runs per step (records of one or
    two k-mers, N runs) and ragged warps at the batch's end."""
    torch = need_gpu()
    from minimizer_sharded_bloom_gb300 import SuperBloomFilter
    rng = np.random.default_rng(4321)
    long = synth.random_records(rng, 6, 5_000, 60_000, n_prob=0.002, lower_prob=0.01)
    short = synth.random_records(rng, 3_000, 31, 33, n_prob=0.01)
    tail = synth.random_records(rng, 37, 0, 900)
    seq = np.concatenate([long.seq, short.seq, tail.seq])
    off = np.concatenate([long.offsets, long.offsets[-1] + short.offsets[1:],
                          long.offsets[-1] + short.offsets[-1] + tail.offsets[1:]])
    sbf = SuperBloomFilter(1 << 34, seed=21, **MAIN)
    assert sbf.specialized
    gpu_insert(torch, sbf, seq, off)
    assert sbf.status() == 0
    img = sbf.to_tensor()
    torch.cuda.synchronize()
    sh, words = oracle.insert_sparse(seq, off, MAIN["k"], MAIN["m"], MAIN["s"], MAIN["H"], sbf.num_shards, 21)
    nz = int((img != 0).any(dim=1).sum().item())
    assert nz == sh.size
    got = img.index_select(0, torch.from_numpy(sh.astype(np.int64)).cuda()).cpu().numpy().view(np.uint64)
    assert np.array_equal(got, words)
    # and the same batch answers present everywhere it has a valid k-mer
    out = gpu_query(torch, sbf, seq, off)
    want = oracle.query(np.zeros((1, 4), np.uint64) + np.uint64(2**64 - 1), seq, off, MAIN["k"], MAIN["m"],
                        MAIN["s"], MAIN["H"], 21)
    assert_words_equal(out, want, off)
    sbf.close()
