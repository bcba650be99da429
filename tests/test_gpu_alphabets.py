"""Parity of the protein and DNA-triplet kernels (through the C ABI) with the
CPU oracle ("cuSBF", Sec. IV-A alphabets): bit-exact filter images and answer
words on seeded inputs spanning many tiles with ragged tails, on the edge cases
of the contract, and through the host-facing entry points with chunk edges
that cut records inside a codon."""
import numpy as np
import pytest

from minimizer_sharded_bloom_gb300 import synth
from _gpu_helpers import (assert_images_equal, assert_words_equal, gpu_insert, gpu_query, need_gpu,
                          oracle_answers, oracle_image, answer_bits)

pytestmark = pytest.mark.gpu

# the compile-time specialised points (the benchmark's parameters)
PROTEIN = dict(k=12, m=8, s=10, H=4)
TRIPLET = dict(k=10, m=5, s=8, H=4)


def _specialized(alphabet, params):
    return params == (PROTEIN if alphabet == "protein" else TRIPLET)


@pytest.fixture(scope="module")
def torch():
    return need_gpu()


def _filter(num_bits, params, seed, alphabet):
    from minimizer_sharded_bloom_gb300 import SuperBloomFilter
    f = SuperBloomFilter(num_bits, seed=seed, alphabet=alphabet, **params)
    assert f.specialized == _specialized(alphabet, params)
    return f


def _records(rng, alphabet, n, lo, hi, dirty):
    if alphabet == "protein":
        return synth.random_protein_records(rng, n, lo, hi, lower_prob=0.05 * dirty,
                                            junk_prob=0.002 * dirty)
    return synth.random_records(rng, n, lo, hi, n_prob=0.002 * dirty, lower_prob=0.05 * dirty,
                                junk_prob=0.0005 * dirty)


def _roundtrip(torch, alphabet, ins, qry, params, num_bits, seed, pad_front=0):
    sbf = _filter(num_bits, params, seed, alphabet)
    gpu_insert(torch, sbf, ins.seq, ins.offsets, pad_front)
    F = oracle_image(ins.seq, ins.offsets, params, num_bits, seed, alphabet=alphabet)
    assert_images_equal(sbf.to_numpy(), F)
    got = gpu_query(torch, sbf, qry.seq, qry.offsets, pad_front, sentinel=-1)
    want = oracle_answers(F, qry.seq, qry.offsets, params, seed, alphabet=alphabet)
    assert_words_equal(got, want, qry.offsets)
    sbf.close()
    return F, got


def _with_own(ins, other):
    """Query batch: the inserted records, then others."""
    return synth.Workload(np.concatenate([ins.seq, other.seq]),
                          np.concatenate([ins.offsets, ins.offsets[-1] + other.offsets[1:]]))


@pytest.mark.parametrize("case", range(12))
@pytest.mark.parametrize("alphabet", ["protein", "dna_triplet"])
def test_mixed_records_random_params(torch, alphabet, case):
    """Random (k, m, s, H) within the 64-bit packing limit (H up to 32: the
    salted multiply for H > 10), random shard counts, mixed records (invalid
    symbols, lowercase, empty and short records, lengths not divisible by 3),
    tens of tiles with a ragged tail, an unaligned sequence pointer for odd
    cases."""
    rng = np.random.default_rng(7000 + case + (0 if alphabet == "protein" else 100))
    kmax = 12 if alphabet == "protein" else 10
    k = int(rng.integers(1, kmax + 1))
    params = dict(k=k, m=int(rng.integers(1, k + 1)), s=int(rng.integers(1, k + 1)),
                  H=int(rng.integers(1, 11)) if case % 4 else int(rng.integers(11, 33)))
    num_bits = int(2 ** rng.integers(8, 22))
    ins = _records(rng, alphabet, int(rng.integers(1, 80)), 0, int(rng.integers(20, 6000)), case % 3)
    qry = _with_own(ins, _records(rng, alphabet, int(rng.integers(1, 80)), 0, 3000, 1))
    _roundtrip(torch, alphabet, ins, qry, params, num_bits, seed=int(rng.integers(0, 2**62)),
               pad_front=case % 2 * 5)


@pytest.mark.parametrize("alphabet,params", [
    ("protein", PROTEIN), ("dna_triplet", TRIPLET),
    ("protein", dict(k=12, m=6, s=10, H=4)), ("dna_triplet", dict(k=10, m=6, s=8, H=4))])
def test_benchmark_params_long_records(torch, alphabet, params):
    """The benchmark's parameters (compile-time kernels) and neighbours of
    them (runtime kernels) on long records (many tiles per record, frame kept
    across tiles) and offsets[0] > 0, not a multiple of 32."""
    rng = np.random.default_rng(71)
    body = _records(rng, alphabet, 7, 20_000, 60_000, 1)
    lead = 77
    ins = synth.Workload(np.concatenate([np.full(lead, ord("A"), np.uint8), body.seq]),
                         np.concatenate([[lead], lead + body.offsets[1:]]))
    qry = _with_own(ins, _records(rng, alphabet, 300, 1, 400, 1))
    F, got = _roundtrip(torch, alphabet, ins, qry, params, 1 << 22, seed=5)
    # every inserted valid k-mer answers present
    own = np.arange(lead, int(ins.offsets[-1]))
    want = oracle_answers(F, ins.seq, ins.offsets, params, 5, alphabet=alphabet)
    assert np.array_equal(answer_bits(got, own), answer_bits(want, own))


@pytest.mark.parametrize("case", range(6))
def test_protein_strip_kernel_mixed(torch, case):
    """The protein point runs the strip kernel (5-bit codes rolled per
    position, cooperative run flushes): dirty ragged records (invalid bytes,
    lowercase, empty and 1-byte records) over tens of tiles, on aligned
    (bulk-copied tiles) and unaligned (direct loads) sequence pointers, and
    shard counts from 1 to 2^20."""
    rng = np.random.default_rng(7500 + case)
    ins = _records(rng, "protein", int(rng.integers(20, 400)), 0, int(rng.integers(50, 4000)), 1 + case % 2)
    qry = _with_own(ins, _records(rng, "protein", 300, 0, 300, 1))
    num_bits = [256, 1 << 12, 1 << 16, 1 << 20, 1 << 24, 1 << 28][case]
    _roundtrip(torch, "protein", ins, qry, PROTEIN, num_bits, seed=int(rng.integers(0, 2**62)),
               pad_front=3 * (case % 2))


def _triplet_batch(rng, case):
    """Record layouts that reach every branch of the triplet kernel's frame-pass
    skip: boundaries of all three residues mod 3 in one tile (ragged lengths),
    one residue only (lengths a multiple of 3, after a lead that is not), a
    residue that turns every record (lengths = 1 mod 3), tiles with no boundary
    at all (records longer than a 23 kB tile), and empty and 1-2 byte records."""
    if case == 0:
        return _records(rng, "dna_triplet", 2500, 0, 400, 1)
    if case == 1:
        body = _records(rng, "dna_triplet", 3000, 150, 150, 0)
        lead = 77
        return synth.Workload(np.concatenate([np.full(lead, ord("C"), np.uint8), body.seq]),
                              np.concatenate([[lead], lead + body.offsets[1:]]))
    if case == 2:
        return _records(rng, "dna_triplet", 2000, 151, 151, 1)
    if case == 3:
        return _records(rng, "dna_triplet", 12, 25_000, 70_000, 1)
    if case == 4:
        long = _records(rng, "dna_triplet", 6, 30_000, 50_000, 0)
        short = _records(rng, "dna_triplet", 1500, 0, 2, 0)
        return synth.Workload(np.concatenate([long.seq, short.seq, long.seq]),
                              np.concatenate([long.offsets, long.offsets[-1] + short.offsets[1:],
                                              long.offsets[-1] + short.offsets[-1] + long.offsets[1:]]))
    return _records(rng, "dna_triplet", 600, 0, 2000, 2)


@pytest.mark.parametrize("case", range(6))
def test_triplet_strip_kernel_mixed(torch, case):
    """The triplet point runs the strip kernel (three frame passes per tile, a
    pass with no codon in frame skipped by the whole block): tens of tiles of
    the layouts of _triplet_batch, inserted and queried, on aligned (bulk-copied
    tiles) and unaligned (direct loads) sequence pointers."""
    rng = np.random.default_rng(7700 + case)
    ins = _triplet_batch(rng, case)
    qry = _with_own(ins, _triplet_batch(np.random.default_rng(7800 + case), (case + 1) % 6))
    _roundtrip(torch, "dna_triplet", ins, qry, TRIPLET, [1 << 12, 1 << 16, 1 << 20, 1 << 22, 1 << 24, 1 << 18][case],
               seed=int(rng.integers(0, 2**62)), pad_front=3 * (case % 2))


@pytest.mark.parametrize("alphabet", ["protein", "dna_triplet"])
def test_edge_cases(torch, alphabet):
    """n = 0 (no work, output untouched); only empty records; records shorter
    than a k-mer; exactly one k-mer (3k bytes for triplets, +1 and +2 bytes);
    k = m = s = 1; the maximum k; thousands of 1-4 byte records (many record
    boundaries per tile)."""
    from minimizer_sharded_bloom_gb300 import _native as N
    kmax = 12 if alphabet == "protein" else 10
    B = 1 if alphabet == "protein" else 3
    sym = b"MKVLAQWERTYIPASDFGHCNY" if alphabet == "protein" else b"ACGTTGCAAGCTTCGA"
    # n = 0
    sbf = _filter(1 << 12, PROTEIN if alphabet == "protein" else TRIPLET, 1, alphabet)
    seq = torch.zeros(16, dtype=torch.uint8, device="cuda")
    off = torch.zeros(1, dtype=torch.int64, device="cuda")
    out = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    sbf.query(seq, off, out=out)
    torch.cuda.synchronize()
    assert (out.cpu().numpy() == -1).all()
    sbf.close()
    rng = np.random.default_rng(72)
    cases = []
    cases.append(synth.Workload(np.zeros(0, np.uint8), synth.csr([0, 0, 0])))
    text = (sym * 40)[: B * kmax + 2]
    for extra in (-1, 0, 1, 2):
        L = B * kmax + extra
        cases.append(synth.Workload(np.frombuffer(text[:L], np.uint8).copy(), synth.csr([L])))
    tiny = _records(rng, alphabet, 5000, 1, 4, 0)
    cases.append(tiny)
    for p in (dict(k=1, m=1, s=1, H=1), dict(k=kmax, m=kmax, s=kmax, H=32),
              dict(k=kmax, m=1, s=1, H=7), dict(k=kmax, m=2, s=kmax - 1, H=5),
              PROTEIN if alphabet == "protein" else TRIPLET):
        for wl in cases:
            _roundtrip(torch, alphabet, wl, wl, p, 1 << 10, seed=9)
    assert N.sbf_get_alphabet(_filter(1 << 10, dict(k=3, m=2, s=2, H=2), 1, alphabet).handle) == \
        N.alphabet_id(alphabet)


@pytest.mark.parametrize("alphabet", ["protein", "dna_triplet"])
def test_create_rejects_k_beyond_packing(torch, alphabet):
    from minimizer_sharded_bloom_gb300 import SuperBloomFilter, _native as N
    kmax = 12 if alphabet == "protein" else 10
    with pytest.raises(N.SBFError):
        SuperBloomFilter(1 << 10, k=kmax + 1, m=2, s=2, H=2, alphabet=alphabet)
    with pytest.raises(ValueError):
        SuperBloomFilter(1 << 10, k=5, m=2, s=2, H=2, alphabet="rna")


@pytest.mark.parametrize("mode", [0, 1, 2])
@pytest.mark.parametrize("pinned", [False, True])
@pytest.mark.parametrize("alphabet,params", [("protein", PROTEIN), ("dna_triplet", TRIPLET)])
def test_host_entry_points(torch, alphabet, params, pinned, mode):
    """sbf_insert_host / sbf_query_host in place (mode 2, and mode 0 for
    pageable buffers) and staged in chunks of 4096 positions (mode 1, and
    mode 0 for pinned buffers): chunk edges cut records at every phase of
    their codon frame, which each chunk must keep."""
    from minimizer_sharded_bloom_gb300 import _native as N
    rng = np.random.default_rng(73)
    ins = _records(rng, alphabet, 30, 0, 5000, 1)
    qry = _with_own(ins, _records(rng, alphabet, 50, 0, 900, 1))
    sbf = _filter(1 << 16, params, 21, alphabet)
    N.sbf_set_host_chunk(sbf.handle, 4096)
    N.sbf_set_host_mode(sbf.handle, mode)
    keep = []

    def host(a):
        if not pinned:
            return np.ascontiguousarray(a)
        t = torch.from_numpy(np.ascontiguousarray(a)).pin_memory()
        keep.append(t)
        return t.numpy()
    sbf.insert_host(host(ins.seq), host(ins.offsets))
    F = oracle_image(ins.seq, ins.offsets, params, 1 << 16, 21, alphabet=alphabet)
    assert_images_equal(sbf.to_numpy(), F)
    out = host(np.zeros((int(qry.offsets[-1]) + 31) // 32 + 1, dtype=np.uint32))
    sbf.query_host(host(qry.seq), host(qry.offsets), out=out)
    assert_words_equal(out, oracle_answers(F, qry.seq, qry.offsets, params, 21, alphabet=alphabet),
                       qry.offsets)


def test_protein_fasta_and_fastq_files(torch, tmp_path):
    """Protein records through the file entry points: sbf_insert_fastx of a
    FASTA file and sbf_query_fastx of a FASTQ file equal the oracle on the
    same records (the reader keeps every byte of a sequence line)."""
    import ctypes
    from minimizer_sharded_bloom_gb300 import _native as N
    rng = np.random.default_rng(74)
    ins = _records(rng, "protein", 60, 0, 900, 1)
    recs = [ins.seq[ins.offsets[r]:ins.offsets[r + 1]].tobytes() for r in range(ins.n_records)]
    fa = tmp_path / "prot.fa"
    fa.write_bytes(b"".join(b">p%d\n%s\n" % (i, r) for i, r in enumerate(recs)))
    sbf = _filter(1 << 16, PROTEIN, 31, "protein")
    n_rec, n_res = N.sbf_insert_fastx(sbf.handle, str(fa), batch_bases=7_000)
    assert (n_rec, n_res) == (len(recs), int(ins.offsets[-1]))
    F = oracle_image(ins.seq, ins.offsets, PROTEIN, 1 << 16, 31, alphabet="protein")
    assert_images_equal(sbf.to_numpy(), F)
    q = _records(rng, "protein", 200, 0, 120, 1)
    qrecs = [q.seq[q.offsets[r]:q.offsets[r + 1]].tobytes() for r in range(q.n_records)]
    fq = tmp_path / "frags.fq"
    fq.write_bytes(b"".join(b"@f%d\n%s\n+\n%s\n" % (i, r, b"I" * len(r)) for i, r in enumerate(qrecs)))
    got = []

    def sink(s, o, n, b):
        offs = np.ctypeslib.as_array((ctypes.c_int64 * (n + 1)).from_address(o)).copy()
        words = np.ctypeslib.as_array((ctypes.c_uint32 * ((int(offs[-1]) + 31) // 32 + 1)).from_address(b)).copy()
        got.append((offs, words))
        return 0

    N.sbf_query_fastx(sbf.handle, str(fq), sink, batch_bases=3_000)
    pos = 0
    for offs, words in got:
        n = offs.size - 1
        batch = qrecs[pos:pos + n]
        pos += n
        bseq = np.frombuffer(b"".join(batch), dtype=np.uint8) if batch else np.zeros(0, np.uint8)
        assert_words_equal(words, oracle_answers(F, bseq, offs, PROTEIN, 31, alphabet="protein"), offs)
    assert pos == len(qrecs)


def test_triplet_noalloc_query(torch):
    """sbf_query_host_noalloc on a triplet filter equals the oracle (the
    no-alloc path stages the batch and runs the filter's own query kernel)."""
    from minimizer_sharded_bloom_gb300 import _native as N
    L = N.load()
    rng = np.random.default_rng(75)
    ins = _records(rng, "dna_triplet", 40, 0, 3000, 1)
    qry = _with_own(ins, _records(rng, "dna_triplet", 60, 0, 500, 1))
    sbf = _filter(1 << 16, TRIPLET, 41, "dna_triplet")
    sbf.insert_host(ins.seq, ins.offsets)
    F = oracle_image(ins.seq, ins.offsets, TRIPLET, 1 << 16, 41, alphabet="dna_triplet")
    assert_images_equal(sbf.to_numpy(), F)
    got = np.full((int(qry.offsets[-1]) + 31) // 32 + 1, 0xDEADBEEF, dtype=np.uint32)
    rc = L.sbf_query_host_noalloc(sbf.handle, qry.seq.ctypes.data, qry.offsets.ctypes.data, qry.n_records,
                                  got.ctypes.data, None)
    assert rc == N.SBF_OK, N.last_error()
    assert_words_equal(got, oracle_answers(F, qry.seq, qry.offsets, TRIPLET, 41, alphabet="dna_triplet"),
                       qry.offsets)
