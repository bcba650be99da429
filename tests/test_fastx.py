"""FASTA/FASTQ input (plain and gzip): the library's reader returns exactly the
records a file holds; inserting/querying a file through the library equals the
oracle on the same records."""
import gzip
import os

import numpy as np
import pytest

from minimizer_sharded_bloom_gb300 import synth


def _records(seed, n=40, lo=0, hi=700):
    rng = np.random.default_rng(seed)
    wl = synth.random_records(rng, n, lo, hi, n_prob=0.01, lower_prob=0.05)
    return [wl.seq[wl.offsets[r]:wl.offsets[r + 1]].tobytes() for r in range(wl.n_records)], rng


def _write_fasta(path, recs, width=60, crlf=False, blank=False, gz=False):
    nl = b"\r\n" if crlf else b"\n"
    out = []
    for i, r in enumerate(recs):
        out.append(b">read%d some description" % i + nl)
        for c in range(0, len(r), width):
            out.append(r[c:c + width] + nl)
        if blank:
            out.append(nl)
    data = b"".join(out)
    with (gzip.open(path, "wb") if gz else open(path, "wb")) as f:
        f.write(data)


def _write_fastq(path, recs, rng, gz=False):
    out = []
    for i, r in enumerate(recs):
        qual = bytes(rng.integers(33, 74, size=len(r), dtype=np.uint8))
        # '@' and '+' can start quality lines too
        if len(qual) > 2:
            qual = b"@+" + qual[2:]
        out.append(b"@q%d\n%s\n+\n%s\n" % (i, r, qual))
    data = b"".join(out)
    with (gzip.open(path, "wb") if gz else open(path, "wb")) as f:
        f.write(data)


@pytest.fixture(scope="module")
def N():
    from minimizer_sharded_bloom_gb300 import _native, build_lib
    build_lib.build()
    return _native


def _read_all(N, path, cap=1 << 16, max_records=1 << 12):
    r = N.sbf_fastx_open(str(path))
    seq = np.zeros(cap, dtype=np.uint8)
    off = np.zeros(max_records + 1, dtype=np.int64)
    recs = []
    try:
        while True:
            n, used = N.sbf_fastx_next(r, seq.ctypes.data, cap, off.ctypes.data, max_records)
            if n == 0:
                break
            assert off[n] == used
            recs += [seq[off[i]:off[i + 1]].tobytes() for i in range(n)]
    finally:
        N.sbf_fastx_close(r)
    return recs


@pytest.mark.parametrize("kind", ["fasta", "fasta-crlf-blank", "fasta-wide", "fastq"])
@pytest.mark.parametrize("gz", [False, True])
def test_reader_returns_the_records(tmp_path, N, kind, gz):
    if gz and not N.sbf_fastx_has_gzip():
        pytest.skip("libsbf built without zlib")
    recs, rng = _records(7 + len(kind) + gz)
    path = tmp_path / ("in." + kind + (".gz" if gz else ""))
    if kind == "fastq":
        _write_fastq(path, recs, rng, gz=gz)
    elif kind == "fasta-crlf-blank":
        _write_fasta(path, recs, width=70, crlf=True, blank=True, gz=gz)
    elif kind == "fasta-wide":
        _write_fasta(path, recs, width=100000, gz=gz)
    else:
        _write_fasta(path, recs, gz=gz)
    assert _read_all(N, path) == recs
    # small batches: records never split, every batch within capacity
    assert _read_all(N, path, cap=1500, max_records=3) == recs


def test_oversize_record_reports_the_size_needed(tmp_path, N):
    recs, _ = _records(3, n=3, lo=100, hi=200)
    recs[1] = b"ACGT" * 1000
    path = tmp_path / "big.fa"
    _write_fasta(path, recs)
    r = N.sbf_fastx_open(str(path))
    seq = np.zeros(1024, dtype=np.uint8)
    off = np.zeros(9, dtype=np.int64)
    try:
        n, _ = N.sbf_fastx_next(r, seq.ctypes.data, 1024, off.ctypes.data, 8)
        assert n == 1 and seq[:off[1]].tobytes() == recs[0]
        with pytest.raises(N.SBFError):
            N.sbf_fastx_next(r, seq.ctypes.data, 1024, off.ctypes.data, 8)
        assert N.sbf_fastx_pending_bases(r) == 4000
        big = np.zeros(8192, dtype=np.uint8)
        n, _ = N.sbf_fastx_next(r, big.ctypes.data, 8192, off.ctypes.data, 8)
        assert n == 2 and big[:off[1]].tobytes() == recs[1]
    finally:
        N.sbf_fastx_close(r)


def test_malformed_input_is_rejected(tmp_path, N):
    bad = tmp_path / "bad.fq"
    bad.write_bytes(b"@r1\nACGT\n+\nII\n")
    r = N.sbf_fastx_open(str(bad))
    seq = np.zeros(64, dtype=np.uint8)
    off = np.zeros(5, dtype=np.int64)
    try:
        with pytest.raises(N.SBFError):
            N.sbf_fastx_next(r, seq.ctypes.data, 64, off.ctypes.data, 4)
    finally:
        N.sbf_fastx_close(r)
    with pytest.raises(N.SBFError):
        N.sbf_fastx_open(str(tmp_path / "missing.fa"))


@pytest.mark.gpu
def test_fastx_insert_and_query_match_the_oracle(tmp_path):
    from _gpu_helpers import MAIN, need_gpu, oracle_answers, oracle_image, assert_words_equal
    need_gpu()
    from minimizer_sharded_bloom_gb300 import _native as N
    recs, rng = _records(11, n=120, lo=0, hi=3000)
    fa = tmp_path / "ref.fa.gz" if N.sbf_fastx_has_gzip() else tmp_path / "ref.fa"
    _write_fasta(fa, recs, gz=N.sbf_fastx_has_gzip())
    seq = np.frombuffer(b"".join(recs), dtype=np.uint8)
    off = synth.csr([len(r) for r in recs])
    f = N.sbf_create(1 << 16, 31, 16, 28, 4, 3)
    try:
        n_rec, n_bases = N.sbf_insert_fastx(f, str(fa), batch_bases=20_000)
        assert (n_rec, n_bases) == (len(recs), int(off[-1]))
        img = np.zeros((N.sbf_num_shards(f), 4), dtype=np.uint64)
        N.sbf_copy_bits(f, img.ctypes.data, img.nbytes, 0)
        F = oracle_image(seq, off, MAIN, 1 << 16, 3)
        assert np.array_equal(img, F)
        qrecs, qrng = _records(12, n=300, lo=0, hi=300)
        fq = tmp_path / "reads.fq"
        _write_fastq(fq, qrecs, qrng)
        got = []

        def sink(s, o, n, b):
            offs = np.ctypeslib.as_array((ctypes_i64 * (n + 1)).from_address(o)).copy()
            words = np.ctypeslib.as_array((ctypes_u32 * ((int(offs[-1]) + 31) // 32 + 1)).from_address(b)).copy()
            got.append((offs, words))
            return 0

        import ctypes
        ctypes_i64, ctypes_u32 = ctypes.c_int64, ctypes.c_uint32
        N.sbf_query_fastx(f, str(fq), sink, batch_bases=10_000)
        pos = 0
        for offs, words in got:
            n = offs.size - 1
            batch = qrecs[pos:pos + n]
            pos += n
            bseq = np.frombuffer(b"".join(batch), dtype=np.uint8) if batch else np.zeros(0, np.uint8)
            want = oracle_answers(F, bseq, offs, MAIN, 3)
            assert_words_equal(words, want, offs)
        assert pos == len(qrecs)
    finally:
        N.sbf_destroy(f)
