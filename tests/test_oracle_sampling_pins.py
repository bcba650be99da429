"""Pins of the oracle's sampling entry points: ``kmer_batch`` (per-position
shard and bit masks), ``query_sampled`` (Algorithm 2 on selected positions
against a supplied shard lookup), ``insert_sparse`` (the image of a whole
insert as sorted non-zero shards) and ``count_runs`` (Fig. 3's runs).

The full-size GPU parity checks of large workloads lean on these helpers, so
each one is compared here with something other than itself: the independent
pure-Python brute force (``oracle/brute.py``) on tiny inputs, and the already
pinned whole-batch ``insert`` / ``query`` / ``kmer_info`` on medium inputs.
DNA, protein and DNA-triplet inputs, with empty and short records, N runs,
lowercase and junk bytes, and a first offset that is not zero.

Source: "cuSBF: A Minimizer-Aware Bloom Filter for Genomic Sequence Data on
Modern GPUs", Algorithm 1 (insert), Algorithm 2 (query), Fig. 3 (runs).
"""
import numpy as np
import pytest

import oracle
from oracle import brute
from minimizer_sharded_bloom_gb300 import synth

ALPHABETS = ["dna", "protein", "dna_triplet"]


def _u64(rng):
    return int(rng.integers(0, 2**63, dtype=np.int64)) * 2 + int(rng.integers(0, 2))


def _params(rng, alphabet, case):
    kmax = {"dna": 32, "protein": 12, "dna_triplet": 10}[alphabet]
    k = int(rng.integers(1, kmax + 1))
    m = int(rng.integers(1, k + 1))
    s = int(rng.integers(1, k + 1))
    H = int(rng.integers(1, 11)) if case % 3 else int(rng.integers(11, 33))
    return k, m, s, H


def _records(rng, alphabet, n, lo, hi, lead=0):
    """Random mixed records; `lead` junk bytes before the first record (so
    offsets[0] > 0 and positions below it belong to no record)."""
    if alphabet == "protein":
        wl = synth.random_protein_records(rng, n, lo, hi, lower_prob=0.1, junk_prob=0.01)
    else:
        wl = synth.random_records(rng, n, lo, hi, n_prob=0.005, lower_prob=0.1, junk_prob=0.002)
    if lead:
        seq = np.concatenate([np.full(lead, ord("A"), np.uint8), wl.seq])
        return synth.Workload(seq, wl.offsets + lead)
    return wl


def _brute_rows(wl, k, m, s, H, shards, seed, alphabet):
    """{absolute position: (shard, words)} of every valid k-mer, by brute force."""
    rows = {}
    for start, rec in brute.records_of(wl.seq.tobytes(), wl.offsets):
        for p, text in brute.kmers_of(rec, k, alphabet):
            if brute.is_valid(text, alphabet):
                rows[start + p] = brute.kmer(text, k, m, s, H, shards, seed, alphabet)
    return rows


@pytest.mark.parametrize("alphabet", ALPHABETS)
@pytest.mark.parametrize("case", range(10))
def test_kmer_batch_matches_brute_force(alphabet, case):
    """Every position of the batch plus positions outside it, in a shuffled
    order: valid, shard and the four words equal the brute force's for valid
    k-mers; everything else (invalid symbol, off-frame codon, too close to a
    record's end, outside [offsets[0], offsets[-1])) is invalid with zeros."""
    rng = np.random.default_rng(7100 + case + 100 * ALPHABETS.index(alphabet))
    k, m, s, H = _params(rng, alphabet, case)
    shards = int(2 ** rng.integers(0, 10))
    seed = _u64(rng)
    wl = _records(rng, alphabet, int(rng.integers(1, 10)), 0, 160, lead=int(rng.integers(0, 40)))
    rows = _brute_rows(wl, k, m, s, H, shards, seed, alphabet)
    lo, hi = int(wl.offsets[0]), int(wl.offsets[-1])
    pos = np.concatenate([np.arange(lo, hi), [lo - 1, hi, hi + 5]]).astype(np.int64)
    pos = pos[pos >= 0]
    rng.shuffle(pos)
    if hi == lo:
        pos = pos[(pos < lo) | (pos >= hi)]
    valid, shard, K = oracle.kmer_batch(wl.seq, wl.offsets, pos, k, m, s, H, shards, seed, alphabet)
    assert valid.size == pos.size
    for i, g in enumerate(pos.tolist()):
        if g in rows:
            sh, words = rows[g]
            assert valid[i], g
            assert int(shard[i]) == sh, g
            assert [int(x) for x in K[i]] == words, g
        else:
            assert not valid[i], g
            assert int(shard[i]) == 0 and not K[i].any(), g
    assert int(valid.sum()) == len(rows)


@pytest.mark.parametrize("alphabet", ALPHABETS)
@pytest.mark.parametrize("case", range(8))
def test_insert_sparse_matches_brute_force_image(alphabet, case):
    """insert_sparse's (sorted shards, words) equal the non-zero shards of the
    brute force's insert, and the dense image of the whole-batch insert."""
    rng = np.random.default_rng(7300 + case + 100 * ALPHABETS.index(alphabet))
    k, m, s, H = _params(rng, alphabet, case)
    shards = int(2 ** rng.integers(0, 12))
    seed = _u64(rng)
    wl = _records(rng, alphabet, int(rng.integers(1, 12)), 0, 200, lead=int(rng.integers(0, 3)) * 17)
    idx, words = oracle.insert_sparse(wl.seq, wl.offsets, k, m, s, H, shards, seed, alphabet)
    assert idx.dtype == np.uint64 and words.shape == (idx.size, 4)
    assert np.all(np.diff(idx.astype(np.int64)) > 0), "shards sorted and distinct"
    ref = brute.insert(wl.seq.tobytes(), wl.offsets, k, m, s, H, shards, seed, alphabet=alphabet)
    ref = {i: w for i, w in ref.items() if any(w)}
    got = {int(i): [int(x) for x in w] for i, w in zip(idx, words)}
    assert got == ref
    F = np.zeros((shards, 4), dtype=np.uint64)
    oracle.insert(F, wl.seq, wl.offsets, k, m, s, H, seed, alphabet=alphabet)
    nz = np.flatnonzero(F.any(axis=1))
    assert np.array_equal(nz.astype(np.uint64), idx)
    assert np.array_equal(F[nz], words)


@pytest.mark.parametrize("alphabet", ALPHABETS)
@pytest.mark.parametrize("case", range(8))
def test_query_sampled_matches_brute_force(alphabet, case):
    """Answers at sampled positions, with the image supplied shard by shard,
    equal the brute force's query of the same image; the lookup is asked only
    for the shards of valid k-mers, in sample order."""
    rng = np.random.default_rng(7500 + case + 100 * ALPHABETS.index(alphabet))
    k, m, s, H = _params(rng, alphabet, case)
    shards = int(2 ** rng.integers(0, 8))
    seed = _u64(rng)
    ins = _records(rng, alphabet, int(rng.integers(1, 10)), 0, 200)
    ref = brute.insert(ins.seq.tobytes(), ins.offsets, k, m, s, H, shards, seed, alphabet=alphabet)
    # query: the inserted records again (all valid ones present) plus fresh ones
    q2 = _records(rng, alphabet, int(rng.integers(1, 8)), 0, 150)
    qseq = np.concatenate([ins.seq, q2.seq])
    qoff = np.concatenate([ins.offsets, ins.offsets[-1] + q2.offsets[1:]])
    hits = brute.query(ref, qseq.tobytes(), qoff, k, m, s, H, shards, seed, alphabet=alphabet)
    lo, hi = int(qoff[0]), int(qoff[-1])
    pos = rng.integers(lo, max(hi, lo + 1), size=min(400, max(hi - lo, 1))).astype(np.int64)
    asked = []

    def lookup(idx):
        asked.append(np.array(idx, copy=True))
        return np.array([ref.get(int(i), [0, 0, 0, 0]) for i in idx], dtype=np.uint64)

    got = oracle.query_sampled(lookup, qseq, qoff, pos, k, m, s, H, shards, seed, alphabet)
    assert got.dtype == bool and got.size == pos.size
    for i, g in enumerate(pos.tolist()):
        assert bool(got[i]) == (g in hits), g
    valid, shard, _ = oracle.kmer_batch(qseq, qoff, pos, k, m, s, H, shards, seed, alphabet)
    if valid.any():
        assert len(asked) == 1 and np.array_equal(asked[0], shard[valid])
    else:
        assert not asked


@pytest.mark.parametrize("alphabet", ALPHABETS)
def test_sampling_helpers_match_whole_batch_oracle_medium(alphabet):
    """Medium batches (tens of kbp, hundreds of records including empty and
    short ones, N runs): kmer_batch on every position equals kmer_info;
    insert_sparse equals the whole-batch insert's non-zero shards; and
    query_sampled on every position equals the whole-batch query's bits on a
    filter that is a quarter full (so the subset test decides)."""
    rng = np.random.default_rng({"dna": 81, "protein": 82, "dna_triplet": 83}[alphabet])
    k, m, s, H = {"dna": (31, 16, 28, 4), "protein": (12, 8, 10, 4), "dna_triplet": (10, 5, 8, 4)}[alphabet]
    shards = 1 << 9
    seed = _u64(rng)
    wl = _records(rng, alphabet, 300, 0, 300, lead=5)
    lo, hi = int(wl.offsets[0]), int(wl.offsets[-1])
    pos = np.arange(lo, hi, dtype=np.int64)
    valid, shard, K = oracle.kmer_batch(wl.seq, wl.offsets, pos, k, m, s, H, shards, seed, alphabet)
    for g in rng.choice(pos, size=300, replace=False).tolist():
        ok, sh, w = oracle.kmer_info(wl.seq, wl.offsets, g, k, m, s, H, shards, seed, alphabet)
        i = g - lo
        assert bool(valid[i]) == ok
        if ok:
            assert int(shard[i]) == sh and [int(x) for x in K[i]] == w
    assert valid.sum() > 1000
    # insert half of the records; the image is then partly full
    half = synth.Workload(wl.seq, wl.offsets[: wl.offsets.size // 2 + 1])
    F = np.zeros((shards, 4), dtype=np.uint64)
    oracle.insert(F, half.seq, half.offsets, k, m, s, H, seed, alphabet=alphabet)
    idx, words = oracle.insert_sparse(half.seq, half.offsets, k, m, s, H, shards, seed, alphabet)
    nz = np.flatnonzero(F.any(axis=1))
    assert np.array_equal(nz.astype(np.uint64), idx) and np.array_equal(F[nz], words)
    want = oracle.query(F, wl.seq, wl.offsets, k, m, s, H, seed, alphabet=alphabet)
    got = oracle.query_sampled(lambda ix: F[ix.astype(np.int64)], wl.seq, wl.offsets, pos,
                               k, m, s, H, shards, seed, alphabet)
    want_bits = ((want[pos >> 5] >> (pos & 31).astype(np.uint32)) & 1).astype(bool)
    assert np.array_equal(got, want_bits)
    # both answers occur: the subset test is exercised
    assert got.any() and (valid & ~got).any()


def _brute_runs(wl, k, m, s, H, shards, seed, alphabet):
    """(valid k-mers, runs, non-zero words summed over runs), by brute force:
    a run is a maximal stretch of consecutive valid k-mers (one symbol apart)
    of one record with one shard (Fig. 3)."""
    nv = nr = na = 0
    width = 3 if alphabet == "dna_triplet" else 1
    for _, rec in brute.records_of(wl.seq.tobytes(), wl.offsets):
        cur = None
        acc = None
        for p in range(0, len(rec), width):
            text = rec[p:p + width * k]
            ok = len(text) == width * k and brute.is_valid(text, alphabet)
            if ok:
                sh, words = brute.kmer(text, k, m, s, H, shards, seed, alphabet)
                nv += 1
                if cur is not None and sh == cur:
                    acc = [a | b for a, b in zip(acc, words)]
                    continue
                if cur is not None:
                    na += sum(1 for a in acc if a)
                nr += 1
                cur, acc = sh, list(words)
            else:
                if cur is not None:
                    na += sum(1 for a in acc if a)
                cur = None
        if cur is not None:
            na += sum(1 for a in acc if a)
    return nv, nr, na


@pytest.mark.parametrize("alphabet", ALPHABETS)
@pytest.mark.parametrize("case", range(6))
def test_count_runs_matches_brute_force(alphabet, case):
    """count_runs (whose run count sets the benchmark's algorithmic bytes)
    equals a brute-force count of Fig. 3's runs and of their non-zero words."""
    rng = np.random.default_rng(7700 + case + 100 * ALPHABETS.index(alphabet))
    k, m, s, H = _params(rng, alphabet, case)
    shards = int(2 ** rng.integers(0, 6))
    seed = _u64(rng)
    wl = _records(rng, alphabet, int(rng.integers(1, 10)), 0, 200)
    assert oracle.count_runs(wl.seq, wl.offsets, k, m, s, H, shards, seed, alphabet) == \
        _brute_runs(wl, k, m, s, H, shards, seed, alphabet)
