"""Seeded synthetic DNA and protein workloads.

This module only draws inputs: byte sequences over ACGT (plus N runs) or over
amino-acid letters, and CSR offsets.  It holds none of the filter's arithmetic, so both the CUDA path's
tests and the CPU oracle's tests may use it.  Every generator uses numpy's
PCG64 with an explicit seed and is deterministic.

The public genomes of the cuSBF evaluation (C. elegans, T2T-CHM13, Sec. V-A)
are not available; these workloads stand in for them:

* tiny          -- 100 kbp uniform; query = the same 100 kbp + an independent
                   100 kbp (seeds 1, 2);
* genome_like   -- 50 Mbp uniform with 20 % of its length made of copies of
                   earlier 1-10 kbp segments at 1 % substitution; 1 M reads of
                   150 bp, half from it at 1 % substitution, half uniform
                   (seeds 3, 4);
* out_of_cache  -- 1 Gbp in 10,000 log-normal contigs (median 50 kbp,
                   sigma = sqrt(2 ln 2)); 6,666,666 reads of 150 bp, half from
                   the contigs at 1 % substitution, half uniform (seeds 5, 6);
* sweep_queries -- 10 M uniform 31-mers (one per record) none of which occurs
                   in the inserted sequence (seed 7);
* irregular     -- 200,000 long reads, log-normal lengths (median 8 kbp,
                   sigma 1.0, clipped to [1, 100,000]), ~0.1 % N in runs of
                   1-50; two independent sets (seeds 8, 9);
* protein_like  -- 500 M residues uniform over the 20 standard amino-acid
                   letters in log-normal proteins (median 300, sigma 0.6,
                   clipped to [30, 5,000]); 10 M fragments of 50 residues,
                   half from the proteins at 1 % substitution, half uniform
                   (seeds 10, 11).  No protein database is available; the
                   cuSBF paper evaluates DNA only.
"""
from __future__ import annotations

import numpy as np

ACGT = np.frombuffer(b"ACGT", dtype=np.uint8)
# the 20 standard amino acids, sorted
AMINO20 = np.frombuffer(b"ACDEFGHIKLMNPQRSTVWY", dtype=np.uint8)


def fingerprint(seq: np.ndarray, offsets: np.ndarray) -> str:
    """A short identity of a generated input: sha256 of the offsets, every
    4,097th byte of the sequence and its length.  Lets a stored per-input
    count be matched to the input it was computed on."""
    import hashlib
    h = hashlib.sha256()
    h.update(np.ascontiguousarray(offsets, dtype=np.int64).tobytes())
    h.update(np.ascontiguousarray(seq[::4097]).tobytes())
    h.update(str(seq.size).encode())
    return h.hexdigest()[:32]


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


_CHUNK = 1 << 26


def uniform_bases(rng: np.random.Generator, n: int, symbols: np.ndarray = ACGT) -> np.ndarray:
    """n i.i.d. uniform symbols, ACGT by default (drawn in chunks of 2^26)."""
    out = np.empty(n, dtype=np.uint8)
    for c in range(0, n, _CHUNK):
        m = min(_CHUNK, n - c)
        out[c:c + m] = symbols[rng.integers(0, symbols.size, size=m, dtype=np.uint8)]
    return out


def substitute(rng: np.random.Generator, seq: np.ndarray, rate: float,
               symbols: np.ndarray = ACGT) -> np.ndarray:
    """Each symbol independently, with probability `rate`, becomes one of the
    other symbols of the (sorted) alphabet, chosen uniformly.  Returns a new
    array (chunks of 2^26: a uniform draw per symbol, then a uniform shift of
    1..len-1 for the hit ones)."""
    out = seq.copy()
    a = symbols.size
    for c in range(0, seq.size, _CHUNK):
        part = out[c:c + _CHUNK]
        hit = np.flatnonzero(rng.random(part.size) < rate)
        if hit.size:
            idx = np.searchsorted(symbols, part[hit])
            shift = rng.integers(1, a, size=hit.size)
            part[hit] = symbols[(idx + shift) % a]
    return out


def csr(lengths) -> np.ndarray:
    off = np.zeros(len(lengths) + 1, dtype=np.int64)
    np.cumsum(np.asarray(lengths, dtype=np.int64), out=off[1:])
    return off


class Workload:
    """One side of a config: a byte buffer plus CSR record offsets."""

    def __init__(self, seq: np.ndarray, offsets: np.ndarray, note: str = "", **meta):
        self.seq = np.ascontiguousarray(seq, dtype=np.uint8)
        self.offsets = np.ascontiguousarray(offsets, dtype=np.int64)
        self.note = note
        self.meta = meta

    @property
    def n_records(self) -> int:
        return self.offsets.size - 1

    @property
    def n_bases(self) -> int:
        return int(self.offsets[-1] - self.offsets[0])

    def kmer_positions(self, k: int) -> int:
        lengths = np.diff(self.offsets)
        return int(np.maximum(lengths - k + 1, 0).sum())


def tiny(seed_insert: int = 1, seed_query: int = 2):
    ref = uniform_bases(_rng(seed_insert), 100_000)
    other = uniform_bases(_rng(seed_query), 100_000)
    ins = Workload(ref, csr([ref.size]), "tiny insert: 100,000 bp uniform")
    qry = Workload(np.concatenate([ref, other]), csr([ref.size, other.size]),
                   "tiny query: the inserted 100,000 bp + 100,000 bp uniform",
                   is_random=np.array([False, True]))
    return ins, qry


def genome_like_reference(seed: int = 3, length: int = 50_000_000,
                          copy_fraction: float = 0.20) -> np.ndarray:
    """Left to right: uniform blocks (length uniform in [1, 44,000], mean
    22 kbp) each followed by one copy event -- a copy of an earlier segment of
    length uniform in [1,000, 10,000], source start uniform over what exists,
    with 1 % substitutions -- until the copies total copy_fraction * length;
    then uniform bases to the end, truncated to exactly `length`."""
    rng = _rng(seed)
    parts, have, copied = [], 0, 0
    budget = int(round(copy_fraction * length))
    buf = np.empty(length, dtype=np.uint8)
    while have < length:
        blk = int(rng.integers(1, 44_001))
        blk = min(blk, length - have)
        buf[have:have + blk] = uniform_bases(rng, blk)
        have += blk
        if have >= length or copied >= budget:
            if copied >= budget and have < length:
                rest = length - have
                buf[have:] = uniform_bases(rng, rest)
                have = length
            continue
        clen = int(rng.integers(1_000, 10_001))
        clen = min(clen, budget - copied, length - have)
        if clen <= 0 or have < clen:
            continue
        src = int(rng.integers(0, have - clen + 1))
        buf[have:have + clen] = substitute(rng, buf[src:src + clen], 0.01)
        have += clen
        copied += clen
    del parts
    return buf


def sample_reads(rng: np.random.Generator, source: np.ndarray, source_offsets: np.ndarray,
                 n_from_source: int, n_random: int, read_len: int, error: float,
                 symbols: np.ndarray = ACGT):
    """Reads of read_len bp: n_from_source taken from the source records
    (record chosen with probability proportional to its number of read
    starts, start uniform within it, forward strand, `error` substitution
    rate) and n_random uniform reads, shuffled together.  Returns the
    concatenated reads, their offsets and a boolean 'is uniform-random' per
    read."""
    lengths = np.diff(source_offsets)
    starts_per = np.maximum(lengths - read_len + 1, 0)
    total = int(starts_per.sum())
    if n_from_source and total <= 0:
        raise ValueError("source records are shorter than the read length")
    pick = rng.integers(0, total, size=n_from_source) if n_from_source else np.zeros(0, np.int64)
    cum = np.concatenate([[0], np.cumsum(starts_per)])
    rec = np.searchsorted(cum, pick, side="right") - 1
    start = source_offsets[rec] + (pick - cum[rec])
    n = n_from_source + n_random
    reads = np.empty((n, read_len), dtype=np.uint8)
    order = rng.permutation(n)
    src_slots, rnd_slots = order[:n_from_source], order[n_from_source:]
    # gather the source reads in chunks to bound memory
    chunk = 1 << 20
    for c in range(0, n_from_source, chunk):
        st = start[c:c + chunk]
        idx = st[:, None] + np.arange(read_len, dtype=np.int64)[None, :]
        reads[src_slots[c:c + chunk]] = source[idx]
    if n_from_source:
        flat = reads[src_slots].reshape(-1)
        reads[src_slots] = substitute(rng, flat, error, symbols).reshape(-1, read_len)
    if n_random:
        reads[rnd_slots] = uniform_bases(rng, n_random * read_len, symbols).reshape(-1, read_len)
    is_random = np.zeros(n, dtype=bool)
    is_random[rnd_slots] = True
    return reads.reshape(-1), csr(np.full(n, read_len)), is_random


def genome_like(seed_insert: int = 3, seed_query: int = 4, length: int = 50_000_000,
                n_reads: int = 1_000_000, read_len: int = 150):
    ref = genome_like_reference(seed_insert, length)
    ins = Workload(ref, csr([ref.size]),
                   f"genome-like insert: {length:,} bp, 20% copied segments at 1% error")
    reads, off, is_random = sample_reads(_rng(seed_query), ref, ins.offsets,
                                         n_reads // 2, n_reads - n_reads // 2, read_len, 0.01)
    qry = Workload(reads, off, f"genome-like query: {n_reads:,} reads x {read_len} bp",
                   is_random=is_random)
    return ins, qry


def lognormal_lengths(rng: np.random.Generator, n: int, median: float, sigma: float) -> np.ndarray:
    return rng.lognormal(mean=np.log(median), sigma=sigma, size=n)


def out_of_cache_contigs(seed: int = 5, total: int = 1_000_000_000, n_contigs: int = 10_000):
    rng = _rng(seed)
    raw = lognormal_lengths(rng, n_contigs, 50_000.0, np.sqrt(2.0 * np.log(2.0)))
    lengths = np.floor(raw * (total / raw.sum())).astype(np.int64)
    lengths = np.maximum(lengths, 1)
    lengths[np.argmax(lengths)] += total - int(lengths.sum())
    seq = uniform_bases(rng, total)
    return Workload(seq, csr(lengths),
                    f"out-of-cache insert: {total:,} bp in {n_contigs:,} log-normal contigs")


def out_of_cache(seed_insert: int = 5, seed_query: int = 6, total: int = 1_000_000_000,
                 n_contigs: int = 10_000, read_len: int = 150):
    ins = out_of_cache_contigs(seed_insert, total, n_contigs)
    n_reads = total // read_len
    reads, off, is_random = sample_reads(_rng(seed_query), ins.seq, ins.offsets,
                                         n_reads // 2, n_reads - n_reads // 2, read_len, 0.01)
    qry = Workload(reads, off, f"out-of-cache query: {n_reads:,} reads x {read_len} bp",
                   is_random=is_random)
    return ins, qry


def _identity_codes(windows: np.ndarray) -> np.ndarray:
    """Injective integer for each row of ACGT bytes (bits 1-2 of each byte:
    A0 C1 T2 G3).  Used only to test string equality between 31-mers."""
    k = windows.shape[1]
    assert k <= 32
    codes = ((windows >> 1) & 3).astype(np.uint64)
    out = np.zeros(windows.shape[0], dtype=np.uint64)
    for i in range(k):
        out = (out << np.uint64(2)) | codes[:, i]
    return out


def distinct_kmer_codes(seq: np.ndarray, offsets: np.ndarray, k: int) -> np.ndarray:
    """Sorted unique identity codes of every ACGT-only k-mer of every record."""
    out = []
    for r in range(offsets.size - 1):
        rec = seq[offsets[r]:offsets[r + 1]]
        if rec.size < k:
            continue
        for c in range(0, rec.size - k + 1, 1 << 24):
            part = rec[c:min(rec.size, c + (1 << 24) + k - 1)]
            win = np.lib.stride_tricks.sliding_window_view(part, k)
            ok = np.isin(win, ACGT).all(axis=1)
            out.append(_identity_codes(win[ok]))
    if not out:
        return np.zeros(0, dtype=np.uint64)
    return np.unique(np.concatenate(out))


def sweep_queries(inserted: Workload, seed: int = 7, n: int = 10_000_000, k: int = 31):
    """n uniform k-mers, one per record, redrawn until none occurs in the
    inserted sequence (exact check on the strings)."""
    rng = _rng(seed)
    present = distinct_kmer_codes(inserted.seq, inserted.offsets, k)
    kmers = uniform_bases(rng, n * k).reshape(n, k)
    for _ in range(100):
        codes = _identity_codes(kmers)
        pos = np.searchsorted(present, codes)
        pos = np.minimum(pos, max(present.size - 1, 0))
        clash = np.flatnonzero(present[pos] == codes) if present.size else np.zeros(0, np.int64)
        if clash.size == 0:
            break
        kmers[clash] = uniform_bases(rng, clash.size * k).reshape(-1, k)
    else:  # pragma: no cover
        raise RuntimeError("could not draw absent k-mers")
    return Workload(kmers.reshape(-1), csr(np.full(n, k)),
                    f"sweep query: {n:,} uniform {k}-mers absent from the inserted set",
                    is_random=np.ones(n, dtype=bool))


def irregular_set(seed: int, n_reads: int = 200_000, median: float = 8_000.0,
                  sigma: float = 1.0, max_len: int = 100_000, n_rate: float = 0.001,
                  max_run: int = 50):
    """Long reads with log-normal lengths and N runs: each base starts an N run
    with probability n_rate / mean_run (mean_run = (1 + max_run) / 2), run
    length uniform in [1, max_run], so ~n_rate of all bases are N."""
    rng = _rng(seed)
    lengths = np.clip(np.rint(lognormal_lengths(rng, n_reads, median, sigma)), 1, max_len)
    lengths = lengths.astype(np.int64)
    off = csr(lengths)
    total = int(off[-1])
    seq = uniform_bases(rng, total)
    mean_run = (1 + max_run) / 2.0
    n_runs = int(rng.binomial(total, n_rate / mean_run))
    starts = rng.integers(0, total, size=n_runs)
    run_len = rng.integers(1, max_run + 1, size=n_runs)
    # expand the runs without a python loop
    idx = np.repeat(starts, run_len) + (np.arange(run_len.sum()) -
                                        np.repeat(np.cumsum(run_len) - run_len, run_len))
    idx = idx[idx < total]
    seq[idx] = ord("N")
    return Workload(seq, off, f"irregular: {n_reads:,} long reads, {total:,} bp, ~0.1% N")


def irregular(seed_insert: int = 8, seed_query: int = 9, **kw):
    return irregular_set(seed_insert, **kw), irregular_set(seed_query, **kw)


def protein_like(seed_insert: int = 10, seed_query: int = 11, total: int = 500_000_000,
                 median: float = 300.0, sigma: float = 0.6, frag_len: int = 50):
    """Protein stand-in: `total` residues uniform over AMINO20 in log-normal
    proteins; fragments of frag_len residues, half from the proteins at 1 %
    substitution, half uniform."""
    rng = _rng(seed_insert)
    n = max(1, int(total / (median * np.exp(sigma * sigma / 2))))
    lengths = np.clip(np.rint(lognormal_lengths(rng, n, median, sigma)), 30, 5_000).astype(np.int64)
    lengths = lengths[np.cumsum(lengths) <= total]
    if lengths.sum() < total:
        lengths = np.append(lengths, total - lengths.sum())
    seq = uniform_bases(rng, total, AMINO20)
    ins = Workload(seq, csr(lengths), f"protein-like insert: {total:,} residues in {lengths.size:,} proteins")
    n_frag = total // frag_len
    frags, off, is_random = sample_reads(_rng(seed_query), ins.seq, ins.offsets, n_frag // 2,
                                         n_frag - n_frag // 2, frag_len, 0.01, AMINO20)
    qry = Workload(frags, off, f"protein-like query: {n_frag:,} fragments x {frag_len} residues",
                   is_random=is_random)
    return ins, qry


def random_protein_records(rng: np.random.Generator, n_records: int, min_len: int, max_len: int,
                           lower_prob: float = 0.0, junk_prob: float = 0.0):
    """Small mixed protein inputs: uniform over all 26 letters, optional
    lowercase letters and other bytes (stop '*', gap '-', digits, controls)."""
    lengths = rng.integers(min_len, max_len + 1, size=n_records)
    off = csr(lengths)
    letters = np.arange(ord("A"), ord("Z") + 1, dtype=np.uint8)
    seq = uniform_bases(rng, int(off[-1]), letters)
    if lower_prob:
        low = rng.random(seq.size) < lower_prob
        seq[low] |= 0x20
    if junk_prob:
        junk = rng.random(seq.size) < junk_prob
        seq[junk] = rng.choice(np.frombuffer(b"*-.019@[`{\x00\xff\xc1\xe1", dtype=np.uint8),
                               size=int(junk.sum()))
    return Workload(seq, off, "random mixed protein records")


def random_records(rng: np.random.Generator, n_records: int, min_len: int, max_len: int,
                   n_prob: float = 0.0, lower_prob: float = 0.0, junk_prob: float = 0.0):
    """Small mixed test inputs: record lengths uniform in [min_len, max_len],
    uniform ACGT with optional N bases, lowercase bases and other bytes."""
    lengths = rng.integers(min_len, max_len + 1, size=n_records)
    off = csr(lengths)
    seq = uniform_bases(rng, int(off[-1]))
    if n_prob:
        seq[rng.random(seq.size) < n_prob] = ord("N")
    if lower_prob:
        low = rng.random(seq.size) < lower_prob
        seq[low] = np.where(seq[low] == ord("N"), seq[low], seq[low] | 0x20)
    if junk_prob:
        junk = rng.random(seq.size) < junk_prob
        seq[junk] = rng.choice(np.frombuffer(b"RYKMSWnx-*.\x00\xff", dtype=np.uint8),
                               size=int(junk.sum()))
    return Workload(seq, off, "random mixed records")
