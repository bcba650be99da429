"""Pins of the oracle's hash-chosen-sector option (an extension of the paper's
layout, not the paper's default).

"cuSBF" Sec. IV-B (and Algorithm 2) puts hash i of an s-mer in word i mod 4 of
its 256-bit shard; with H < 4 words H..3 of every shard then stay empty and a
k-mer's bits fall in only 64 H of the 256.  With sectors = 1, hash i of an
H < 4 filter goes to the word numbered by the two bits of its slice (Sec.
IV-G bit-slicing, slice width floor(64/H) >= 21) just above its six position
bits; H >= 4 keeps i mod 4.

Each test checks the option against something other than the oracle's own
code: the independent pure-Python brute force, the paper's default layout
(identical images when the option cannot apply), the spread of bits over the
four words, and Eq. 1 with all 256 bits of a shard in play.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import brute
from minimizer_sharded_bloom_gb300 import synth


def _u64(rng):
    return int(rng.integers(0, 2**63, dtype=np.int64)) * 2 + int(rng.integers(0, 2))


def _image_dict(F):
    nz = np.flatnonzero(F.any(axis=1))
    return {int(i): [int(x) for x in F[i]] for i in nz}


def _bits_to_set(out, off):
    lo, hi = int(off[0]), int(off[-1])
    return {g for g in range(lo, hi) if (int(out[g >> 5]) >> (g & 31)) & 1}


@pytest.mark.parametrize("alphabet", ["dna", "protein", "dna_triplet"])
@pytest.mark.parametrize("case", range(12))
def test_hashed_sectors_agree_with_brute_force(alphabet, case):
    """C oracle == brute force with sectors = 1: image and answers, random
    tiny inputs, H mostly below 4 (where the option applies)."""
    rng = np.random.default_rng(9100 + case + {"dna": 0, "protein": 300, "dna_triplet": 600}[alphabet])
    kmax = {"dna": 32, "protein": 12, "dna_triplet": 10}[alphabet]
    k = int(rng.integers(1, kmax + 1))
    m = int(rng.integers(1, k + 1))
    s = int(rng.integers(1, k + 1))
    H = int(rng.integers(1, 4)) if case % 4 else int(rng.integers(4, 17))
    shards = int(2 ** rng.integers(0, 7))
    seed = _u64(rng)
    if alphabet == "protein":
        wl = synth.random_protein_records(rng, int(rng.integers(1, 10)), 0, 90, lower_prob=0.1, junk_prob=0.01)
        q = synth.random_protein_records(rng, int(rng.integers(1, 6)), 0, 70)
    else:
        wl = synth.random_records(rng, int(rng.integers(1, 10)), 0, 200, n_prob=0.005, lower_prob=0.1)
        q = synth.random_records(rng, int(rng.integers(1, 6)), 0, 150, n_prob=0.005)
    F = np.zeros((shards, 4), dtype=np.uint64)
    oracle.insert(F, wl.seq, wl.offsets, k, m, s, H, seed, alphabet=alphabet, sectors=1)
    ref = brute.insert(wl.seq.tobytes(), wl.offsets, k, m, s, H, shards, seed, alphabet=alphabet, sectors=1)
    assert _image_dict(F) == {i: w for i, w in ref.items() if any(w)}
    qseq = np.concatenate([wl.seq, q.seq])
    qoff = np.concatenate([wl.offsets, wl.offsets[-1] + q.offsets[1:]])
    out = oracle.query(F, qseq, qoff, k, m, s, H, seed, alphabet=alphabet, sectors=1)
    hits = brute.query(ref, qseq.tobytes(), qoff, k, m, s, H, shards, seed, alphabet=alphabet, sectors=1)
    assert _bits_to_set(out, qoff) == hits


@pytest.mark.parametrize("H", [4, 5, 6, 8, 10, 12, 16])
def test_hashed_sectors_leave_h4_and_above_unchanged(H):
    """From H = 4 on every word already takes hashes (i mod 4), and the option
    does not apply: images equal the paper's layout bit for bit."""
    rng = np.random.default_rng(9400 + H)
    wl = synth.random_records(rng, 20, 50, 2000, n_prob=0.002)
    imgs = []
    for sectors in (0, 1):
        F = np.zeros((64, 4), dtype=np.uint64)
        oracle.insert(F, wl.seq, wl.offsets, 31, 16, 28, H, 77, sectors=sectors)
        imgs.append(F)
    assert np.array_equal(imgs[0], imgs[1]) and imgs[0].any()


@pytest.mark.parametrize("H", [1, 2, 3])
def test_hashed_sectors_spread_bits_over_all_four_words(H):
    """Over random s-mer hashes: with the paper's layout words H..3 never
    receive a bit; with hash-chosen sectors each word receives a quarter of
    them (chi-square, 3 degrees of freedom) and, inside each word, the 64
    positions are equally likely (chi-square, 63 degrees of freedom)."""
    rng = np.random.default_rng(9500 + H)
    n = 40_000
    per_word = np.zeros(4)
    per_pos = np.zeros((4, 64))
    fixed = np.zeros(4)
    for _ in range(n):
        h = _u64(rng)
        w = oracle.smer_bits(h, H, 1)
        w0 = oracle.smer_bits(h, H, 0)
        for j in range(4):
            x, y = w[j], w0[j]
            fixed[j] += bin(y).count("1")
            while x:
                b = (x & -x).bit_length() - 1
                per_word[j] += 1
                per_pos[j, b] += 1
                x &= x - 1
    assert fixed[H:].sum() == 0 and fixed[:H].sum() > 0
    exp = per_word.sum() / 4
    chi2 = ((per_word - exp) ** 2 / exp).sum()
    assert chi2 < 16.3, per_word  # p = 0.001
    for j in range(4):
        e = per_pos[j].sum() / 64
        assert ((per_pos[j] - e) ** 2 / e).sum() < 103.4  # p = 0.001 at 63 dof


def _random_kmers(rng, n, k):
    return synth.uniform_bases(rng, n * k), synth.csr(np.full(n, k))


@pytest.mark.parametrize("H", [1, 2, 3])
def test_fpr_with_hashed_sectors_matches_eq1_over_256_bits(H):
    """Eq. 1 inside a shard with all 256 bits in play: with s = k (one s-mer
    per k-mer) each of an alien k-mer's H bits lands on a uniform position of
    the 256 bits of its uniform shard, so the expected false-positive rate is
    the mean over shards of (set bits / 256)^H.  The measured rate matches it
    and is well below the paper's-layout prediction for the same image, which
    would confine the bits to 64 H of the 256."""
    rng = np.random.default_rng(9600 + H)
    k = s = 31
    S, seed = 256, 4242
    n_ins = {1: 60_000, 2: 30_000, 3: 20_000}[H]
    seq, off = _random_kmers(rng, n_ins, k)
    F = oracle.insert(np.zeros((S, 4), np.uint64), seq, off, k, 16, s, H, seed, nthreads=4, sectors=1)
    bits = np.unpackbits(F.view(np.uint8)).reshape(S, 4, 64)
    pop = bits.sum(axis=(1, 2))
    expect = np.mean((pop / 256.0) ** H)
    # what the paper's layout would predict for this many set bits per shard
    confined = np.mean(np.minimum(pop / (64.0 * H), 1.0) ** H)
    qseq, qoff = _random_kmers(rng, 200_000, k)
    out = oracle.query(F, qseq, qoff, k, 16, s, H, seed, nthreads=4, sectors=1)
    starts = qoff[:-1]
    hits = (out[starts >> 5] >> (starts & 31).astype(np.uint32)) & 1
    rate, n = hits.mean(), hits.size
    sigma = math.sqrt(expect * (1 - expect) / n)
    assert abs(rate - expect) < 5 * sigma + 0.02 * expect, (rate, expect)
    assert confined > 1.5 * expect
    # every word of the shards took bits
    assert (bits.sum(axis=2) > 0).all(axis=0).all()
