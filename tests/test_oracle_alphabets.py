"""Pins of the CPU oracle's protein and DNA-triplet alphabets ("cuSBF",
Sec. IV-A: proteins, 26 symbols in 5 bits; DNA triplets, 64 symbols in 6 bits,
one symbol over several bytes; Sec. IV-C: a k-mer packs into one 64-bit word).

Each test checks the oracle against something other than itself: the
independent pure-Python brute force, Python's own base-32 integer parsing, the
already pinned 2-bit DNA packing, the record-relative codon frame, the
parameter limits that the 64-bit packing implies, and the paper's Eq. 2 and
2/(w+1) density laws on protein input.  None of them needs a GPU.
"""
import math

import numpy as np
import pytest

import oracle
from oracle import brute
from minimizer_sharded_bloom_gb300 import synth

_DIGITS32 = "0123456789abcdefghijklmnopqrstuv"


def _u64(rng):
    return int(rng.integers(0, 2**63, dtype=np.int64)) * 2 + int(rng.integers(0, 2))


def _image_dict(F):
    nz = np.flatnonzero(F.any(axis=1))
    return {int(i): [int(x) for x in F[i]] for i in nz}


def _bits_to_set(out, off):
    lo, hi = int(off[0]), int(off[-1])
    return {g for g in range(lo, hi) if (int(out[g >> 5]) >> (g & 31)) & 1}


def _csr_of(texts):
    seq = "".join(texts).encode()
    return np.frombuffer(seq, dtype=np.uint8).copy(), synth.csr([len(t) for t in texts])


# ------------------------------------------------------------------ symbols ---

def test_protein_code_map_all_bytes():
    """Every byte: the 26 letters, either case, are 0..25 in alphabet order;
    everything else (stop '*', gap '-', digits, '@', '[', '`', '{', high
    bytes) is invalid."""
    for b in range(256):
        want = b - 65 if 65 <= b <= 90 else b - 97 if 97 <= b <= 122 else -1
        assert oracle.symbol_code(bytes([b]), "protein") == want, b


def test_protein_pack_is_a_base32_number():
    """A protein t-mer packs to the number whose base-32 digits are its
    letters' indices (Python's int(text, 32) on the digit string)."""
    rng = np.random.default_rng(5)
    for t in range(1, 13):
        for _ in range(20):
            idx = rng.integers(0, 26, size=t)
            text = bytes(65 + int(i) + (32 if rng.random() < 0.3 else 0) for i in idx)
            want = int("".join(_DIGITS32[int(i)] for i in idx), 32)
            assert oracle.pack_symbols(text, "protein") == want


def test_triplet_pack_equals_dna_pack_of_its_bases():
    """Six bits per codon, first base most significant, is the 2-bit DNA
    packing of the same 3t bases (the DNA packing is pinned separately as a
    base-4 number); a codon with any invalid base is an invalid symbol."""
    rng = np.random.default_rng(6)
    for t in range(1, 11):
        for _ in range(20):
            text = synth.uniform_bases(rng, 3 * t).tobytes()
            assert oracle.pack_symbols(text, "triplet") == oracle.pack(text)
            assert oracle.pack_symbols(text, "triplet") == int(
                "".join(str("ACGT".index(c)) for c in text.decode()), 4)
    for codon in [b"ACN", b"NAC", b"A-C", b"acg", b"ACG"]:
        bad = any(c not in b"ACGTacgt" for c in codon)
        code = oracle.symbol_code(codon, "triplet")
        assert (code == -1) == bad
    assert oracle.symbol_code(b"acg", "triplet") == oracle.symbol_code(b"ACG", "triplet") == 6


def test_symbol_widths():
    assert [oracle.symbol_bits(a) for a in ("dna", "protein", "triplet")] == [2, 5, 6]


@pytest.mark.parametrize("alphabet,kmax", [("dna", 32), ("protein", 12), ("triplet", 10)])
def test_k_limit_is_64_bit_packing(alphabet, kmax):
    """Sec. IV-C: k symbols pack into one 64-bit word, so k * bits <= 64."""
    seq, off = _csr_of(["A" * 120])
    F = np.zeros((4, 4), np.uint64)
    oracle.insert(F, seq, off, kmax, 1, 1, 4, 1, alphabet=alphabet)
    with pytest.raises(ValueError):
        oracle.insert(F, seq, off, kmax + 1, 1, 1, 4, 1, alphabet=alphabet)


# ---------------------------------------------------------- brute-force match ---

@pytest.mark.parametrize("case", range(20))
@pytest.mark.parametrize("alphabet", ["protein", "dna_triplet"])
def test_brute_force_agrees(alphabet, case):
    """C oracle == pure-Python brute force, bit for bit, on tiny random
    records (ragged, empty, shorter than a k-mer, lowercase, invalid symbols)
    for random (k, m, s, H, shards, seed) within the 64-bit packing limit."""
    rng = np.random.default_rng(1000 + case + (0 if alphabet == "protein" else 500))
    kmax = 12 if alphabet == "protein" else 10
    k = int(rng.integers(1, kmax + 1))
    m = int(rng.integers(1, k + 1))
    s = int(rng.integers(1, k + 1))
    H = int(rng.integers(1, 11)) if case % 3 else int(rng.integers(11, 33))
    shards = int(2 ** rng.integers(0, 8))
    seed = _u64(rng)
    if alphabet == "protein":
        wl = synth.random_protein_records(rng, int(rng.integers(1, 12)), 0, 90,
                                          lower_prob=0.1, junk_prob=0.01)
        q = synth.random_protein_records(rng, int(rng.integers(1, 8)), 0, 70, junk_prob=0.01)
    else:
        wl = synth.random_records(rng, int(rng.integers(1, 12)), 0, 200, n_prob=0.005,
                                  lower_prob=0.1, junk_prob=0.002)
        q = synth.random_records(rng, int(rng.integers(1, 8)), 0, 150, n_prob=0.005)
    F = np.zeros((shards, 4), dtype=np.uint64)
    oracle.insert(F, wl.seq, wl.offsets, k, m, s, H, seed, alphabet=alphabet)
    ref = brute.insert(wl.seq.tobytes(), wl.offsets, k, m, s, H, shards, seed, alphabet=alphabet)
    assert _image_dict(F) == {i: w for i, w in ref.items() if any(w)}
    qseq = np.concatenate([wl.seq, q.seq])
    qoff = np.concatenate([wl.offsets, wl.offsets[-1] + q.offsets[1:]])
    out = oracle.query(F, qseq, qoff, k, m, s, H, seed, alphabet=alphabet)
    hits = brute.query(ref, qseq.tobytes(), qoff, k, m, s, H, shards, seed, alphabet=alphabet)
    assert _bits_to_set(out, qoff) == hits
    # every inserted valid k-mer answers present (no false negatives)
    own = oracle.query(F, wl.seq, wl.offsets, k, m, s, H, seed, alphabet=alphabet)
    for g in range(int(wl.offsets[0]), int(wl.offsets[-1])):
        ok, _, _ = oracle.kmer_info(wl.seq, wl.offsets, g, k, m, s, H, shards, seed, alphabet)
        assert ((int(own[g >> 5]) >> (g & 31)) & 1) == ok


# ------------------------------------------------------------- codon frame ---

def test_triplet_frame_is_record_relative():
    """Codons are read in frame from each record's start: a clean record of L
    bases holds floor(L/3) - k + 1 k-mers, at offsets 0, 3, 6, ...; prefixing
    three bases shifts every k-mer by 3 and keeps it, prefixing one base
    changes the frame."""
    rng = np.random.default_rng(8)
    k, m, s, H, S, seed = 5, 3, 4, 4, 64, 99
    x = synth.uniform_bases(rng, 61).tobytes().decode()
    for L in (3 * k - 1, 3 * k, 3 * k + 1, 3 * k + 2, 61):
        seq, off = _csr_of(["GG", x[:L]])
        got = [g - 2 for g in range(2, 2 + L)
               if oracle.kmer_info(seq, off, g, k, m, s, H, S, seed, "triplet")[0]]
        assert got == list(range(0, 3 * (L // 3 - k + 1), 3)), L
    seq0, off0 = _csr_of([x])
    seq3, off3 = _csr_of(["CAT" + x])
    seq1, off1 = _csr_of(["C" + x])
    for i in range(0, len(x) // 3 - k + 1):
        a = oracle.kmer_info(seq0, off0, 3 * i, k, m, s, H, S, seed, "triplet")
        b = oracle.kmer_info(seq3, off3, 3 * i + 3, k, m, s, H, S, seed, "triplet")
        assert a == b and a[0]
        assert not oracle.kmer_info(seq1, off1, 3 * i + 1, k, m, s, H, S, seed, "triplet")[0]
    # the query answers only at in-frame first bytes
    F = oracle.insert(np.zeros((S, 4), np.uint64), seq0, off0, k, m, s, H, seed, alphabet="triplet")
    out = oracle.query(F, seq0, off0, k, m, s, H, seed, alphabet="triplet")
    assert _bits_to_set(out, off0) == set(range(0, 3 * (len(x) // 3 - k + 1), 3))


def test_protein_k_equals_m_equals_s():
    """m = s = k: one m-mer and one s-mer per k-mer; two distinct k-mers that
    share their shard differ in their bits unless hashes collide."""
    seq, off = _csr_of(["MKVLAAGIVLLLW"])
    ok, shard, K = oracle.kmer_info(seq, off, 0, 12, 12, 12, 4, 1 << 20, 5, "protein")
    v = oracle.pack_symbols(b"MKVLAAGIVLLL", "protein")
    assert ok and shard == oracle.hash_m(v, 5) & ((1 << 20) - 1)
    assert K == oracle.smer_bits(oracle.hash_s(v, ~5), 4)


# ------------------------------------------------------- statistical law pins ---

def test_protein_fpr_matches_eq2_findere():
    """Eq. 2 on protein 12-mers (s = 10, three s-mers): the measured rate of
    uniform alien k-mers matches the image's exact conditional prediction
    mean_shard(prod_w f_w^(z+1))."""
    rng = np.random.default_rng(33)
    k, m, s, H, S, seed = 12, 6, 10, 4, 64, 2024
    z1 = k - s + 1
    seq = synth.uniform_bases(rng, 1_500 * k, synth.AMINO20)
    off = synth.csr(np.full(1_500, k))
    F = oracle.insert(np.zeros((S, 4), np.uint64), seq, off, k, m, s, H, seed, alphabet="protein")
    f = np.unpackbits(F.view(np.uint8)).reshape(S, 4, 64).sum(axis=2) / 64.0
    pred = np.mean(f.prod(axis=1) ** z1)
    n = 200_000
    qseq = synth.uniform_bases(rng, n * k, synth.AMINO20)
    qoff = synth.csr(np.full(n, k))
    out = oracle.query(F, qseq, qoff, k, m, s, H, seed, nthreads=4, alphabet="protein")
    starts = qoff[:-1]
    rate = ((out[starts >> 5] >> (starts & 31).astype(np.uint32)) & 1).mean()
    assert pred * n >= 10
    sigma = math.sqrt(pred * (1 - pred) / n)
    assert abs(rate - pred) < 5 * sigma + 0.03 * pred, (rate, pred)


@pytest.mark.parametrize("alphabet,k,m", [("protein", 12, 6), ("triplet", 10, 5)])
def test_minimizer_density_two_over_w_plus_one(alphabet, k, m):
    """Sec. II-B1's 2/(w+1) density holds per symbol for any alphabet: mean
    super-k-mer length (w+1)/2 on random sequence (2^62 shards: a run is a
    super-k-mer)."""
    rng = np.random.default_rng(41)
    w = k - m + 1
    symbols = synth.AMINO20 if alphabet == "protein" else synth.ACGT
    seq = synth.uniform_bases(rng, 600_000, symbols)
    off = synth.csr([seq.size])
    valid, runs, _ = oracle.count_runs(seq, off, k, m, k, 4, 1 << 62, 9, alphabet)
    mean_len = valid / runs
    assert abs(mean_len - (w + 1) / 2) / ((w + 1) / 2) < 0.03, mean_len
