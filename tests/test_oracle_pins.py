"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a closed form, a worked example printed in
the cuSBF paper (tests/golden/), the independent pure-Python brute force, an
invariant, or a statistical law the paper states (Eq. 1, Eq. 2, the 2/(w+1)
minimizer density).  None of them needs a GPU.
"""
import math
import os

import numpy as np
import pytest

import oracle
from oracle import brute
from minimizer_sharded_bloom_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
M64 = (1 << 64) - 1


def _csr_of(texts):
    seq = "".join(texts).encode()
    off = synth.csr([len(t) for t in texts])
    return np.frombuffer(seq, dtype=np.uint8).copy(), off


def _read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _image_dict(F):
    nz = np.flatnonzero(F.any(axis=1))
    return {int(i): [int(x) for x in F[i]] for i in nz}


def _bits_to_set(out, off):
    pos = set()
    lo, hi = int(off[0]), int(off[-1])
    for g in range(lo, hi):
        if (int(out[g >> 5]) >> (g & 31)) & 1:
            pos.add(g)
    return pos


# ---------------------------------------------------------------- constants ---

def test_constants_closed_form():
    """C1 = floor(2^64 / phi) ("golden-ratio-derived", Sec. IV-G) and
    C2 = floor((sqrt 2 - 1) 2^64) | 1, from integer square roots."""
    c1, c2 = oracle.constants()
    two64 = 1 << 64
    assert c1 == (math.isqrt(5 * two64 * two64) - two64) // 2
    assert c2 == (math.isqrt(2 * two64 * two64) - two64) | 1
    assert c1 & 1 and c2 & 1  # odd, hence invertible mod 2^64


def test_base_code_map_all_bytes():
    """2-bit DNA (Sec. IV-C) with every non-ACGT byte invalid (Sec. IV-F)."""
    L = oracle.lib()
    want = {ord("A"): 0, ord("C"): 1, ord("G"): 2, ord("T"): 3,
            ord("a"): 0, ord("c"): 1, ord("g"): 2, ord("t"): 3}
    for b in range(256):
        assert L.orc_base_code(b) == want.get(b, -1), b


def test_pack_is_base4_number():
    """A t-mer packs to the base-4 number whose leading digit is its first
    base (shift-and-OR, Sec. IV-C / IV-E)."""
    rng = np.random.default_rng(11)
    for t in list(range(1, 33)) * 4:
        txt = "".join(rng.choice(list("ACGTacgt"), size=t))
        digits = txt.upper().translate(str.maketrans("ACGT", "0123"))
        assert oracle.pack(txt.encode()) == int(digits, 4)


# -------------------------------------------------------------- hash inverses ---

def _u64(rng):
    hi, lo = (int(v) for v in rng.integers(0, 1 << 32, size=2, dtype=np.int64))
    return (hi << 32) | lo


def _inv_xorshift_right(y, shift):
    x = y
    for _ in range(64 // shift + 1):
        x = y ^ (x >> shift)
    return x & M64


def test_hash_m_inverts():
    """hm is x -> (x ^ seed) * C1 -> t ^ (t >> 32); undoing each step in turn
    (xorshift inverse, multiply by C1^-1 mod 2^64, xor seed) returns x."""
    c1, _ = oracle.constants()
    c1_inv = pow(c1, -1, 1 << 64)
    rng = np.random.default_rng(12)
    for _ in range(3000):
        x, seed = _u64(rng), _u64(rng)
        h = oracle.hash_m(x, seed)
        t = _inv_xorshift_right(h, 32)
        assert ((t * c1_inv) & M64) ^ seed == x


def test_hash_s_inverts():
    """hs is (x ^ seed_s) * C1, ^>>32, * C2, ^>>29; the inverse chain returns x."""
    c1, c2 = oracle.constants()
    c1_inv, c2_inv = pow(c1, -1, 1 << 64), pow(c2, -1, 1 << 64)
    rng = np.random.default_rng(13)
    for _ in range(3000):
        x, seed = _u64(rng), _u64(rng)
        h = oracle.hash_s(x, seed)
        t = _inv_xorshift_right(h, 29)
        t = (t * c2_inv) & M64
        t = _inv_xorshift_right(t, 32)
        assert ((t * c1_inv) & M64) ^ seed == x


def test_hash_m_low_bits_depend_on_first_base():
    """The shard uses the low bits of the minimizer hash (Algorithm 1's
    minHash & (NumShards - 1)); they must change when only the first base of
    the m-mer does."""
    seed = 0x1234
    changed = 0
    for tail in range(200):
        a = (0 << 30) | tail
        b = (3 << 30) | tail
        changed += (oracle.hash_m(a, seed) & 0xFFFF) != (oracle.hash_m(b, seed) & 0xFFFF)
    assert changed >= 195


def test_smer_bits_structure():
    """Sec. IV-B / IV-G: hash i lands in word i mod 4; each hash sets exactly
    one bit of its word, so word w holds at most ceil((H - w) / 4) bits and
    words >= H are empty for H < 4 (slicing for H <= 10, salted multiply
    beyond)."""
    rng = np.random.default_rng(14)
    for H in list(range(1, 17)) + [24, 32]:
        for _ in range(200):
            hs = _u64(rng)
            words = oracle.smer_bits(hs, H)
            for w in range(4):
                n_hash = len(range(w, H, 4))
                assert 1 <= bin(words[w]).count("1") <= n_hash if n_hash else words[w] == 0
            assert words == brute.smer_words(hs, H)


# ---------------------------------------------------------- brute-force match ---

@pytest.mark.parametrize("case", range(24))
def test_brute_force_agrees(case):
    """C oracle == pure-Python brute force, bit for bit, on tiny random inputs
    with N bases, lowercase, junk bytes, empty/short records and random
    (k, m, s, H, shards, seed)."""
    rng = np.random.default_rng(100 + case)
    k = int(rng.integers(1, 33))
    m = int(rng.integers(1, k + 1))
    s = int(rng.integers(1, k + 1))
    H = int(rng.integers(1, 11)) if case % 3 else int(rng.integers(11, 33))
    shards = int(2 ** rng.integers(0, 8))
    seed = _u64(rng)
    wl = synth.random_records(rng, int(rng.integers(1, 12)), 0, 160, n_prob=0.02,
                              lower_prob=0.1, junk_prob=0.005)
    F = np.zeros((shards, 4), dtype=np.uint64)
    oracle.insert(F, wl.seq, wl.offsets, k, m, s, H, seed)
    ref = brute.insert(wl.seq.tobytes(), wl.offsets, k, m, s, H, shards, seed)
    assert _image_dict(F) == {i: w for i, w in ref.items() if any(w)}
    # query the same records and a fresh set against the same image
    q = synth.random_records(rng, int(rng.integers(1, 8)), 0, 120, n_prob=0.02)
    qseq = np.concatenate([wl.seq, q.seq])
    qoff = np.concatenate([wl.offsets, wl.offsets[-1] + q.offsets[1:]])
    out = oracle.query(F, qseq, qoff, k, m, s, H, seed)
    hits = brute.query(ref, qseq.tobytes(), qoff, k, m, s, H, shards, seed)
    assert _bits_to_set(out, qoff) == hits


def test_threads_do_not_change_results():
    rng = np.random.default_rng(7)
    wl = synth.random_records(rng, 40, 0, 3000, n_prob=0.001)
    args = (31, 16, 28, 4, 12345)
    F1 = oracle.insert(np.zeros((256, 4), np.uint64), wl.seq, wl.offsets, *args, nthreads=1)
    F4 = oracle.insert(np.zeros((256, 4), np.uint64), wl.seq, wl.offsets, *args, nthreads=5)
    assert np.array_equal(F1, F4)
    o1 = oracle.query(F1, wl.seq, wl.offsets, *args, nthreads=1)
    o4 = oracle.query(F1, wl.seq, wl.offsets, *args, nthreads=7)
    assert np.array_equal(o1, o4)


# ------------------------------------------------------------- worked examples ---

def test_fig2b_findere_decomposition():
    """Fig. 2b: the k-mer ACTGAAACT (k=9, s=6) is represented by exactly the
    four printed s-mers: its bits are the OR of theirs (each s-mer inserted on
    its own with k = s = 6 has no other s-mer)."""
    rows = _read_golden("fig2_worked_example.txt")
    kv = {r[0]: r[1:] for r in rows}
    k, m, s = int(kv["k"][0]), int(kv["m"][0]), int(kv["s"][0])
    kmer = kv["findere_kmer"][0]
    smers = [r[1] for r in rows if r[0] == "smer"]
    assert len(smers) == k - s + 1 == 4
    for H in (1, 4, 7):
        seed = 99
        seq, off = _csr_of([kmer])
        ok, _, K = oracle.kmer_info(seq, off, 0, k, m, s, H, 1, seed)
        assert ok
        want = [0, 0, 0, 0]
        for sm in smers:
            sseq, soff = _csr_of([sm])
            ok_s, _, Ks = oracle.kmer_info(sseq, soff, 0, s, min(m, s), s, H, 1, seed)
            assert ok_s
            want = [a | b for a, b in zip(want, Ks)]
        assert K == want


def test_fig2a_shared_minimizer_selects_one_shard():
    """Fig. 2a: the k-mers of ACTGAAACTTAG that contain GAAAC all target the
    shard of GAAAC when it has the minimum hash.  Choose seeds (by the
    independent brute-force hash) for which GAAAC is the global minimum, and
    check every k-mer's shard is hm(GAAAC) & (S - 1); for seeds where GAAAC
    is the global maximum, no k-mer holding another m-mer picks it."""
    rows = _read_golden("fig2_worked_example.txt")
    kv = {r[0]: r[1:] for r in rows}
    S_txt = kv["sequence"][0]
    k, m, s = int(kv["k"][0]), int(kv["m"][0]), int(kv["s"][0])
    shared = kv["shared_mmer"][0]
    fig_kmers = [(int(r[1]), r[2]) for r in rows if r[0] == "kmer"]
    for p, txt in fig_kmers:
        assert S_txt[p:p + k] == txt and shared in txt
    mmers = {S_txt[i:i + m] for i in range(len(S_txt) - m + 1)}
    seq, off = _csr_of([S_txt])
    shards = 1 << 20
    found_min = found_max = 0
    for seed in range(20000):
        hv = {mm: brute.hm(brute.kmer_value(mm), seed) for mm in mmers}
        order = sorted(hv, key=hv.get)
        if order[0] == shared and found_min < 5:
            found_min += 1
            for p in range(len(S_txt) - k + 1):
                ok, sh, _ = oracle.kmer_info(seq, off, p, k, m, s, 4, shards, seed)
                assert ok and sh == hv[shared] & (shards - 1)
        if order[-1] == shared and found_max < 5:
            found_max += 1
            for p in range(len(S_txt) - k + 1):
                ok, sh, _ = oracle.kmer_info(seq, off, p, k, m, s, 4, shards, seed)
                window = [S_txt[p + i:p + i + m] for i in range(k - m + 1)]
                assert sh == min(hv[w] for w in window) & (shards - 1)
                assert sh != hv[shared] & (shards - 1) or len(set(window)) == 1
        if found_min >= 5 and found_max >= 5:
            break
    assert found_min >= 5 and found_max >= 5


def test_fig3_run_and_atomic_count():
    """Fig. 3: seven active lanes in runs A,A,A,B,B,C,C followed by an inactive
    one give three run heads and 3 x 4 = 12 atomics instead of 28.  The input
    is found by searching sequences with the independent brute-force hash;
    the oracle's run count must agree."""
    rows = _read_golden("fig3_runs.txt")
    kv = {r[0]: r[1:] for r in rows}
    lanes = kv["lanes"]
    active = [x for x in lanes if x != "-"]
    k, m, s, H, shards = 9, 5, 6, 4, 16
    rng = np.random.default_rng(31)
    for attempt in range(200000):
        seed = int(rng.integers(0, 2**40))
        txt = "".join(rng.choice(list("ACGT"), size=len(active) + k - 1)) + "N"
        got = [brute.kmer(txt[p:p + k], k, m, s, H, shards, seed)[0] for p in range(len(active))]
        label = {}
        pattern = [label.setdefault(g, "ABC"[min(len(label), 2)]) for g in got]
        if pattern == active and len(label) == 3:
            break
    else:
        pytest.fail("no input with the Fig. 3 run pattern found")
    seq, off = _csr_of([txt])
    valid, runs, atomics = oracle.count_runs(seq, off, k, m, s, H, shards, seed)
    assert valid == len(active)
    assert runs == len(kv["heads"]) == 3
    assert atomics == int(kv["atomics_with_merging"][0]) == 12
    assert valid * 4 == int(kv["atomics_without_merging"][0])


# ------------------------------------------------------------- special cases ---

def test_m_equals_k_minimizer_is_the_kmer():
    """With m = k there is one window: the shard is hm(k-mer) & (S - 1)."""
    rng = np.random.default_rng(21)
    for k in (5, 16, 31, 32):
        txt = "".join(rng.choice(list("ACGT"), size=k))
        seq, off = _csr_of([txt])
        v = int(txt.translate(str.maketrans("ACGT", "0123")), 4)
        for seed in (0, 77, M64):
            ok, sh, _ = oracle.kmer_info(seq, off, 0, k, k, k, 4, 1 << 30, seed)
            assert ok and sh == oracle.hash_m(v, seed) & ((1 << 30) - 1)


def test_s_equals_k_is_one_smer():
    """With s = k the Findere set is the k-mer itself: its bits are those of
    hs(k-mer) alone."""
    rng = np.random.default_rng(22)
    for k in (7, 31):
        txt = "".join(rng.choice(list("ACGT"), size=k))
        seq, off = _csr_of([txt])
        v = int(txt.translate(str.maketrans("ACGT", "0123")), 4)
        for H in (1, 4, 10):
            ok, _, K = oracle.kmer_info(seq, off, 0, k, 12 if k > 12 else k, k, H, 8, 5)
            assert ok and K == oracle.smer_bits(oracle.hash_s(v, ~5 & M64), H)


def test_validity_closed_form():
    """Sec. IV-F: a k-mer holding an invalid symbol is skipped.  A record of
    length L with one N at i has (L - k + 1) - (#windows holding i) valid
    k-mers; records shorter than k have none; k-mers never span records."""
    rng = np.random.default_rng(23)
    k = 31
    for L, i in [(100, 40), (100, 0), (100, 99), (31, 15), (45, 44), (62, 30)]:
        txt = list("".join(rng.choice(list("ACGT"), size=L)))
        txt[i] = "N"
        seq, off = _csr_of(["".join(txt)])
        valid, _, _ = oracle.count_runs(seq, off, k, 16, 28, 4, 64, 1)
        covering = sum(1 for p in range(L - k + 1) if p <= i <= p + k - 1)
        assert valid == (L - k + 1) - covering
    texts = ["ACGT" * 10, "", "A" * 30, "C" * 31, "acgt" * 8, "G" * 33]
    seq, off = _csr_of(texts)
    valid, _, _ = oracle.count_runs(seq, off, k, 16, 28, 4, 64, 1)
    assert valid == sum(max(0, len(t) - k + 1) for t in texts)


# ------------------------------------------------------------------ invariants ---

def test_filter_invariants():
    """No false negatives; an empty filter answers all-negative; the image is
    independent of record order and of splitting the insert; inserting twice
    changes nothing; image(A u B) = image(A) | image(B)."""
    rng = np.random.default_rng(24)
    args = (31, 16, 28, 4, 4242)
    a = synth.random_records(rng, 30, 20, 800, n_prob=0.003)
    b = synth.random_records(rng, 30, 20, 800, n_prob=0.003)
    S = 512
    Fa = oracle.insert(np.zeros((S, 4), np.uint64), a.seq, a.offsets, *args)
    Fb = oracle.insert(np.zeros((S, 4), np.uint64), b.seq, b.offsets, *args)
    both_seq = np.concatenate([b.seq, a.seq])
    both_off = np.concatenate([b.offsets, b.offsets[-1] + a.offsets[1:]])
    Fab = oracle.insert(np.zeros((S, 4), np.uint64), both_seq, both_off, *args)
    assert np.array_equal(Fab, Fa | Fb)
    again = oracle.insert(Fab.copy(), a.seq, a.offsets, *args)
    assert np.array_equal(again, Fab)
    # no false negatives: every valid k-mer of a answers present
    out = oracle.query(Fa, a.seq, a.offsets, *args)
    valid, _, _ = oracle.count_runs(a.seq, a.offsets, *args[:4], S, args[4])
    assert int(np.unpackbits(out.view(np.uint8)).sum()) == valid
    empty = oracle.query(np.zeros((S, 4), np.uint64), a.seq, a.offsets, *args)
    assert not empty.any()


def test_query_output_layout():
    """Bit g of word g >> 5 (LSB first) answers the k-mer at absolute
    position g; positions without a valid k-mer answer 0."""
    rng = np.random.default_rng(25)
    k = 9
    texts = ["".join(rng.choice(list("ACGT"), size=n)) for n in (40, 5, 70)]
    seq, off = _csr_of(texts)
    F = oracle.insert(np.zeros((4, 4), np.uint64), seq, off, k, 5, 6, 4, 3)
    out = oracle.query(F, seq, off, k, 5, 6, 4, 3)
    expect = set()
    for r in range(3):
        for p in range(int(off[r]), int(off[r + 1]) - k + 1):
            expect.add(p)
    assert _bits_to_set(out, off) == expect


# ------------------------------------------------------- statistical law pins ---

def _random_kmers(rng, n, k):
    return synth.uniform_bases(rng, n * k), synth.csr(np.full(n, k))


def _shard_counts(seq, off, k, m, s, H, S, seed):
    counts = np.zeros(S, dtype=np.int64)
    for r in range(off.size - 1):
        ok, sh, _ = oracle.kmer_info(seq, off, int(off[r]), k, m, s, H, S, seed)
        counts[sh] += ok
    return counts


def _measured_rate(out, off, k):
    starts = off[:-1]
    hits = (out[starts >> 5] >> (starts & 31).astype(np.uint32)) & 1
    return hits.mean(), hits.size


def test_fpr_matches_eq1_single_smer():
    """Eq. 1 per shard: with s = k (one s-mer) and H = 4 (one bit per word),
    an alien k-mer in a shard holding n items is a false positive with
    probability (1 - (1 - 1/64)^n)^4 ~ (1 - e^{-Hn/256})^H.  The mean over the
    alien's uniform shard must match the measured rate."""
    rng = np.random.default_rng(31)
    k = m = s = 31
    H, S, seed, n_ins, n_q = 4, 256, 2024, 10_500, 200_000
    seq, off = _random_kmers(rng, n_ins, k)
    F = oracle.insert(np.zeros((S, 4), np.uint64), seq, off, k, 16, s, H, seed)
    n_sh = _shard_counts(seq, off, k, 16, s, H, S, seed)
    exact = np.mean((1 - (63 / 64) ** n_sh) ** 4)
    eq1 = np.mean((1 - np.exp(-H * n_sh / 256)) ** H)
    assert abs(exact - eq1) / exact < 0.03
    qseq, qoff = _random_kmers(rng, n_q, k)
    out = oracle.query(F, qseq, qoff, k, 16, s, H, seed, nthreads=4)
    rate, n = _measured_rate(out, qoff, k)
    sigma = math.sqrt(exact * (1 - exact) / n)
    assert abs(rate - exact) < 5 * sigma + 0.02 * exact, (rate, exact)
    # the image holds the expected number of distinct bits (insert side)
    pop = np.unpackbits(F.view(np.uint8)).reshape(S, 4, 64).sum(axis=2)
    assert abs(pop.mean() / 64 - np.mean(1 - (63 / 64) ** n_sh)) < 0.01


def test_fpr_matches_eq2_findere():
    """Eq. 2: with z + 1 = k - s + 1 s-mers per k-mer, a random alien k-mer is
    a false positive with probability ~ eps^(z+1), eps the per-s-mer rate of
    its shard.  Given the image, the exact conditional rate of a shard is
    prod_w f_w^((z+1) c_w) (f_w = set fraction of word w, c_w = hashes in word
    w); the measured k-mer rate must match its mean.  A one-base-mutated
    ("almost alien") k-mer instead reverts to ~eps."""
    rng = np.random.default_rng(32)
    k, m, s, H, S, seed = 31, 16, 28, 4, 64, 77
    z1 = k - s + 1
    seq, off = _random_kmers(rng, 1_400, k)
    F = oracle.insert(np.zeros((S, 4), np.uint64), seq, off, k, m, s, H, seed)
    f = np.unpackbits(F.view(np.uint8)).reshape(S, 4, 64).sum(axis=2) / 64.0
    eps = f.prod(axis=1)  # c_w = 1 for H = 4
    pred = np.mean(eps ** z1)
    qseq, qoff = _random_kmers(rng, 200_000, k)
    out = oracle.query(F, qseq, qoff, k, m, s, H, seed, nthreads=4)
    rate, n = _measured_rate(out, qoff, k)
    assert pred * n >= 10
    sigma = math.sqrt(pred * (1 - pred) / n)
    assert abs(rate - pred) < 5 * sigma + 0.03 * pred, (rate, pred)
    # almost-aliens: mutate the last base of inserted k-mers; only the last
    # s-mer changes, so the rate is near eps (>> eps^(z+1)) when the shard stays.
    mut = seq.reshape(-1, k).copy()
    idx = np.searchsorted(synth.ACGT, mut[:, -1])
    mut[:, -1] = synth.ACGT[(idx + rng.integers(1, 4, size=idx.size)) % 4]
    out2 = oracle.query(F, mut.reshape(-1), off, k, m, s, H, seed, nthreads=4)
    rate2, _ = _measured_rate(out2, off, k)
    assert 0.5 * eps.mean() < rate2 < 1.5 * eps.mean()
    assert rate2 > 5 * rate


@pytest.mark.parametrize("m", [12, 16, 21])
def test_minimizer_density_two_over_w_plus_one(m):
    """Sec. II-B1: random minimizers on random sequence have density
    ~ 2/(w+1), i.e. a mean super-k-mer length of (w+1)/2 (8.5 at k=31,
    m=16).  With 2^62 shards a run is a super-k-mer."""
    rng = np.random.default_rng(40 + m)
    k = 31
    w = k - m + 1
    seq = synth.uniform_bases(rng, 400_000)
    off = synth.csr([seq.size])
    valid, runs, _ = oracle.count_runs(seq, off, k, m, 28, 4, 1 << 62, 9)
    mean_len = valid / runs
    assert abs(mean_len - (w + 1) / 2) / ((w + 1) / 2) < 0.03, mean_len


# SplitMix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
# generators", OOPSLA 2014): published first outputs from state 0.
SPLITMIX64_FROM_ZERO = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_salts_are_splitmix64_outputs():
    """The large-H salts are the SplitMix64 sequence (golden-ratio increment)
    made odd: check against the generator's published first outputs."""
    L = oracle.lib()
    for i, v in enumerate(SPLITMIX64_FROM_ZERO):
        assert int(L.orc_salt(i)) == v | 1
        assert brute.salt(i) == v | 1


def test_large_h_positions_are_salted_multiplies():
    """Sec. IV-G fallback for 64/H < 6: position i = top 6 bits of
    hs * salt(i) mod 2^64; recomputed here with Python integers."""
    rng = np.random.default_rng(15)
    salts = [int(oracle.lib().orc_salt(i)) for i in range(32)]
    for H in (11, 12, 16, 32):
        for _ in range(300):
            hs = _u64(rng)
            want = [0, 0, 0, 0]
            for i in range(H):
                pos = ((hs * salts[i]) % (1 << 64)) >> 58
                want[i % 4] |= 1 << pos
            assert oracle.smer_bits(hs, H) == want


@pytest.mark.parametrize("H", [12, 16])
def test_fpr_large_h_matches_popcount_predictor(H):
    """With H > 10 hashes per s-mer (c_w = H/4 per word), an alien single-s-mer
    k-mer is a false positive with probability prod_w f_w^(c_w) given the image
    (f_w = set fraction of word w): the measured rate must match.  A fallback
    that reused one position per word would inflate the rate far above it."""
    rng = np.random.default_rng(60 + H)
    k = s = 31
    S, seed = 256, 99
    seq, off = _random_kmers(rng, 3_000, k)
    F = oracle.insert(np.zeros((S, 4), np.uint64), seq, off, k, 16, s, H, seed)
    f = np.unpackbits(F.view(np.uint8)).reshape(S, 4, 64).sum(axis=2) / 64.0
    pred = np.mean(np.prod(f ** (H // 4), axis=1))
    qseq, qoff = _random_kmers(rng, 200_000, k)
    out = oracle.query(F, qseq, qoff, k, 16, s, H, seed, nthreads=4)
    rate, n = _measured_rate(out, qoff, k)
    assert pred * n >= 10
    sigma = math.sqrt(pred * (1 - pred) / n)
    assert abs(rate - pred) < 5 * sigma + 0.05 * pred, (rate, pred)
