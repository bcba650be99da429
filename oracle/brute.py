"""Pure-Python brute force of SBF insert/query, for tiny inputs only.

Alphabets (Sec. IV-A): "dna" (one base per symbol, radix 4), "protein" (one
letter per symbol, A..Z = 0..25, radix 32) and "dna_triplet" (one codon of
three bases per symbol, read in frame from the record start, radix 64).

TEST INFRASTRUCTURE ONLY.  Written independently of ``sbf_oracle.c`` (Python
strings and integers, no shared code) so that the two can pin each other.

Source: "cuSBF: A Minimizer-Aware Bloom Filter for Genomic Sequence Data on
Modern GPUs", Sec. II-B1 (minimizer = the m-mer of minimum hash among the
k-m+1 windows of a k-mer), Sec. II-B2 (Findere: all k-s+1 s-mers), Sec. IV-B
(four 64-bit words per 256-bit shard, hash i in word i mod 4), Sec. IV-G
(bit-slicing; role-specialised hashes) and Algorithms 1 and 2.  The concrete
hash functions are this library's reading of Sec. IV-G:
hm(x) = t ^ (t >> 32), t = (x ^ seed) * C1;  hs(x): t = (x ^ ~seed) * C1,
t ^= t >> 32, t *= C2, t ^= t >> 29, all modulo 2^64.
"""
from __future__ import annotations

MASK64 = (1 << 64) - 1
C1 = 0x9E3779B97F4A7C15
C2 = 0x6A09E667F3BCC909
_DIGIT = {"A": "0", "C": "1", "G": "2", "T": "3"}


_LETTERS = "ABCDEFGHIJKLMNOPQRSTUVWXYZ"
# radix and input characters per symbol
_SHAPE = {"dna": (4, 1), "protein": (32, 1), "dna_triplet": (64, 3)}


def symbols(text: str, alphabet: str = "dna"):
    """The symbol codes of text (length a multiple of the symbol's width)."""
    _, width = _SHAPE[alphabet]
    if alphabet == "protein":
        return [_LETTERS.index(ch.upper()) for ch in text]
    if alphabet == "dna_triplet":
        return [int("".join(_DIGIT[ch] for ch in text[i:i + 3].upper()), 4)
                for i in range(0, len(text), width)]
    return [int(_DIGIT[ch.upper()]) for ch in text]


def kmer_value(text: str, alphabet: str = "dna") -> int:
    """The symbols as digits of one number, first symbol most significant
    (DNA: base 4 with A0 C1 G2 T3)."""
    radix, _ = _SHAPE[alphabet]
    v = 0
    for c in symbols(text, alphabet):
        v = v * radix + c
    return v


def is_valid(text: str, alphabet: str = "dna") -> bool:
    if alphabet == "protein":
        return all(ch.upper() in _LETTERS and ch.isascii() for ch in text)
    return all(ch in "ACGTacgt" for ch in text)


def hm(x: int, seed: int) -> int:
    t = ((x ^ seed) * C1) & MASK64
    return t ^ (t >> 32)


def hs(x: int, seed: int) -> int:
    t = ((x ^ (~seed & MASK64)) * C1) & MASK64
    t ^= t >> 32
    t = (t * C2) & MASK64
    t ^= t >> 29
    return t


def salt(i: int) -> int:
    """Output i of SplitMix64 started at state 0 (state += C1), made odd."""
    z = ((i + 1) * C1) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    z ^= z >> 31
    return z | 1


def smer_words(h: int, H: int, sectors: int = 0):
    """Bit i: the low 6 bits of slice i while slices are >= 6 bits wide,
    otherwise the top 6 bits of h * salt(i) mod 2^64; in word i mod 4, or,
    with sectors = 1 and H < 4, in the word numbered by the two bits of slice
    i that follow its six position bits."""
    words = [0, 0, 0, 0]
    width = 64 // H
    for i in range(H):
        if width >= 6:
            pos = (h >> (i * width)) & 63
        else:
            pos = ((h * salt(i)) & MASK64) >> 58
        word = i % 4
        if sectors and H < 4:
            word = (h >> (i * width + 6)) & 3
        words[word] |= 1 << pos
    return words


def kmer(text: str, k: int, m: int, s: int, H: int, num_shards: int, seed: int,
         alphabet: str = "dna", sectors: int = 0):
    """(shard, words) of one valid k-mer given as its k symbols' characters."""
    _, cw = _SHAPE[alphabet]
    minimizer = min(hm(kmer_value(text[cw * i:cw * (i + m)], alphabet), seed)
                    for i in range(k - m + 1))
    shard = minimizer % num_shards
    words = [0, 0, 0, 0]
    for j in range(k - s + 1):
        for w, bits in enumerate(smer_words(hs(kmer_value(text[cw * j:cw * (j + s)], alphabet), seed), H, sectors)):
            words[w] |= bits
    return shard, words


def records_of(seq: bytes, offsets):
    return [(int(offsets[r]), seq[int(offsets[r]):int(offsets[r + 1])].decode("latin-1"))
            for r in range(len(offsets) - 1)]


def kmers_of(rec: str, k: int, alphabet: str = "dna"):
    """(offset in the record, characters) of every k-mer of one record: one
    per symbol, symbols read in frame from the record's start."""
    _, cw = _SHAPE[alphabet]
    for p in range(0, len(rec) - cw * k + 1, cw):
        yield p, rec[p:p + cw * k]


def insert(seq: bytes, offsets, k, m, s, H, num_shards, seed, filt=None, alphabet: str = "dna",
           sectors: int = 0):
    """Return {shard: [w0, w1, w2, w3]} with every valid k-mer inserted."""
    filt = {} if filt is None else filt
    for _, rec in records_of(seq, offsets):
        for p, text in kmers_of(rec, k, alphabet):
            if not is_valid(text, alphabet):
                continue
            shard, words = kmer(text, k, m, s, H, num_shards, seed, alphabet, sectors)
            cur = filt.setdefault(shard, [0, 0, 0, 0])
            for w in range(4):
                cur[w] |= words[w]
    return filt


def query(filt, seq: bytes, offsets, k, m, s, H, num_shards, seed, alphabet: str = "dna",
          sectors: int = 0):
    """Return the set of absolute positions whose k-mer answers present."""
    hits = set()
    for start, rec in records_of(seq, offsets):
        for p, text in kmers_of(rec, k, alphabet):
            if not is_valid(text, alphabet):
                continue
            shard, words = kmer(text, k, m, s, H, num_shards, seed, alphabet, sectors)
            have = filt.get(shard, [0, 0, 0, 0])
            if all((words[w] & ~have[w]) == 0 for w in range(4)):
                hits.add(start + p)
    return hits
