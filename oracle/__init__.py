"""CPU oracle for Super Bloom filter insert/query over DNA, protein and DNA-triplet sequences.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the product library never does.  It shares
no code with the CUDA path.

Two independent implementations live here:

* ``sbf_oracle.c`` (wrapped below): the plain C definition, every k-mer
  recomputed from scratch, optionally split over threads;
* ``brute.py``: a pure-Python brute force over strings for tiny inputs.

Source: "cuSBF: A Minimizer-Aware Bloom Filter for Genomic Sequence Data on
Modern GPUs", Sec. II-B (minimizers, Findere, Eq. 2), Sec. IV-B..IV-G and
Algorithms 1 and 2.  The hash functions and the other readings the paper leaves
open are stated in the header of ``sbf_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sbf_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libsbf_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (plain -O2, no target-specific flags)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
                           "-Wall", "-Wextra", "-o", tmp, _SRC])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            u64, i64, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_int
            vp = ctypes.c_void_p
            L.orc_const_c1.restype = u64
            L.orc_const_c2.restype = u64
            L.orc_base_code.argtypes = [ctypes.c_uint8]
            L.orc_base_code.restype = i32
            L.orc_pack.argtypes = [ctypes.c_char_p, i32]
            L.orc_pack.restype = u64
            L.orc_hash_m.argtypes = [u64, u64]
            L.orc_hash_m.restype = u64
            L.orc_hash_s.argtypes = [u64, u64]
            L.orc_hash_s.restype = u64
            L.orc_salt.argtypes = [i32]
            L.orc_salt.restype = u64
            L.orc_smer_bits.argtypes = [u64, i32, vp]
            L.orc_smer_bits.restype = None
            L.orc_smer_bits_sectors.argtypes = [u64, i32, i32, vp]
            L.orc_smer_bits_sectors.restype = None
            L.orc_symbol_bits.argtypes = [i32]
            L.orc_symbol_bits.restype = i32
            L.orc_symbol_bytes.argtypes = [i32]
            L.orc_symbol_bytes.restype = i32
            L.orc_symbol_code.argtypes = [i32, ctypes.c_char_p]
            L.orc_symbol_code.restype = i32
            L.orc_pack_symbols.argtypes = [i32, ctypes.c_char_p, i32]
            L.orc_pack_symbols.restype = u64
            L.orc_insert.argtypes = [vp, vp, vp, i64, i32, i32, i32, i32, u64, u64, i32, i32, i32]
            L.orc_insert.restype = i32
            L.orc_query.argtypes = [vp, vp, vp, i64, i32, i32, i32, i32, u64, u64, i32, i32, vp, i32]
            L.orc_query.restype = i32
            L.orc_kmer_info.argtypes = [vp, vp, i64, i64, i32, i32, i32, i32, u64, u64, i32, i32, vp, vp]
            L.orc_kmer_info.restype = i32
            L.orc_count_runs.argtypes = [vp, vp, i64, i32, i32, i32, i32, u64, u64, i32, i32, vp, vp, vp]
            L.orc_count_runs.restype = i32
            L.orc_kmer_batch.argtypes = [vp, vp, i64, vp, i64, i32, i32, i32, i32, u64, u64, i32, i32,
                                         vp, vp, vp]
            L.orc_kmer_batch.restype = i32
            L.orc_kmer_rows.argtypes = [vp, vp, i64, i32, i32, i32, i32, u64, u64, i32, i32, vp, vp, vp]
            L.orc_kmer_rows.restype = i32
            _lib = L
    return _lib


# Sec. IV-A alphabets
DNA, PROTEIN, DNA_TRIPLET = 0, 1, 2
_ALPHABETS = {"dna": DNA, "protein": PROTEIN, "dna_triplet": DNA_TRIPLET, "triplet": DNA_TRIPLET}


def alphabet_id(alphabet) -> int:
    """0 (DNA), 1 (protein) or 2 (DNA triplet), from a name or an id."""
    if isinstance(alphabet, str):
        return _ALPHABETS[alphabet.lower()]
    a = int(alphabet)
    if a not in (DNA, PROTEIN, DNA_TRIPLET):
        raise ValueError(f"unknown alphabet {alphabet!r}")
    return a


def num_shards_for(num_bits: int) -> int:
    """Shard count for a filter of num_bits bits: ceil(num_bits / 256) rounded
    up to a power of two (Sec. IV-B: "rounded up to the next power of two")."""
    if num_bits < 1:
        raise ValueError("num_bits must be >= 1")
    shards = -(-num_bits // 256)
    p = 1
    while p < shards:
        p <<= 1
    return p


def _u8(seq) -> np.ndarray:
    if isinstance(seq, (bytes, bytearray)):
        seq = np.frombuffer(bytes(seq), dtype=np.uint8)
    a = np.ascontiguousarray(seq, dtype=np.uint8)
    if a.size == 0:  # keep a valid pointer for empty inputs
        a = np.zeros(1, dtype=np.uint8)
    return a


def _i64(off) -> np.ndarray:
    return np.ascontiguousarray(off, dtype=np.int64)


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def insert(filter_words: np.ndarray, seq, offsets, k, m, s, H, seed, nthreads=1,
           alphabet=DNA, sectors=0) -> np.ndarray:
    """OR every valid k-mer of every record into filter_words (uint64[S, 4]),
    in place, and return it.  sectors = 1: hash-chosen words for H < 4 (see
    smer_bits)."""
    F = filter_words
    assert F.dtype == np.uint64 and F.ndim == 2 and F.shape[1] == 4 and F.flags.c_contiguous
    a, o = _u8(seq), _i64(offsets)
    rc = lib().orc_insert(_ptr(F), _ptr(a), _ptr(o), o.size - 1, k, m, s, H,
                          F.shape[0], seed & (2**64 - 1), alphabet_id(alphabet), int(sectors), nthreads)
    if rc != 0:
        raise ValueError("orc_insert rejected its arguments")
    return F


def new_filter(num_bits: int) -> np.ndarray:
    return np.zeros((num_shards_for(num_bits), 4), dtype=np.uint64)


def query(filter_words: np.ndarray, seq, offsets, k, m, s, H, seed, nthreads=1,
          alphabet=DNA, sectors=0) -> np.ndarray:
    """Answer bits for every absolute position of [offsets[0], offsets[-1]).

    Returns uint32[(offsets[-1] + 31) // 32]; words below offsets[0] >> 5 stay
    zero, bit g (word g >> 5, bit g & 31) is the answer for the k-mer at g."""
    F = filter_words
    assert F.dtype == np.uint64 and F.ndim == 2 and F.shape[1] == 4 and F.flags.c_contiguous
    a, o = _u8(seq), _i64(offsets)
    out = np.zeros(max(1, (int(o[-1]) + 31) // 32), dtype=np.uint32)
    rc = lib().orc_query(_ptr(F), _ptr(a), _ptr(o), o.size - 1, k, m, s, H,
                         F.shape[0], seed & (2**64 - 1), alphabet_id(alphabet), int(sectors), _ptr(out),
                         nthreads)
    if rc != 0:
        raise ValueError("orc_query rejected its arguments")
    return out


def kmer_info(seq, offsets, g, k, m, s, H, num_shards, seed, alphabet=DNA, sectors=0):
    """(valid, shard, K[4]) for the k-mer at absolute position g."""
    a, o = _u8(seq), _i64(offsets)
    shard = np.zeros(1, dtype=np.uint64)
    K = np.zeros(4, dtype=np.uint64)
    rc = lib().orc_kmer_info(_ptr(a), _ptr(o), o.size - 1, int(g), k, m, s, H,
                             num_shards, seed & (2**64 - 1), alphabet_id(alphabet), int(sectors), _ptr(shard),
                             _ptr(K))
    if rc < 0:
        raise ValueError("orc_kmer_info rejected its arguments")
    return bool(rc), int(shard[0]), [int(x) for x in K]


def count_runs(seq, offsets, k, m, s, H, num_shards, seed, alphabet=DNA, sectors=0):
    """(valid k-mers, runs, atomics): runs are maximal stretches of consecutive
    valid k-mers of one record sharing a shard (Fig. 3); atomics counts the
    non-zero words over all runs."""
    a, o = _u8(seq), _i64(offsets)
    res = np.zeros(3, dtype=np.int64)
    rc = lib().orc_count_runs(_ptr(a), _ptr(o), o.size - 1, k, m, s, H, num_shards,
                              seed & (2**64 - 1), alphabet_id(alphabet), int(sectors), _ptr(res[0:]), _ptr(res[1:]),
                              _ptr(res[2:]))
    if rc != 0:
        raise ValueError("orc_count_runs rejected its arguments")
    return int(res[0]), int(res[1]), int(res[2])


def hash_m(x: int, seed_m: int) -> int:
    return int(lib().orc_hash_m(x & (2**64 - 1), seed_m & (2**64 - 1)))


def hash_s(x: int, seed_s: int) -> int:
    return int(lib().orc_hash_s(x & (2**64 - 1), seed_s & (2**64 - 1)))


def pack(t_mer: bytes) -> int:
    return int(lib().orc_pack(bytes(t_mer), len(t_mer)))


def pack_symbols(t_mer: bytes, alphabet) -> int:
    """Packed value of a t-mer given as its bytes (3 per symbol for triplets)."""
    a = alphabet_id(alphabet)
    t = len(t_mer) // int(lib().orc_symbol_bytes(a))
    return int(lib().orc_pack_symbols(a, bytes(t_mer), t))


def symbol_code(sym: bytes, alphabet) -> int:
    return int(lib().orc_symbol_code(alphabet_id(alphabet), bytes(sym)))


def symbol_bits(alphabet) -> int:
    return int(lib().orc_symbol_bits(alphabet_id(alphabet)))


def smer_bits(hs: int, H: int, sectors: int = 0):
    """The four word masks of one s-mer hash (Sec. IV-B, IV-G); sectors = 1
    puts hash i of an H < 4 filter in the word given by the two slice bits
    above its position bits instead of word i mod 4."""
    w = np.zeros(4, dtype=np.uint64)
    lib().orc_smer_bits_sectors(hs & (2**64 - 1), H, int(sectors), _ptr(w))
    return [int(x) for x in w]


def constants():
    L = lib()
    return int(L.orc_const_c1()), int(L.orc_const_c2())


def kmer_batch(seq, offsets, positions, k, m, s, H, num_shards, seed, alphabet=DNA, sectors=0):
    """(valid[bool], shard[uint64], K[uint64, 4]) for each absolute position."""
    a, o = _u8(seq), _i64(offsets)
    pos = np.ascontiguousarray(positions, dtype=np.int64)
    valid = np.zeros(pos.size, dtype=np.uint8)
    shard = np.zeros(pos.size, dtype=np.uint64)
    K = np.zeros((pos.size, 4), dtype=np.uint64)
    if pos.size:
        rc = lib().orc_kmer_batch(_ptr(a), _ptr(o), o.size - 1, _ptr(pos), pos.size, k, m, s, H,
                                  num_shards, seed & (2**64 - 1), alphabet_id(alphabet), int(sectors), _ptr(valid),
                                  _ptr(shard), _ptr(K))
        if rc != 0:
            raise ValueError("orc_kmer_batch rejected its arguments")
    return valid.astype(bool), shard, K


def query_sampled(shard_words, seq, offsets, positions, k, m, s, H, num_shards, seed, alphabet=DNA, sectors=0):
    """Answers for selected absolute positions only, for filters too large to
    copy whole.  shard_words(uint64 array of shards) -> uint64[len, 4] supplies
    the image words of the requested shards.  Each answer follows Algorithm 2:
    present iff the k-mer is valid and every bit of its s-mers is set in its
    shard."""
    valid, shard, K = kmer_batch(seq, offsets, positions, k, m, s, H, num_shards, seed, alphabet, sectors)
    out = np.zeros(valid.size, dtype=bool)
    if valid.any():
        F = np.asarray(shard_words(shard[valid]), dtype=np.uint64).reshape(-1, 4)
        out[valid] = ((K[valid] & ~F) == 0).all(axis=1)
    return out


def insert_sparse(seq, offsets, k, m, s, H, num_shards, seed, alphabet=DNA, sectors=0):
    """The image a full insert produces, as (sorted non-zero shard indices,
    uint64[len, 4] words), without allocating num_shards rows: every valid
    k-mer's (shard, K) from scratch, then an OR per shard (a sort and a
    segmented OR-reduce)."""
    a, o = _u8(seq), _i64(offsets)
    total = int(np.maximum(np.diff(o), 0).sum())
    shard = np.zeros(max(total, 1), dtype=np.uint64)
    K = np.zeros((max(total, 1), 4), dtype=np.uint64)
    cnt = np.zeros(1, dtype=np.int64)
    rc = lib().orc_kmer_rows(_ptr(a), _ptr(o), o.size - 1, k, m, s, H, num_shards,
                             seed & (2**64 - 1), alphabet_id(alphabet), int(sectors), _ptr(shard), _ptr(K),
                             _ptr(cnt))
    if rc != 0:
        raise ValueError("orc_kmer_rows rejected its arguments")
    c = int(cnt[0])
    shard, K = shard[:c], K[:c]
    order = np.argsort(shard, kind="stable")
    shard, K = shard[order], K[order]
    if c == 0:
        return shard, K
    starts = np.flatnonzero(np.concatenate([[True], shard[1:] != shard[:-1]]))
    words = np.bitwise_or.reduceat(K, starts, axis=0)
    keep = words.any(axis=1)
    return shard[starts][keep], words[keep]
