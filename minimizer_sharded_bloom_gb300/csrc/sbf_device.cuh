// sbf_device.cuh -- device-side definitions shared by the SBF kernels.
//
// The hash functions, base encoding and bit addressing of the Super Bloom
// filter as this library fixes them ("cuSBF: A Minimizer-Aware Bloom Filter
// for Genomic Sequence Data on Modern GPUs", Sec. IV-B, IV-C, IV-G; the
// concrete constants and shifts are this library's reading of Sec. IV-G's
// "single multiplicative mix" and "stronger mix with an additional xorshift").
#pragma once

#include <cstdint>

namespace sbf {

constexpr uint64_t kC1 = 0x9E3779B97F4A7C15ull;  // floor(2^64 / golden ratio)
constexpr uint64_t kC2 = 0x6A09E667F3BCC909ull;  // floor((sqrt(2) - 1) * 2^64) | 1
constexpr int kStatusBadOffsets = 1;
// Sec. IV-A alphabets (the values of SBF_ALPHABET_* in sbf.h)
constexpr int kAlphabetDNA = 0, kAlphabetProtein = 1, kAlphabetTriplet = 2;
constexpr int kStatusTimeout = 2;  // a bounded device wait gave up

// Everything a kernel launch needs; passed by value (kernel parameter space).
struct LaunchArgs {
    const uint8_t *seq;       // device bytes, readable on [offsets[0], offsets[n])
    const int64_t *offsets;   // device CSR offsets, n + 1 entries
    int64_t n;                // number of records
    uint64_t *words;          // filter: num_shards * 4 words
    uint32_t *out;            // query answer bits (absolute positions)
    int *status;              // sticky device status word
    uint64_t shard_mask;      // num_shards - 1
    uint64_t seed;            // minimizer seed; the s-mer seed is ~seed
    int k, m, s, H;
    int device_seq;           // 1: seq is device memory (tile bytes may use TMA bulk copies)
    int64_t rec_len;          // > 0: a dense batch, record r = seq[r*rec_len, (r+1)*rec_len)
                              // and `offsets` is unused; 0: CSR offsets
    const int *nonuniform;    // CSR queries that may run as dense batches: nonzero when the
                              // offsets check saw records of different lengths (else nullptr)
    int64_t out_words_end;    // query: answer words at or past this index are not written
                              // (a chunk of a larger batch cut inside a record); else INT64_MAX
    int sectors;              // 1: hash-chosen sectors for H < 4 (sector_word); 0: word i mod 4
    int wait_test;            // failure-detection test: > 0 = before any work, one thread waits
                              // on an mbarrier that nothing completes, giving up after
                              // wait_test polls; the kernel then reports the timeout and
                              // returns (no copy is in flight).  0 in every normal launch.
};

// Minimizer hash (Sec. IV-G, minimizer role): one multiplicative mix, then an
// xor-fold of the high half into the low half, whose bits pick the shard.
__device__ __forceinline__ uint64_t hash_minimizer(uint64_t x, uint64_t seed_m) {
    const uint64_t t = (x ^ seed_m) * kC1;
    return t ^ (t >> 32);
}

// s-mer hash (Sec. IV-G, Bloom-bit role): stronger mix, extra xorshift.
__device__ __forceinline__ uint64_t hash_smer(uint64_t x, uint64_t seed_s) {
    uint64_t t = (x ^ seed_s) * kC1;
    t ^= t >> 32;
    t *= kC2;
    t ^= t >> 29;
    return t;
}

// 2-bit code of one byte, or -1: A/a 0, C/c 1, G/g 2, T/t 3 (Sec. IV-C).
// Bits 1 and 2 of the ASCII letters give A0 C1 G3 T2; xor-ing bit 1 into bit 0
// of that pair gives A0 C1 G2 T3.  Validity: the byte's top bits are 01x and its
// low five bits are 1 (A), 3 (C), 7 (G) or 20 (T).
__device__ __forceinline__ int base_code(uint32_t c) {
    const bool ok = ((c & 0xC0u) == 0x40u) && ((0x0010008Au >> (c & 31u)) & 1u);
    const int code = (int)(((c >> 1) ^ (c >> 2)) & 3u);
    return ok ? code : -1;
}

// Protein symbol code of one byte (Sec. IV-A: 26 letters, 5 bits): A..Z and
// a..z -> 0..25; any other byte -> a value >= 26 (0xFF).
__device__ __forceinline__ uint32_t protein_code(uint32_t c) {
    const uint32_t u = (c | 0x20u) - (uint32_t)'a';
    return u < 26u ? u : 0xFFu;
}

// Salt of hash index i for H > 10 (Sec. IV-G: "per-hash-index golden-ratio-
// derived salt"): output i of SplitMix64 from state 0, whose state advances by
// the golden-ratio constant, made odd.
__host__ __device__ constexpr uint64_t salt_of(int i) {
    uint64_t z = (uint64_t)(i + 1) * kC1;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    z ^= z >> 31;
    return z | 1ull;
}
constexpr int kMaxH = 32;
__constant__ const uint64_t kSalt[kMaxH] = {
    salt_of(0),  salt_of(1),  salt_of(2),  salt_of(3),  salt_of(4),  salt_of(5),  salt_of(6),  salt_of(7),
    salt_of(8),  salt_of(9),  salt_of(10), salt_of(11), salt_of(12), salt_of(13), salt_of(14), salt_of(15),
    salt_of(16), salt_of(17), salt_of(18), salt_of(19), salt_of(20), salt_of(21), salt_of(22), salt_of(23),
    salt_of(24), salt_of(25), salt_of(26), salt_of(27), salt_of(28), salt_of(29), salt_of(30), salt_of(31)};

// The word of hash i with hash-chosen sectors (filters created with
// SBF_FLAG_HASHED_SECTORS, H < 4 only): the two bits of slice i (width W =
// floor(64/H) >= 21) just above its six position bits.  The paper's layout
// (Sec. IV-B) uses word i mod 4, which leaves words H..3 empty when H < 4.
__device__ __forceinline__ uint32_t sector_word(uint64_t hs, int i, int W) {
    return (uint32_t)(hs >> (i * W + 6)) & 3u;
}

// x into the word K[w] of a runtime w, without indexing K dynamically (K
// stays in registers).
__device__ __forceinline__ void or_into_word(uint64_t K[4], uint32_t w, uint64_t x) {
#pragma unroll
    for (int q = 0; q < 4; ++q) K[q] |= w == (uint32_t)q ? x : 0ull;
}

// OR the H bits of one s-mer hash into four word masks (Sec. IV-B: hash i ->
// word i mod 4; with `sectors` and H < 4, sector_word).  Sec. IV-G:
// bit-slicing with slice width floor(64/H) while it is at least 6 bits;
// beyond, the top 6 bits of hs * salt(i).
// (Loops unrolled to their bounds so that K stays in registers.)
__device__ __forceinline__ void smer_bits_runtime(uint64_t hs, int H, uint64_t K[4], int sectors = 0) {
    const int W = 64 / H;
    if (sectors && H < 4) {
#pragma unroll
        for (int i = 0; i < 3; ++i)
            if (i < H) or_into_word(K, sector_word(hs, i, W), 1ull << ((hs >> (i * W)) & 63u));
    } else if (W >= 6) {
#pragma unroll
        for (int i = 0; i < 10; ++i)
            if (i < H) K[i & 3] |= 1ull << ((hs >> (i * W)) & 63u);
    } else {
        // groups of four hashes: word q of the group is constant per unrolled step
#pragma unroll 1
        for (int i0 = 0; i0 < H; i0 += 4)
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (i0 + q < H) K[q] |= 1ull << ((hs * kSalt[i0 + q]) >> 58);
    }
}

__device__ __forceinline__ uint64_t low_mask(int symbols) {
    return symbols >= 32 ? ~0ull : ((1ull << (2 * symbols)) - 1ull);
}

// First record boundary r in [0, n] with offsets[r] > x (n + 1 if none), by
// one warp: an interpolation probe of 32 consecutive boundaries around the
// guess for evenly sized records, then 32-way searches (one load round each).
__device__ __forceinline__ int64_t warp_find_boundary(const int64_t *off, int64_t n, int64_t x, int64_t lo,
                                                      int64_t hi, int lane) {
    int64_t r_lo = 0, r_hi = n + 1;  // offsets[r] <= x for r < r_lo; > x for r >= r_hi
    {
        const double frac = hi > lo ? (double)(x - lo) / (double)(hi - lo) : 0.0;
        int64_t g = (int64_t)(frac * (double)n);
        g = g < 0 ? 0 : (g > n ? n : g);
        int64_t p = g - 15 + lane;
        p = p < 0 ? 0 : (p > n ? n : p);
        const unsigned b = __ballot_sync(0xffffffffu, off[p] > x);
        const int64_t p31 = __shfl_sync(0xffffffffu, p, 31);
        if (b == 0) {
            r_lo = p31 + 1;
        } else {
            const int f = __ffs(b) - 1;
            const int64_t pf = __shfl_sync(0xffffffffu, p, f);
            const int64_t pf1 = __shfl_sync(0xffffffffu, p, f > 0 ? f - 1 : 0);
            r_hi = pf;
            if (f > 0) r_lo = pf1 + 1;
        }
    }
    while (r_lo < r_hi) {
        const int64_t span = r_hi - r_lo;
        const int64_t p = r_lo + (span * lane) / 32;
        const unsigned b = __ballot_sync(0xffffffffu, off[p] > x);
        if (b == 0) {
            r_lo = __shfl_sync(0xffffffffu, p, 31) + 1;
        } else {
            const int f = __ffs(b) - 1;
            const int64_t pf = __shfl_sync(0xffffffffu, p, f);
            const int64_t pf1 = __shfl_sync(0xffffffffu, p, f > 0 ? f - 1 : 0);
            r_hi = pf;
            if (f > 0) r_lo = pf1 + 1;
        }
    }
    return r_lo;
}

}  // namespace sbf
