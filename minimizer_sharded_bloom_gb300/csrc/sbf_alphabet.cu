// sbf_alphabet.cu -- SBF insert/query kernels for the protein and DNA-triplet
// alphabets ("cuSBF", Sec. IV-A: proteins, 26 symbols in 5 bits; DNA triplets,
// 64 symbols in 6 bits, each symbol read from several input bytes).  Runtime
// k, m, s, H with k * bits <= 64 (Sec. IV-C: one k-mer packs into one 64-bit
// word, so protein k <= 12 and triplet k <= 10).
//
// Symbols.  Protein: the 26 letters, either case, A..Z = 0..25; every other
// byte is invalid.  Triplet: a codon of three bases read in frame from the
// start of its record, code 16*c0 + 4*c1 + c2 (2-bit base codes, first base
// most significant); a codon holding an invalid base is invalid.  A k-mer
// starts on a symbol boundary of its record and covers B*k bytes (B = 1 or
// 3); its query answer goes to the bit of its first byte, every other bit of
// the answer range is 0.
//
// Work layout (the paper's shared tile preparation, Sec. IV-C, with the
// per-position hashes kept in shared memory instead of recomputed per
// k-mer):
//  * a block owns a tile of TB = 256*B consecutive bytes starting at a
//    multiple of 32, and walks the tiles grid-stride;
//  * warp 0 locates the record boundaries that fall in the tile (plus the
//    k-mer overhang) and marks them in a bitmap; the other warps load the
//    tile's bytes and turn them into symbol codes;
//  * the tile is covered in B passes; in pass p lane t owns byte B*t + p, so
//    within one record the lanes of a pass that start a symbol hold
//    consecutive k-mers (for triplets, one pass of three carries each
//    record's frame);
//  * per pass, every position computes its m-mer hash and its s-mer's four
//    word masks once (shared memory), then every k-mer takes the minimum over
//    its w = k-m+1 m-mer hashes (Algorithm 1) and ORs its k-s+1 s-mer masks;
//  * insert: lanes holding consecutive valid k-mers with one shard are
//    merged by a segmented OR over the warp (the paper's super-k-mer runs,
//    Fig. 3) and the head lane issues one atomicOr per non-zero word;
//    query: each valid k-mer tests its shard's four words (Algorithm 2) and
//    the answers are assembled in shared memory and stored coalesced.
#include "sbf_device.cuh"
#include "sbf_kernels.h"

namespace sbf {
namespace {

template <int ALPHA>
struct AlphaCfg;
template <>
struct AlphaCfg<kAlphabetProtein> {
    static constexpr int B = 1, BITS = 5, KMAX = 12;
};
template <>
struct AlphaCfg<kAlphabetTriplet> {
    static constexpr int B = 3, BITS = 6, KMAX = 10;
};

constexpr int kAlphaThreads = 256;
constexpr uint32_t kBadCode = 0xFFu;

template <int ALPHA>
struct AlphaTile {
    static constexpr int B = AlphaCfg<ALPHA>::B, BITS = AlphaCfg<ALPHA>::BITS, KMAX = AlphaCfg<ALPHA>::KMAX;
    static constexpr int NT = kAlphaThreads;
    static constexpr int TB = NT * B;                  // tile bytes (k-mer start positions)
    static constexpr int CODES = TB + B * (KMAX - 1);  // symbol codes, one per start byte
    static constexpr int RAW = CODES + B - 1;          // bytes the codes read
    static constexpr int HN = NT + KMAX - 1;           // hash slots per pass
    static constexpr int SPAN = TB + B * KMAX;         // boundary bitmap reach
    static constexpr int BW = (SPAN + 31) / 32 + 1;    // bitmap words (+1: two-word reads)
    static constexpr int OUTW = TB / 32;               // answer words per tile
    static_assert(TB % 32 == 0, "tiles must cover whole answer words");
    static_assert(B * KMAX - 1 < 32, "a k-mer's inner boundaries must fit one 32-bit window");
};

template <int ALPHA>
struct AlphaSmem {
    using T = AlphaTile<ALPHA>;
    uint64_t hm[T::HN];      // m-mer hash at slot u (byte B*u + pass)
    uint64_t sk[4][T::HN];   // s-mer word masks at slot u
    uint32_t starts[T::BW];  // bit i: a record boundary at byte t0 + i (i >= 1)
    uint32_t ans[T::OUTW];
    int64_t prev_start;      // last boundary <= t0, or kNoStart
    uint8_t mok[T::HN];      // m-mer at slot u is valid
    uint8_t raw[ALPHA == kAlphabetTriplet ? T::RAW : 1];
    uint8_t code[T::CODES];
};

constexpr int64_t kNoStart = INT64_MIN;

__device__ __forceinline__ uint32_t protein_code(uint32_t c) {
    const uint32_t u = (c | 0x20u) - (uint32_t)'a';  // A..Z and a..z -> 0..25
    return u < 26u ? u : kBadCode;
}

__device__ __forceinline__ uint32_t codon_code(uint32_t c0, uint32_t c1, uint32_t c2) {
    const int a = base_code(c0), b = base_code(c1), c = base_code(c2);
    return (a | b | c) < 0 ? kBadCode : (uint32_t)(a * 16 + b * 4 + c);
}

// Any bit in [from, from + len) of the bitmap, 0 <= len <= 31.
__device__ __forceinline__ bool any_bit(const uint32_t *bm, int from, int len) {
    const int w = from >> 5;
    const uint64_t two = (uint64_t)bm[w] | ((uint64_t)bm[w + 1] << 32);
    return ((two >> (from & 31)) & ((1ull << len) - 1ull)) != 0;
}

// Highest boundary at or below tile byte j (absolute), else prev.
__device__ __forceinline__ int64_t start_at_or_below(const uint32_t *bm, int j, int64_t t0, int64_t prev) {
    int w = j >> 5;
    uint32_t b = bm[w] & (0xFFFFFFFFu >> (31 - (j & 31)));
    while (!b && w > 0) b = bm[--w];
    return b ? t0 + 32 * w + 31 - __clz(b) : prev;
}

template <int ALPHA, bool kQuery>
__global__ void __launch_bounds__(kAlphaThreads) alphabet_kernel(LaunchArgs a) {
    using T = AlphaTile<ALPHA>;
    constexpr int B = T::B, BITS = T::BITS, KMAX = T::KMAX, NT = T::NT, TB = T::TB;
    __shared__ AlphaSmem<ALPHA> sm;
    if (*reinterpret_cast<volatile int *>(a.status) & kStatusBadOffsets) return;
    const int64_t lo = a.offsets[0], hi = a.offsets[a.n];
    if (hi <= lo) return;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int k = a.k, m = a.m, s = a.s, w = k - m + 1, z1 = k - s + 1;
    const int kspan = B * k;
    const uint64_t seed_s = ~a.seed;
    const int n_words = a.H < 4 ? a.H : 4;
    const int64_t base = lo & ~int64_t(31);
    const int64_t n_tiles = (hi - base + TB - 1) / TB;

    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int64_t t0 = base + tile * TB;
        // ---- record boundaries (warp 0) and symbol codes (warps 1..7)
        for (int i = t; i < T::BW; i += NT) sm.starts[i] = 0u;
        if (kQuery)
            for (int i = t; i < T::OUTW; i += NT) sm.ans[i] = 0u;
        __syncthreads();
        if (warp == 0) {
            const int64_t r0 = warp_find_boundary(a.offsets, a.n, t0, lo, hi, lane);
            if (lane == 0) sm.prev_start = r0 >= 1 ? a.offsets[r0 - 1] : kNoStart;
            const int64_t lim = t0 + T::SPAN;
            // boundaries r0, r0+1, ... are > t0 and non-decreasing: stop once
            // the warp's last one reaches lim (or runs past offsets[n])
            for (int64_t rb = r0; rb <= a.n; rb += 32) {
                const int64_t r = rb + lane;
                const int64_t p = r <= a.n ? a.offsets[r] : lim;
                if (p < lim) atomicOr(&sm.starts[(p - t0) >> 5], 1u << ((p - t0) & 31));
                if (__shfl_sync(0xffffffffu, p, 31) >= lim) break;
            }
        } else {
            if constexpr (B == 1) {
                for (int u = t - 32; u < T::CODES; u += NT - 32) {
                    const int64_t g = t0 + u;
                    sm.code[u] = (uint8_t)(g >= lo && g < hi ? protein_code(a.seq[g]) : kBadCode);
                }
            } else {
                for (int u = t - 32; u < T::RAW; u += NT - 32) {
                    const int64_t g = t0 + u;
                    sm.raw[u] = g >= lo && g < hi ? a.seq[g] : (uint8_t)0;
                }
            }
        }
        __syncthreads();
        if constexpr (B > 1) {
            for (int u = t; u < T::CODES; u += NT)
                sm.code[u] = (uint8_t)codon_code(sm.raw[u], sm.raw[u + 1], sm.raw[u + 2]);
            __syncthreads();
        }

        for (int pass = 0; pass < B; ++pass) {
            // ---- this lane's k-mer: inside [lo, hi), in frame, inside one record
            const int j = B * t + pass;
            const int64_t g = t0 + j;
            bool in_frame = g >= lo && g < hi;
            if constexpr (B > 1) {
                if (in_frame) {
                    const int64_t rs = start_at_or_below(sm.starts, j, t0, sm.prev_start);
                    in_frame = rs != kNoStart && (g - rs) % B == 0;
                }
                if (!__syncthreads_or(in_frame)) continue;
            }
            const bool placed = in_frame && g + kspan <= hi && !any_bit(sm.starts, j + 1, kspan - 1);

            // ---- per-slot hashes: slot u covers byte B*u + pass
            auto fill = [&](int u) {
                const int pos = B * u + pass;
                if (u < NT + w - 1) {
                    uint64_t v = 0;
                    uint32_t bad = 0;
#pragma unroll
                    for (int i = 0; i < KMAX; ++i)
                        if (i < m) {
                            const uint32_t c = sm.code[pos + B * i];
                            bad |= c;
                            v = (v << BITS) | c;
                        }
                    sm.hm[u] = hash_minimizer(v, a.seed);
                    sm.mok[u] = (uint8_t)((bad & 0x80u) == 0);
                }
                if (u < NT + z1 - 1) {
                    uint64_t v = 0;
                    uint32_t bad = 0;
#pragma unroll
                    for (int i = 0; i < KMAX; ++i)
                        if (i < s) {
                            const uint32_t c = sm.code[pos + B * i];
                            bad |= c;
                            v = (v << BITS) | c;
                        }
                    uint64_t K[4] = {0, 0, 0, 0};
                    smer_bits_runtime(hash_smer(v, seed_s), a.H, K);
                    const bool ok = (bad & 0x80u) == 0;
#pragma unroll
                    for (int q = 0; q < 4; ++q) sm.sk[q][u] = ok ? K[q] : 0ull;
                }
            };
            // an out-of-frame slot is never read by a placed k-mer of this pass
            if (B == 1 || in_frame) fill(t);
            if (t < KMAX - 1) fill(NT + t);
            __syncthreads();

            // ---- this lane's k-mer from the slots
            bool valid = placed;
            uint64_t shard = 0, K[4] = {0, 0, 0, 0};
            if (placed) {
                uint64_t mu = ~0ull;
#pragma unroll
                for (int i = 0; i < KMAX; ++i)
                    if (i < w) {
                        valid &= sm.mok[t + i] != 0;
                        const uint64_t h = sm.hm[t + i];
                        mu = h < mu ? h : mu;
                    }
                shard = mu & a.shard_mask;
#pragma unroll
                for (int i = 0; i < KMAX; ++i)
                    if (i < z1) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) K[q] |= sm.sk[q][t + i];
                    }
            }
            if (kQuery) {
                bool present = false;
                if (valid) {
                    const ulonglong2 *F = reinterpret_cast<const ulonglong2 *>(a.words + shard * 4);
                    const ulonglong2 f01 = __ldg(F), f23 = __ldg(F + 1);
                    present = ((K[0] & ~f01.x) | (K[1] & ~f01.y) | (K[2] & ~f23.x) | (K[3] & ~f23.y)) == 0;
                }
                if constexpr (B == 1) {
                    const unsigned bits = __ballot_sync(0xffffffffu, present);
                    if (lane == 0) sm.ans[warp] = bits;
                } else {
                    if (present) atomicOr(&sm.ans[j >> 5], 1u << (j & 31));
                }
            } else {
                // runs of lanes with one shard: segmented OR toward the run head
                const uint64_t key = valid ? shard : (1ull << 63) | (uint64_t)lane;
                const uint64_t prev_key = __shfl_up_sync(0xffffffffu, key, 1);
                const bool head = lane == 0 || prev_key != key;
                const unsigned heads = __ballot_sync(0xffffffffu, head);
                const unsigned after = heads & ~((2u << lane) - 1u);
                const int end = after ? __ffs(after) - 1 : 32;
                if (__any_sync(0xffffffffu, end > lane + 1)) {
#pragma unroll
                    for (int d = 1; d < 32; d <<= 1)
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const uint64_t v = __shfl_down_sync(0xffffffffu, K[q], d);
                            if (lane + d < end) K[q] |= v;
                        }
                }
                if (head && valid) {
                    unsigned long long *F = reinterpret_cast<unsigned long long *>(a.words + shard * 4);
                    for (int q = 0; q < n_words; ++q)
                        if (K[q]) atomicOr(F + q, K[q]);
                }
            }
            __syncthreads();
        }

        if (kQuery) {
            const int64_t w_lo = lo >> 5, w_hi = (hi + 31) >> 5;
            for (int i = t; i < T::OUTW; i += NT) {
                const int64_t gw = (t0 >> 5) + i;
                if (gw >= w_lo && gw < w_hi) a.out[gw] = sm.ans[i];
            }
        }
        __syncthreads();
    }
}

}  // namespace

const void *alphabet_insert_kernel(int alphabet) {
    if (alphabet == kAlphabetProtein) return reinterpret_cast<const void *>(&alphabet_kernel<kAlphabetProtein, false>);
    if (alphabet == kAlphabetTriplet) return reinterpret_cast<const void *>(&alphabet_kernel<kAlphabetTriplet, false>);
    return nullptr;
}

const void *alphabet_query_kernel(int alphabet) {
    if (alphabet == kAlphabetProtein) return reinterpret_cast<const void *>(&alphabet_kernel<kAlphabetProtein, true>);
    if (alphabet == kAlphabetTriplet) return reinterpret_cast<const void *>(&alphabet_kernel<kAlphabetTriplet, true>);
    return nullptr;
}

}  // namespace sbf
