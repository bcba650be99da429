// sbf_alphabet.cu -- SBF insert/query kernels for the protein and DNA-triplet
// alphabets ("cuSBF", Sec. IV-A: proteins, 26 symbols in 5 bits; DNA triplets,
// 64 symbols in 6 bits, each symbol read from several input bytes).  k * bits
// <= 64 (Sec. IV-C: one k-mer packs into one 64-bit word, so protein k <= 12
// and triplet k <= 10).
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
//  * a block owns a contiguous range of tiles of TB = 256*B bytes (tile
//    starts are multiples of 32); the record boundaries of a tile (plus the
//    k-mer overhang) are loaded in one parallel round from the first boundary
//    after the tile start, carried over from the previous tile, and marked in
//    a bitmap; the tile's bytes become one symbol code per byte;
//  * the tile is covered in B passes; in pass p lane t owns byte B*t + p, so
//    within one record the lanes of a pass that start a symbol hold
//    consecutive k-mers (for triplets, one pass of three carries each
//    record's frame);
//  * per pass, every slot packs its symbols once and stores its m-mer hash and
//    its s-mer's four word masks (shared memory); symbol validity is one
//    ballot bit per slot.  Every k-mer then takes the minimum over its
//    w = k-m+1 m-mer hashes (Algorithm 1);
//  * insert: lanes holding consecutive valid k-mers with one shard form a run
//    (the paper's super-k-mer runs, Fig. 3); the run's head lane ORs the s-mer
//    masks of the run's contiguous s-mer slots and issues one atomicOr per
//    non-zero word.  Query: each valid k-mer ORs its k-s+1 s-mer masks, tests
//    its shard's four words (Algorithm 2) and the answers are assembled in
//    shared memory and stored coalesced.
// The benchmarked parameter points have compile-time specialisations; every
// other valid (k, m, s, H) runs the same kernel with runtime loop bounds.
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
constexpr int64_t kNoStart = INT64_MIN;

template <int ALPHA>
struct AlphaTile {
    static constexpr int B = AlphaCfg<ALPHA>::B, BITS = AlphaCfg<ALPHA>::BITS, KMAX = AlphaCfg<ALPHA>::KMAX;
    static constexpr int NT = kAlphaThreads;
    static constexpr int TB = NT * B;                 // tile bytes (k-mer start positions)
    static constexpr int HN = NT + KMAX - 1;          // hash slots per pass
    static constexpr int CODES = TB + 2 * B * KMAX;   // symbol codes (one per start byte), padded
    static constexpr int RAW = CODES + B - 1;         // bytes the codes read
    static constexpr int SPAN = TB + B * KMAX;        // boundary bitmap reach
    static constexpr int BW = (SPAN + 31) / 32 + 1;   // bitmap words (+1: two-word reads)
    static constexpr int VW = (HN + 31) / 32 + 1;     // symbol-valid words per pass
    static constexpr int OUTW = TB / 32;              // answer words per tile
    static_assert(TB % 32 == 0, "tiles must cover whole answer words");
    static_assert(B * KMAX - 1 < 32, "a k-mer's inner boundaries must fit one 32-bit window");
    static_assert(KMAX - 1 <= 32, "halo slots are filled by warp 0");
};

template <int ALPHA, bool kQuery>
struct AlphaSmem {
    using T = AlphaTile<ALPHA>;
    uint64_t hm[T::HN];      // m-mer hash at slot u (byte B*u + pass)
    uint64_t sk[4][T::HN];   // s-mer word masks at slot u
    uint32_t starts[T::BW];  // bit i: a record boundary at byte t0 + i (i >= 1)
    uint32_t symok[T::VW];   // bit u: the symbol at slot u is valid
    uint32_t ans[T::OUTW];
    uint32_t racc[8][kQuery ? 1 : T::NT];  // insert: run masks (word halves) by head thread
    int64_t prev_start;      // last boundary <= t0, or kNoStart
    int64_t r_start;         // first boundary index with offsets[r] > t0
    uint8_t raw[ALPHA == kAlphabetTriplet ? T::RAW : 1];
    uint8_t code[T::CODES];
};

__device__ __forceinline__ uint32_t codon_code(uint32_t c0, uint32_t c1, uint32_t c2) {
    const int a = base_code(c0), b = base_code(c1), c = base_code(c2);
    return (a | b | c) < 0 ? kBadCode : (uint32_t)(a * 16 + b * 4 + c);
}

// Bits [from, from + len) of a bitmap as the low bits of a word, 0 <= len <= 32.
__device__ __forceinline__ uint32_t bits_at(const uint32_t *bm, int from, int len) {
    const int w = from >> 5;
    const uint64_t two = (uint64_t)bm[w] | ((uint64_t)bm[w + 1] << 32);
    return (uint32_t)((two >> (from & 31)) & ((1ull << len) - 1ull));
}

// Highest boundary at or below tile byte j (absolute), else prev.
__device__ __forceinline__ int64_t start_at_or_below(const uint32_t *bm, int j, int64_t t0, int64_t prev) {
    int w = j >> 5;
    uint32_t b = bm[w] & (0xFFFFFFFFu >> (31 - (j & 31)));
    while (!b && w > 0) b = bm[--w];
    return b ? t0 + 32 * w + 31 - __clz(b) : prev;
}

// The s-mer's H bits as four word masks; compile-time H when H_ > 0
// (`sectors`: hash-chosen words for H < 4, sector_word).
template <int H_>
__device__ __forceinline__ void smer_words(uint64_t hs, int H, uint64_t K[4], int sectors) {
    K[0] = K[1] = K[2] = K[3] = 0ull;
    if constexpr (H_ > 0) {
        constexpr int SW = 64 / H_;
#pragma unroll
        for (int i = 0; i < H_; ++i) {
            uint32_t pos;
            if constexpr (SW >= 6) pos = (uint32_t)(hs >> (i * SW)) & 63u;
            else pos = (uint32_t)((hs * salt_of(i)) >> 58);
            if (H_ < 4 && sectors)
                or_into_word(K, sector_word(hs, i, SW), 1ull << pos);
            else
                K[i & 3] |= 1ull << pos;
        }
    } else {
        smer_bits_runtime(hs, H, K, sectors);
    }
}

// K_ > 0: compile-time (k, m, s, H); K_ == 0: the launch's runtime values.
template <int ALPHA, int K_, int M_, int S_, int H_, bool kQuery>
__global__ void __launch_bounds__(kAlphaThreads) alphabet_kernel(LaunchArgs a) {
    using T = AlphaTile<ALPHA>;
    constexpr int B = T::B, BITS = T::BITS, KMAX = T::KMAX, NT = T::NT, TB = T::TB;
    constexpr bool kStatic = K_ > 0;
    __shared__ AlphaSmem<ALPHA, kQuery> sm;
    if (*reinterpret_cast<volatile int *>(a.status) & kStatusBadOffsets) return;
    const int64_t lo = a.offsets[0], hi = a.offsets[a.n];
    if (hi <= lo) return;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int k = kStatic ? K_ : a.k, m = kStatic ? M_ : a.m, s = kStatic ? S_ : a.s;
    const int w = k - m + 1, z1 = k - s + 1, L = m > s ? m : s;
    const int kspan = B * k;
    const uint64_t seed_m = a.seed, seed_s = ~a.seed;
    // words a k-mer's bits can reach: 0..H-1 when H < 4 (word i mod 4), all
    // four with hash-chosen sectors or H >= 4
    const int n_words = a.sectors ? 4 : kStatic ? (H_ < 4 ? H_ : 4) : (a.H < 4 ? a.H : 4);
    const int64_t base = lo & ~int64_t(31);
    const int64_t n_tiles = (hi - base + TB - 1) / TB;
    // this block's contiguous tile range
    const int64_t tile_b = n_tiles * blockIdx.x / gridDim.x;
    const int64_t tile_e = n_tiles * (blockIdx.x + 1) / gridDim.x;
    if (tile_b >= tile_e) return;

    // A tile's inputs are loaded one tile ahead into registers (raw bytes, 0
    // outside [lo, hi); the first NT record boundaries from the tile's first
    // boundary index on; the boundary before it) and stored to shared memory
    // after the previous tile's passes, so their latency overlaps compute.
    constexpr int NBYTES = (B == 1) ? T::CODES : T::RAW;
    constexpr int NPF = (NBYTES + NT - 1) / NT;
    uint32_t pf_byte[NPF];
    int64_t pf_bound = INT64_MAX, pf_prev = kNoStart;
    auto prefetch = [&](int64_t t0n, int64_t r_from) {
#pragma unroll
        for (int i = 0; i < NPF; ++i) {
            const int u = t + i * NT;
            const int64_t g = t0n + u;
            pf_byte[i] = (u < NBYTES && g >= lo && g < hi) ? (uint32_t)a.seq[g] : 0u;
        }
        const int64_t r = r_from + t;
        pf_bound = r <= a.n ? a.offsets[r] : INT64_MAX;
        if (t == 0) pf_prev = r_from >= 1 ? a.offsets[r_from - 1] : kNoStart;
    };

    for (int i = t; i < T::BW; i += NT) sm.starts[i] = 0u;
    if (kQuery)
        for (int i = t; i < T::OUTW; i += NT) sm.ans[i] = 0u;
    if (warp == 0) {
        const int64_t r0 = warp_find_boundary(a.offsets, a.n, base + tile_b * TB, lo, hi, lane);
        if (lane == 0) sm.r_start = r0;
    }
    __syncthreads();
    int64_t r_cur = sm.r_start;  // first boundary index with offsets[r] > t0 (block-uniform)
    prefetch(base + tile_b * TB, r_cur);

    for (int64_t tile = tile_b; tile < tile_e; ++tile) {
        const int64_t t0 = base + tile * TB;
        const int64_t lim = t0 + T::SPAN;
        // ---- record boundaries in (t0, lim): the prefetched round, then more
        //      rounds of NT while the last one is still inside
        if (t == 0) sm.prev_start = pf_prev;
        int n_le = 0;  // boundaries <= t0 + TB (block-wide count)
        {
            int64_t p = pf_bound;
            for (int64_t rb = r_cur;;) {
                // (p > t0 holds for every r >= r_cur; checked so that the
                // bitmap index stays in range whatever the offsets hold)
                if (p > t0 && p < lim) atomicOr(&sm.starts[(p - t0) >> 5], 1u << ((p - t0) & 31));
                n_le += __syncthreads_count(p <= t0 + TB);
                if (!__syncthreads_or(t == NT - 1 && p < lim)) break;
                rb += NT;
                const int64_t r = rb + t;
                p = r <= a.n ? a.offsets[r] : INT64_MAX;
            }
        }
        // ---- symbol codes (protein) or raw bytes (triplets)
#pragma unroll
        for (int i = 0; i < NPF; ++i) {
            const int u = t + i * NT;
            if (u < NBYTES) {
                if constexpr (B == 1) sm.code[u] = (uint8_t)protein_code(pf_byte[i]);
                else sm.raw[u] = (uint8_t)pf_byte[i];
            }
        }
        __syncthreads();
        r_cur += n_le;
        if (tile + 1 < tile_e) prefetch(t0 + TB, r_cur);
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
            const bool placed = in_frame && g + kspan <= hi && bits_at(sm.starts, j + 1, kspan - 1) == 0u;

            // ---- per slot (byte B*u + pass): pack max(m, s) symbols once; the
            //      m-mer and s-mer are its leading symbols.  Slots that are out
            //      of frame are never read by a placed k-mer of this pass.
            // (each code is cut to BITS bits: the invalid marker would
            // otherwise spill into the field above it, and a symbol past the
            // shorter of the two windows may be invalid in a valid k-mer)
            auto fill = [&](int u) {
                const int pos = B * u + pass;
                uint64_t v = 0;
#pragma unroll
                for (int i = 0; i < L; ++i) v = (v << BITS) | (sm.code[pos + B * i] & ((1u << BITS) - 1u));
                sm.hm[u] = hash_minimizer(v >> (BITS * (L - m)), seed_m);
                uint64_t K[4];
                smer_words<H_>(hash_smer(v >> (BITS * (L - s)), seed_s), a.H, K, a.sectors);
#pragma unroll
                for (int q = 0; q < 4; ++q) sm.sk[q][u] = K[q];
            };
            if (B == 1 || in_frame) fill(t);
            if (t < KMAX - 1) fill(NT + t);
            {
                const unsigned ok = __ballot_sync(0xffffffffu, sm.code[j] != kBadCode);
                if (lane == 0) sm.symok[warp] = ok;
                if (warp == 0) {
                    const unsigned okh =
                        __ballot_sync(0xffffffffu, lane < KMAX - 1 && sm.code[B * (NT + lane) + pass] != kBadCode);
                    if (lane == 0) sm.symok[NT / 32] = okh;
                }
            }
            __syncthreads();

            // ---- this lane's k-mer from the slots
            bool valid = placed && bits_at(sm.symok, t, k) == (uint32_t)((1ull << k) - 1ull);
            uint64_t shard = 0;
            if (valid) {
                uint64_t mu = ~0ull;
#pragma unroll
                for (int i = 0; i < w; ++i) {
                    const uint64_t h = sm.hm[t + i];
                    mu = h < mu ? h : mu;
                }
                shard = mu & a.shard_mask;
            }
            if constexpr (kQuery) {
                bool present = false;
                if (valid) {
                    uint64_t K0 = 0, K1 = 0, K2 = 0, K3 = 0;
#pragma unroll
                    for (int i = 0; i < z1; ++i) {
                        K0 |= sm.sk[0][t + i];
                        K1 |= sm.sk[1][t + i];
                        K2 |= sm.sk[2][t + i];
                        K3 |= sm.sk[3][t + i];
                    }
                    const ulonglong2 *F = reinterpret_cast<const ulonglong2 *>(a.words + shard * 4);
                    const ulonglong2 f01 = __ldg(F), f23 = __ldg(F + 1);
                    present = ((K0 & ~f01.x) | (K1 & ~f01.y) | (K2 & ~f23.x) | (K3 & ~f23.y)) == 0;
                }
                if constexpr (B == 1) {
                    const unsigned bits = __ballot_sync(0xffffffffu, present);
                    if (lane == 0) sm.ans[warp] = bits;
                } else {
                    if (present) atomicOr(&sm.ans[j >> 5], 1u << (j & 31));
                }
            } else {
                // this k-mer's mask, then runs: consecutive lanes with one shard.
                // Lanes after a run's head OR their masks into the head's column
                // of `racc` (32-bit shared atomics); the head then issues one
                // atomicOr per non-zero word.
                uint64_t Kq[4] = {0, 0, 0, 0};
                if (valid) {
#pragma unroll
                    for (int i = 0; i < z1; ++i) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) Kq[q] |= sm.sk[q][t + i];
                    }
                }
                const uint64_t key = valid ? shard : (1ull << 63) | (uint64_t)lane;
                const uint64_t prev_key = __shfl_up_sync(0xffffffffu, key, 1);
                const bool head = lane == 0 || prev_key != key;
                const unsigned heads = __ballot_sync(0xffffffffu, head);
                const int head_lane = 31 - __clz(heads & (0xFFFFFFFFu >> (31 - lane)));
                if (__any_sync(0xffffffffu, head_lane != lane)) {
                    if (head) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            sm.racc[2 * q][t] = (uint32_t)Kq[q];
                            sm.racc[2 * q + 1][t] = (uint32_t)(Kq[q] >> 32);
                        }
                    }
                    __syncwarp();
                    if (!head && valid) {
                        const int col = (t & ~31) + head_lane;
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (q < n_words) {
                                atomicOr(&sm.racc[2 * q][col], (uint32_t)Kq[q]);
                                atomicOr(&sm.racc[2 * q + 1][col], (uint32_t)(Kq[q] >> 32));
                            }
                    }
                    __syncwarp();
                    if (head) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            Kq[q] = (uint64_t)sm.racc[2 * q][t] | ((uint64_t)sm.racc[2 * q + 1][t] << 32);
                    }
                }
                if (head && valid) {
                    unsigned long long *F = reinterpret_cast<unsigned long long *>(a.words + shard * 4);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (q < n_words && Kq[q]) atomicOr(F + q, Kq[q]);
                }
            }
            __syncthreads();
        }

        if (kQuery) {
            const int64_t w_lo = lo >> 5, w_hi = min((hi + 31) >> 5, a.out_words_end);
            for (int i = t; i < T::OUTW; i += NT) {
                const int64_t gw = (t0 >> 5) + i;
                if (gw >= w_lo && gw < w_hi) a.out[gw] = sm.ans[i];
            }
        }
        __syncthreads();
        for (int i = t; i < T::BW; i += NT) sm.starts[i] = 0u;
        if (kQuery)
            for (int i = t; i < T::OUTW; i += NT) sm.ans[i] = 0u;
        __syncthreads();
    }
}

struct AlphaEntry {
    int alphabet, k, m, s, H;
    const void *insert, *query;
};

template <int ALPHA, int K, int M, int S, int H>
constexpr AlphaEntry alpha_entry() {
    return AlphaEntry{ALPHA, K, M, S, H, reinterpret_cast<const void *>(&alphabet_kernel<ALPHA, K, M, S, H, false>),
                      reinterpret_cast<const void *>(&alphabet_kernel<ALPHA, K, M, S, H, true>)};
}

}  // namespace

bool find_alphabet_kernels(int alphabet, int k, int m, int s, int H, const void **insert, const void **query,
                           bool *specialized, bool may_specialise) {
    // the benchmarked points (protein 12/8/10/4, triplet 10/5/8/4), then the
    // runtime-parameter kernels
    static const AlphaEntry table[] = {
        alpha_entry<kAlphabetProtein, 12, 8, 10, 4>(),
        alpha_entry<kAlphabetTriplet, 10, 5, 8, 4>(),
    };
    for (const AlphaEntry &e : table)
        if (may_specialise && e.alphabet == alphabet && e.k == k && e.m == m && e.s == s && e.H == H) {
            *insert = e.insert;
            *query = e.query;
            *specialized = true;
            return true;
        }
    *specialized = false;
    if (alphabet == kAlphabetProtein) {
        *insert = reinterpret_cast<const void *>(&alphabet_kernel<kAlphabetProtein, 0, 0, 0, 0, false>);
        *query = reinterpret_cast<const void *>(&alphabet_kernel<kAlphabetProtein, 0, 0, 0, 0, true>);
        return true;
    }
    if (alphabet == kAlphabetTriplet) {
        *insert = reinterpret_cast<const void *>(&alphabet_kernel<kAlphabetTriplet, 0, 0, 0, 0, false>);
        *query = reinterpret_cast<const void *>(&alphabet_kernel<kAlphabetTriplet, 0, 0, 0, 0, true>);
        return true;
    }
    return false;
}

}  // namespace sbf
