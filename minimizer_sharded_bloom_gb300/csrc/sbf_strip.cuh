// sbf_strip.cuh -- compile-time specialised SBF insert/query kernels.
//
// Method: "cuSBF: A Minimizer-Aware Bloom Filter for Genomic Sequence Data on
// Modern GPUs" -- Algorithm 1 (insert) and Algorithm 2 (query), Sec. IV-B..G.
// This file keeps the method's results bit-exact and reorganises the work for
// GB300:
//
//  * Tile front end (Sec. IV-C): a CTA owns TILE consecutive k-mer positions.
//    It reads the TILE + k bases it needs once, as 16-byte coalesced loads,
//    converts 16 bytes at a time to 2-bit codes (first base in the high bits)
//    plus an invalid-byte bitmap with SWAR byte arithmetic, marks record starts
//    from the CSR offsets, and derives one validity bit per k-mer with
//    bit-parallel window ORs.  Everything lives in shared memory.
//
//  * Strips instead of one k-mer per thread (Sec. IV-E amortises packing over
//    kStride = 4 k-mers; here every thread owns a strip of L = NB*w
//    consecutive k-mers).  Bases enter a rolling register one at a time, so
//    each m-mer and each s-mer is packed and hashed once, not once per k-mer
//    that contains it.
//
//  * Minimizer (Algorithm 1 lines 5-9) with a Gil-Werman / van Herk sliding
//    minimum: the m-mer hashes are cut into blocks of w = k-m+1; the minimum
//    over a window is min(suffix-min of its first block, prefix-min of the
//    next) -- three 64-bit minimums per k-mer instead of w-1.  Exact, so the
//    shard is the paper's minHash & (NumShards - 1).
//
//  * Two passes per block of w k-mers: pass A (minimizer front) produces the
//    w shards of the block, pass B (s-mer front) hashes the s-mers, builds each
//    k-mer's four word masks and inserts or tests them.  For query, pass A
//    issues an L1 prefetch of each new shard, so the 32-byte shard is on chip
//    by the time pass B reads it (Sec. IV-E/IV-G: one 256-bit non-coherent
//    load per shard).
//
//  * Runs (Fig. 3): consecutive k-mers of a strip with one shard form a run;
//    their masks are ORed in registers and the run issues one 64-bit atomic OR
//    (a fire-and-forget reduction) per non-zero word -- the paper's segmented
//    warp reduction happens inside the thread, where the super-k-mer lies.
//
// Shared-memory indexing: code index ci <-> absolute base position
// T0 - 16 + ci, where T0 (a multiple of 32) is the tile's first k-mer; the
// k-mer at T0 + kk therefore starts at code index kk + 16.
#pragma once

#include <cstdint>

#include "sbf_device.cuh"

namespace sbf {

__device__ __forceinline__ uint32_t shl_clamp(uint32_t a, uint32_t s) {
    uint32_t d;  // PTX shl: shift amounts above 32 give 0
    asm("shl.b32 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(s));
    return d;
}

__device__ __forceinline__ void prefetch_l1(const void *p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// One 256-bit shard through the non-coherent path (Sec. IV-G).
__device__ __forceinline__ void load_shard(const uint64_t *p, uint64_t &a, uint64_t &b, uint64_t &c,
                                           uint64_t &d) {
    asm volatile("ld.global.nc.v4.u64 {%0, %1, %2, %3}, [%4];"
                 : "=l"(a), "=l"(b), "=l"(c), "=l"(d)
                 : "l"(p));
}

// 16 ASCII bytes (w[0] holds bytes 0..3, little-endian) -> 16 2-bit codes with
// the first base in bits 31..30 of `code`, and `bad` with bit i set iff byte i
// is not one of ACGTacgt.
//  * raw = bits 1..2 of each byte: A0 C1 T2 G3 for either case;
//  * the canonical upper-case letter of raw, via a byte permute of "ACTG",
//    equals the byte with bit 5 cleared exactly for the eight valid letters;
//  * code = raw with its low bit xored with its high bit: A0 C1 G2 T3;
//  * four codes x 0x40100401 put the four 2-bit codes, first byte's code
//    highest, in the top byte (the cross products stay below bit 24).
__device__ __forceinline__ void encode16(const uint32_t w[4], uint32_t &code, uint32_t &bad) {
    uint32_t top[4];
    bad = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t raw = (w[q] >> 1) & 0x03030303u;
        const uint32_t nib = raw | (raw >> 4);
        const uint32_t sel = __byte_perm(nib, 0u, 0x4420);
        const uint32_t canon = __byte_perm(0x47544341u, 0u, sel);
        const uint32_t diff = (w[q] & 0xDFDFDFDFu) ^ canon;
        if (diff) {
            const uint32_t hi = (((diff & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | diff) & 0x80808080u;
            bad |= (((hi >> 7) * 0x01020408u) >> 24) << (4 * q);
        }
        const uint32_t c = raw ^ ((raw >> 1) & 0x01010101u);
        top[q] = c * 0x40100401u;
    }
    const uint32_t t01 = __byte_perm(top[1], top[0], 0x7300);
    const uint32_t t23 = __byte_perm(top[3], top[2], 0x0073);
    code = __byte_perm(t23, t01, 0x7610);
}

// bit p (p < 32) = OR of bits p .. p+WD-1 of x
template <int WD>
__device__ __forceinline__ uint32_t window_or(uint64_t x) {
    if constexpr (WD <= 0) {
        return 0u;
    } else {
        constexpr int P = (WD >= 32) ? 32 : (WD >= 16) ? 16 : (WD >= 8) ? 8 : (WD >= 4) ? 4 : (WD >= 2) ? 2 : 1;
        uint64_t a = x;
#pragma unroll
        for (int s = 1; s < P; s <<= 1) a |= a >> s;
        return (uint32_t)(a | (a >> (WD - P)));
    }
}

// 64 bits of a shared bitmap starting at bit `bit`.
__device__ __forceinline__ uint64_t bits64_at(const uint32_t *bm, int bit) {
    const int wi = bit >> 5, sh = bit & 31;
    const uint32_t a = bm[wi], b = bm[wi + 1], c = bm[wi + 2];
    const uint32_t lo = __funnelshift_r(a, b, sh);
    const uint32_t hi = __funnelshift_r(b, c, sh);
    return ((uint64_t)hi << 32) | lo;
}

// 32 bases (64 bits, first base in bit 63..62) starting at code index ci.
__device__ __forceinline__ uint64_t codes32_at(const uint32_t *codes, int ci) {
    const int wi = ci >> 4, sh = (ci & 15) * 2;
    const uint32_t a = codes[wi], b = codes[wi + 1], c = codes[wi + 2];
    const uint32_t hi = __funnelshift_l(b, a, sh);
    const uint32_t lo = __funnelshift_l(c, b, sh);
    return ((uint64_t)hi << 32) | lo;
}

template <int K_, int M_, int S_, int H_>
struct StripCfg {
    static constexpr int K = K_, M = M_, S = S_, H = H_;
    static constexpr int W = K - M + 1;                 // m-mer windows per k-mer; block length
    static constexpr int Z = K - S;                     // s-mers per k-mer minus one
    static constexpr int NB = (W >= 16) ? 8 : (128 + W - 1) / W;  // blocks per strip
    static constexpr int L = NB * W;                    // k-mers per thread
    static constexpr int NT = 128;                      // threads per CTA
    static constexpr int TILE = NT * L;                 // k-mer positions per tile (multiple of 32)
    static constexpr int TILE_WORDS = TILE / 32;
    static constexpr int CODE_WORDS = (TILE + K + 96) / 16 + 4;  // 16 bases per word
    static constexpr int BIT_WORDS = (CODE_WORDS + 1) / 2 + 2;   // one bit per code index
    static constexpr int SW = 64 / H;                   // bit-slice width (Sec. IV-G)
    static constexpr uint64_t MASK_M = (M >= 32) ? ~0ull : ((1ull << (2 * M)) - 1);
    static constexpr uint64_t MASK_S = (S >= 32) ? ~0ull : ((1ull << (2 * S)) - 1);
    static_assert(W >= 1 && W <= 32 && Z >= 0 && H >= 1 && H <= 10, "parameters");
    static_assert(TILE % 32 == 0, "tile must cover whole output words");
};

template <int K, int M, int S, int H>
struct StripSmem {
    using C = StripCfg<K, M, S, H>;
    uint32_t codes[C::CODE_WORDS];
    uint16_t bad16[2 * C::BIT_WORDS];   // bit per code index; read as uint32 words
    uint32_t starts[C::BIT_WORDS];      // record-start bit per code index
    uint32_t valid[C::TILE_WORDS + 2];  // validity bit per k-mer of the tile
    uint32_t outw[C::TILE_WORDS + 2];   // query answer bits of the tile
    int64_t rec_first;
};

// The H bits of one s-mer hash as eight 32-bit halves (word w -> halves 2w, 2w+1).
template <int H>
__device__ __forceinline__ void smer_halves(uint64_t hs, uint32_t m[8]) {
    constexpr int SW = 64 / H;
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = 0u;
#pragma unroll
    for (int i = 0; i < H; ++i) {
        const uint32_t pos = (uint32_t)(hs >> (i * SW)) & 63u;
        m[2 * (i & 3)] |= shl_clamp(1u, pos);
        m[2 * (i & 3) + 1] |= shl_clamp(1u, pos - 32u);
    }
}

template <int K, int M, int S, int H, bool kQuery>
__global__ void __launch_bounds__(StripCfg<K, M, S, H>::NT) strip_kernel(LaunchArgs a) {
    using C = StripCfg<K, M, S, H>;
    constexpr int W = C::W, Z = C::Z, NB = C::NB, L = C::L, NT = C::NT, TILE = C::TILE;
    __shared__ StripSmem<K, M, S, H> sm;

    if (*reinterpret_cast<volatile int *>(a.status) & kStatusBadOffsets) return;
    const int64_t lo = a.offsets[0], hi = a.offsets[a.n];
    if (hi <= lo) return;
    const int64_t base = lo & ~int64_t(31);
    const int64_t n_tiles = (hi - base + TILE - 1) / TILE;
    const int tid = threadIdx.x;
    const bool aligned = ((reinterpret_cast<uintptr_t>(a.seq)) & 15u) == 0;
    const uint32_t smask = (uint32_t)a.shard_mask;
    const uint64_t seed_m = a.seed, seed_s = ~a.seed;
    const uint32_t *bad32 = reinterpret_cast<const uint32_t *>(sm.bad16);

    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int64_t T0 = base + tile * TILE;
        const int64_t A0 = T0 - 16;  // absolute position of code index 0
        // ---- phase 1: bases -> codes + invalid bits; clear per-tile bitmaps
        for (int w = tid; w < C::BIT_WORDS; w += NT) sm.starts[w] = 0u;
        if (kQuery)
            for (int w = tid; w < C::TILE_WORDS + 2; w += NT) sm.outw[w] = 0u;
        if (tid < 2) sm.valid[C::TILE_WORDS + tid] = 0u;
        for (int c = tid; c < C::CODE_WORDS; c += NT) {
            const int64_t p0 = A0 + 16 * (int64_t)c;
            uint32_t w[4];
            if (aligned && p0 >= lo && p0 + 16 <= hi) {
                const uint4 v = __ldg(reinterpret_cast<const uint4 *>(a.seq + p0));
                w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t x = 0;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {
                        const int64_t p = p0 + 4 * q + b;
                        const uint32_t byte = (p >= lo && p < hi) ? (uint32_t)a.seq[p] : 0u;
                        x |= byte << (8 * b);
                    }
                    w[q] = x;
                }
            }
            uint32_t code, bad;
            encode16(w, code, bad);
            sm.codes[c] = code;
            sm.bad16[c] = (uint16_t)bad;
        }
        for (int c = C::CODE_WORDS + tid; c < 2 * C::BIT_WORDS; c += NT) sm.bad16[c] = 0xFFFFu;
        if (tid == 0) {
            // first record boundary r (0..n) with offsets[r] > T0
            int64_t r_lo = 0, r_hi = a.n + 1;
            while (r_lo < r_hi) {
                const int64_t mid = r_lo + ((r_hi - r_lo) >> 1);
                if (a.offsets[mid] > T0) r_hi = mid; else r_lo = mid + 1;
            }
            sm.rec_first = r_lo;
        }
        __syncthreads();
        // ---- phase 2: record starts inside (T0, T0 + TILE + K - 1)
        {
            const int64_t lim = T0 + TILE + K - 1;
            for (int64_t r = sm.rec_first + tid; r <= a.n; r += NT) {
                const int64_t p = a.offsets[r];
                if (p >= lim) break;
                const int ci = (int)(p - A0);
                atomicOr(&sm.starts[ci >> 5], 1u << (ci & 31));
            }
        }
        __syncthreads();
        // ---- phase 3: validity bit per k-mer: no invalid base in its k bases,
        // no record start among its bases 1 .. k-1.
        for (int v = tid; v < C::TILE_WORDS; v += NT) {
            const uint64_t badw = bits64_at(bad32, 32 * v + 16);
            const uint64_t stw = bits64_at(sm.starts, 32 * v + 17);
            sm.valid[v] = ~(window_or<K>(badw) | window_or<K - 1>(stw));
        }
        __syncthreads();

        // ---- phase 4: strips
        const int kk0 = tid * L;  // first k-mer of this thread (tile relative)
        if (T0 + kk0 < hi) {
            // m-front: m-mer u of the strip starts at code index kk0 + 15 + u
            // (the strip's first k-mer is u = 1); s-front follows the k-mers.
            uint64_t rm = 0, rs = 0;
            uint64_t suf[W];
            uint32_t shard[W];
            uint32_t mk[Z + 1][8];
#pragma unroll
            for (int i = 0; i < W; ++i) suf[i] = ~0ull;
#pragma unroll
            for (int z = 0; z <= Z; ++z)
#pragma unroll
                for (int j = 0; j < 8; ++j) mk[z][j] = 0u;
            // warm-up of the m-front: bases u = 0 .. M-2
            {
                const uint64_t win = codes32_at(sm.codes, kk0 + 15);
#pragma unroll
                for (int b = 0; b < M - 1; ++b) rm = (rm << 2) | ((win >> (62 - 2 * b)) & 3u);
            }
            // warm-up of the s-front: bases of k-mer kk0 except its last one,
            // computing the first Z s-mers.
            {
                const uint64_t win = codes32_at(sm.codes, kk0 + 16);
#pragma unroll
                for (int b = 0; b < K - 1; ++b) {
                    rs = (rs << 2) | ((win >> (62 - 2 * b)) & 3u);
                    if (b >= S - 1) {
#pragma unroll
                        for (int z = 0; z < Z; ++z)
#pragma unroll
                            for (int j = 0; j < 8; ++j) mk[z][j] = mk[z + 1][j];
                        smer_halves<H>(hash_smer(rs & C::MASK_S, seed_s), mk[Z]);
                    }
                }
            }
            // run / answer state
            uint32_t cur = 0;
            bool cur_v = false;
            uint32_t acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0u;
            uint64_t F0 = 0, F1 = 0, F2 = 0, F3 = 0;
            uint64_t *const words = a.words;

#pragma unroll 1
            for (int blk = 0; blk <= NB; ++blk) {
                // -- pass A: m-mers u = blk*W .. blk*W + W-1; emits the shards of
                //    k-mers u = (blk-1)*W + 1 .. blk*W (the strip's block blk-1).
                {
                    const uint64_t win = codes32_at(sm.codes, kk0 + 15 + blk * W + M - 1);
                    uint64_t h[W];
                    uint64_t pre = ~0ull;
#pragma unroll
                    for (int i = 0; i < W; ++i) {
                        rm = (rm << 2) | ((win >> (62 - 2 * i)) & 3u);
                        h[i] = hash_minimizer(rm & C::MASK_M, seed_m);
                        pre = h[i] < pre ? h[i] : pre;
                        if (i < W - 1) {
                            const uint64_t mu = suf[i + 1] < pre ? suf[i + 1] : pre;
                            shard[i] = (uint32_t)mu & smask;
                        }
                    }
                    suf[W - 1] = h[W - 1];
#pragma unroll
                    for (int i = W - 2; i >= 0; --i) suf[i] = h[i] < suf[i + 1] ? h[i] : suf[i + 1];
                    shard[W - 1] = (uint32_t)suf[0] & smask;
                    if (kQuery && blk > 0) {
#pragma unroll
                        for (int i = 0; i < W; ++i)
                            if (i == 0 || shard[i] != shard[i - 1]) prefetch_l1(words + (uint64_t)shard[i] * 4);
                    }
                }
                if (blk == 0) continue;
                // -- pass B: k-mers kk = kk0 + (blk-1)*W + i
                {
                    const int kb = kk0 + (blk - 1) * W;
                    const uint64_t win = codes32_at(sm.codes, kb + 16 + K - 1);
                    const uint64_t vwin = bits64_at(sm.valid, kb);
                    uint32_t present = 0;
#pragma unroll
                    for (int i = 0; i < W; ++i) {
                        rs = (rs << 2) | ((win >> (62 - 2 * i)) & 3u);
#pragma unroll
                        for (int z = 0; z < Z; ++z)
#pragma unroll
                            for (int j = 0; j < 8; ++j) mk[z][j] = mk[z + 1][j];
                        smer_halves<H>(hash_smer(rs & C::MASK_S, seed_s), mk[Z]);
                        uint32_t km[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            uint32_t x = mk[0][j];
#pragma unroll
                            for (int z = 1; z <= Z; ++z) x |= mk[z][j];
                            km[j] = x;
                        }
                        const bool v = (vwin >> i) & 1u;
                        const uint32_t sh = shard[i];
                        if (!kQuery) {
                            const bool same = v && cur_v && sh == cur;
                            if (cur_v && !same) {
                                uint64_t *F = words + (uint64_t)cur * 4;
#pragma unroll
                                for (int wd = 0; wd < 4; ++wd) {
                                    if (wd >= H) continue;
                                    const uint64_t val = ((uint64_t)acc[2 * wd + 1] << 32) | acc[2 * wd];
                                    atomicOr(reinterpret_cast<unsigned long long *>(F + wd), val);
                                }
                            }
                            const uint32_t keep = same ? ~0u : 0u;
#pragma unroll
                            for (int j = 0; j < 8; ++j) acc[j] = (acc[j] & keep) | km[j];
                            cur = sh;
                            cur_v = v;
                        } else {
                            if (v && (!cur_v || sh != cur)) {
                                load_shard(words + (uint64_t)sh * 4, F0, F1, F2, F3);
                                cur = sh;
                                cur_v = true;
                            }
                            const uint32_t miss =
                                (km[0] & ~(uint32_t)F0) | (km[1] & ~(uint32_t)(F0 >> 32)) |
                                (km[2] & ~(uint32_t)F1) | (km[3] & ~(uint32_t)(F1 >> 32)) |
                                (km[4] & ~(uint32_t)F2) | (km[5] & ~(uint32_t)(F2 >> 32)) |
                                (km[6] & ~(uint32_t)F3) | (km[7] & ~(uint32_t)(F3 >> 32));
                            present |= (uint32_t)(v && miss == 0u) << i;
                        }
                    }
                    if (kQuery && present) {
                        const int wi = kb >> 5, sh = kb & 31;
                        atomicOr(&sm.outw[wi], present << sh);
                        if (sh + W > 32) atomicOr(&sm.outw[wi + 1], (uint32_t)((uint64_t)present >> (32 - sh)));
                    }
                }
            }
            if (!kQuery && cur_v) {
                uint64_t *F = words + (uint64_t)cur * 4;
#pragma unroll
                for (int wd = 0; wd < 4; ++wd) {
                    if (wd >= H) continue;
                    const uint64_t val = ((uint64_t)acc[2 * wd + 1] << 32) | acc[2 * wd];
                    atomicOr(reinterpret_cast<unsigned long long *>(F + wd), val);
                }
            }
        }
        __syncthreads();
        if (kQuery) {
            const int64_t w_lo = lo >> 5, w_hi = (hi + 31) >> 5;
            for (int w = tid; w < C::TILE_WORDS; w += NT) {
                const int64_t gw = (T0 >> 5) + w;
                if (gw >= w_lo && gw < w_hi) a.out[gw] = sm.outw[w];
            }
            __syncthreads();
        }
    }
}

// Registration helper used by the instantiation files.
struct StripEntry {
    int k, m, s, H;
    const void *insert;
    const void *query;
    int threads;
};

template <int K, int M, int S, int H>
inline StripEntry strip_entry() {
    return StripEntry{K, M, S, H, reinterpret_cast<const void *>(&strip_kernel<K, M, S, H, false>),
                      reinterpret_cast<const void *>(&strip_kernel<K, M, S, H, true>),
                      StripCfg<K, M, S, H>::NT};
}

}  // namespace sbf
