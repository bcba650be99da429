// sbf_strip.cuh -- compile-time specialised SBF insert/query kernels.
//
// Method: "cuSBF: A Minimizer-Aware Bloom Filter for Genomic Sequence Data on
// Modern GPUs" -- Algorithm 1 (insert) and Algorithm 2 (query), Sec. IV-B..G.
// This file keeps the method's results bit-exact and reorganises the work for
// GB300:
//
//  * Tile front end (Sec. IV-C): a CTA owns TILE consecutive k-mer positions.
//    The TILE + k bytes it needs arrive once, by one TMA bulk copy issued a
//    tile ahead (16-byte loads where the copy cannot be used); 16 bytes at a
//    time become 2-bit codes (first base in the high bits) plus an
//    invalid-byte bitmap with SWAR byte arithmetic; record starts come from
//    the CSR offsets (or arithmetically for dense batches), and one validity
//    bit per k-mer from bit-parallel window ORs.  Everything lives in shared
//    memory.
//
//  * Strips instead of one k-mer per thread (Sec. IV-E amortises packing over
//    kStride = 4 k-mers; here every thread owns a strip of L = NB*w
//    consecutive k-mers).  Each m-mer and each s-mer is cut out of a 64-base
//    window of the code tile by funnel shifts and hashed once, not once per
//    k-mer that contains it.
//
//  * Minimizer (Algorithm 1's minimum m-mer hash) with a Gil-Werman / van Herk sliding
//    minimum: the m-mer hashes are cut into blocks of w = k-m+1; the minimum
//    over a window is min(suffix-min of its first block, prefix-min of the
//    next) -- three 64-bit minimums per k-mer instead of w-1.  Exact, so the
//    shard is the paper's minHash & (NumShards - 1).
//
//  * Two passes per block of w k-mers: pass A (minimizer front) produces the
//    w shards of the block, pass B (s-mer front) hashes the s-mers, builds each
//    k-mer's four word masks and inserts or tests them.  For query, pass A
//    copies each run head's 32-byte shard into shared memory (cp.async), so
//    the shard is on chip by the time pass B reads it (Sec. IV-E/IV-G: one
//    256-bit load per shard); heads beyond the block's slots get an L2
//    prefetch instead, and pass B loads them directly.
//
//  * Runs (Fig. 3): consecutive k-mers of a strip with one shard form a run;
//    their masks are ORed in registers and the run issues one 64-bit atomic OR
//    (a fire-and-forget reduction) per non-zero word -- the paper's segmented
//    warp reduction happens inside the thread, where the super-k-mer lies.
//    On filters far larger than L2 (FQ = 1) finished runs go through a
//    per-warp shared-memory queue instead, drained four lanes per run, so a
//    run's four words reach L2 as one 32-byte request.
//
// Shared-memory indexing: code index ci <-> absolute base position
// T0 - 16 + ci, where T0 (a multiple of 32) is the tile's first k-mer; the
// k-mer at T0 + kk therefore starts at code index kk + 16.
//
// Alphabets (Sec. IV-A): A = 0 is DNA as above.  A = 1 is the protein
// alphabet (26 letters, 5 bits per symbol, one byte per symbol): the front end
// stores one 5-bit code per byte instead of the 2-bit words, and pass A / pass
// B roll their m-mer / s-mer values forward by one symbol per position
// (v = v << 5 | code) instead of cutting them out of 64-base windows.  Validity,
// record starts, the sliding minimum, runs and the query's shard slots are the
// same code.  A = 2 is the DNA-triplet alphabet (6-bit codons read in frame):
// a tile covers three times the bytes, in up to three frame passes that each
// form one codon per three bytes and then run the protein machinery; a pass
// with no codon in frame is skipped.
#pragma once

#include <cstdint>

#include "sbf_device.cuh"

namespace sbf {

// Flush one run: a 64-bit OR reduction per non-zero word of the shard.  The
// word values are first copied into registers of their own, so that the
// accumulator can be reset at once instead of waiting until the reductions
// have read their operands.
template <int H>
__device__ __forceinline__ void flush_run(uint64_t *F, const uint32_t acc[8]) {
    uint64_t v[4];
#pragma unroll
    for (int wd = 0; wd < 4; ++wd)
        asm volatile("mov.b64 %0, {%1, %2};" : "=l"(v[wd]) : "r"(acc[2 * wd]), "r"(acc[2 * wd + 1]));
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
        if (wd >= H) continue;
        asm volatile("red.global.or.b64 [%0], %1;" ::"l"(F + wd), "l"(v[wd]) : "memory");
    }
}

// Cooperative flush over the warp's active lanes `am` (protein and triplet
// inserts, whose runs are short): the runs that end at this step are written
// to the warp's staging area (st_key, st_acc: 32 runs) at their rank among
// the flushing lanes, then the active lanes reduce them as (run, word) pairs,
// pair 4r + w on the lane of rank (4r + w) mod n_active, so a run's four
// words leave in one instruction and reach L2 as one 32-byte request.  The
// trip count, ceil(4 * runs / n_active) <= 128, is the same on every active
// lane.
template <int H>
__device__ __forceinline__ void flush_coop(uint64_t *words, uint32_t key, const uint32_t acc[8], bool flush,
                                           unsigned am, uint32_t *st_key, uint4 *st_acc) {
    const unsigned fm = __ballot_sync(am, flush);
    if (!fm) return;
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    if (flush) {
        const int e = __popc(fm & lt);
        st_key[e] = key;
        st_acc[2 * e] = make_uint4(acc[0], acc[1], acc[2], acc[3]);
        st_acc[2 * e + 1] = make_uint4(acc[4], acc[5], acc[6], acc[7]);
    }
    __syncwarp(am);
    const int rank = __popc(am & lt);
    const int n_act = __popc(am);
    const int pairs = 4 * __popc(fm);
    for (int base = 0; base < pairs; base += n_act) {
        const int pidx = base + rank;
        if (pidx < pairs) {
            const int rr = pidx >> 2, wd = pidx & 3;
            const uint2 v = reinterpret_cast<const uint2 *>(st_acc + 2 * rr)[wd];
            if (wd < H && (v.x | v.y)) {
                const uint64_t x = ((uint64_t)v.y << 32) | v.x;
                asm volatile("red.global.or.b64 [%0], %1;" ::"l"(words + (uint64_t)st_key[rr] * 4 + wd), "l"(x)
                             : "memory");
            }
        }
    }
    __syncwarp(am);
}

// A run head's shard in pass B: from its slot when `staged`, else straight
// from global memory (64-byte L2 fetch), chosen by predicate inside one asm
// block rather than by a nested branch.
__device__ __forceinline__ void head_shard(uint64_t &a, uint64_t &b, uint64_t &c, uint64_t &d, uint32_t lo,
                                           uint32_t hi, const uint64_t *src, bool staged) {
    asm volatile("{ .reg .pred q; setp.ne.u32 q, %4, 0;\n\t"
                 "@q ld.shared.v2.u64 {%0, %1}, [%5];\n\t@q ld.shared.v2.u64 {%2, %3}, [%6];\n\t"
                 "@!q ld.global.nc.L2::64B.v4.u64 {%0, %1, %2, %3}, [%7]; }"
                 : "=l"(a), "=l"(b), "=l"(c), "=l"(d)
                 : "r"(staged ? 1u : 0u), "r"(lo), "r"(hi), "l"(src)
                 : "memory");
}

// Per-warp queue of finished runs (DNA insert).  A lane whose run ends
// writes it (shard key, eight half-words) at the queue's tail; once drain_at
// runs wait, the warp drains them in groups of eight, lane l reducing word
// l & 3 of run l >> 2, so that each run's four words reach L2 as one 32-byte
// request instead of four (drain_at = 1: the strip's end, everything, the
// last group partly).  head / tail are warp-uniform counters.  The ring holds
// QN = 128 entries: at most 39 runs wait when a drain starts (7 left over plus
// one step's 32), so the next step's writes land at least 128 - 2 * 39 slots
// away from the entries a drain just read, and the warp need not synchronise
// after a drain; it does before one (the entries it reads were written by
// other lanes).  Called by all 32 lanes.
template <int H, int QN>
__device__ __forceinline__ void drain_group(const uint32_t *q_acc, const uint32_t *q_key, int head, int lane,
                                            uint64_t *words) {
    const int e = (head + (lane >> 2)) & (QN - 1), wd = lane & 3;
    const uint2 v = reinterpret_cast<const uint2 *>(q_acc + 8 * e)[wd];
    const uint64_t x = ((uint64_t)v.y << 32) | v.x;
    if (wd < H && x)
        asm volatile("red.global.or.b64 [%0], %1;" ::"l"(words + (uint64_t)q_key[e] * 4 + wd), "l"(x) : "memory");
}

template <int H, int QN>
__device__ __forceinline__ void queue_runs(uint32_t *q_acc, uint32_t *q_key, int &head, int &tail, bool flush,
                                           uint32_t key, const uint32_t acc[8], int lane, int drain_at,
                                           uint64_t *words) {
    const unsigned fm = __ballot_sync(0xffffffffu, flush);
    const unsigned lt = (1u << lane) - 1u;
    const int e = (tail + __popc(fm & lt)) & (QN - 1);
    if (flush) {
        q_key[e] = key;
        uint4 *d = reinterpret_cast<uint4 *>(q_acc + 8 * e);
        d[0] = make_uint4(acc[0], acc[1], acc[2], acc[3]);
        d[1] = make_uint4(acc[4], acc[5], acc[6], acc[7]);
    }
    tail += __popc(fm);
    if (drain_at > 1) {
        // during the strip: whole groups of eight only
        if (tail - head >= drain_at) {
            __syncwarp();
            do {
                drain_group<H, QN>(q_acc, q_key, head, lane, words);
                head += 8;
            } while (tail - head >= 8);
        }
    } else if (tail > head) {
        // the strip's end: everything, the last group partly
        __syncwarp();
        do {
            if (head + (lane >> 2) < tail) drain_group<H, QN>(q_acc, q_key, head, lane, words);
            head += 8;
        } while (tail > head);
        head = tail;
        __syncwarp();
    }
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

// 16 bytes (w[0] holds bytes 0..3, little-endian) -> 16 protein codes, one
// per byte in the same order (`out`), and `bad` with bit i set iff byte i is
// not a letter.  An invalid byte gets code 31: every code fits 5 bits, so a
// rolling shift never carries into the next symbol's field.
__device__ __forceinline__ void encode16_protein(const uint32_t w[4], uint32_t out[4], uint32_t &bad) {
    bad = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t o = 0;
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const uint32_t c = protein_code((w[q] >> (8 * b)) & 0xFFu);
            bad |= (uint32_t)(c >= 26u) << (4 * q + b);
            o |= (c & 31u) << (8 * b);
        }
        out[q] = o;
    }
}

// 64 bases starting at code index ci, as four words w[0..3] (first base in
// bits 31..30 of w[0]).
__device__ __forceinline__ void codes64_at(const uint32_t *codes, int ci, uint32_t w[4]) {
    const int wi = ci >> 4, sh = (ci & 15) * 2;
    uint32_t a[5];
#pragma unroll
    for (int j = 0; j < 5; ++j) a[j] = codes[wi + j];
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = __funnelshift_l(a[j + 1], a[j], sh);
}

// The packed value of bases [b, b+t) of a 64-base window (first base most
// significant): bits [128 - 2(b+t), 128 - 2b) of w[0]:w[1]:w[2]:w[3].  Called
// with b, t that are constants after unrolling, so every index folds.
__device__ __forceinline__ uint32_t wsel(const uint32_t w[4], int i) {
    return (i >= 0 && i < 4) ? w[i] : 0u;
}

__device__ __forceinline__ uint64_t win_value(const uint32_t w[4], int b, int t) {
    const int lo = 128 - 2 * (b + t), nbits = 2 * t;
    const int q = lo >> 5, r = lo & 31;
    const uint32_t lo32 = r ? __funnelshift_r(wsel(w, 3 - q), wsel(w, 2 - q), r) : wsel(w, 3 - q);
    if (nbits <= 32) return nbits == 32 ? (uint64_t)lo32 : (uint64_t)(lo32 & ((1u << nbits) - 1u));
    uint32_t hi32 = r ? __funnelshift_r(wsel(w, 2 - q), wsel(w, 1 - q), r) : wsel(w, 2 - q);
    if (nbits < 64) hi32 &= (1u << (nbits - 32)) - 1u;
    return ((uint64_t)hi32 << 32) | lo32;
}

// x * b for b in {0, 1}: keeps or clears x with one integer multiply-add
// (issued on the FMA pipe, which the logic-heavy loop leaves idle).
__device__ __forceinline__ uint32_t keep_if(uint32_t x, uint32_t b) {
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, 0;" : "=r"(d) : "r"(x), "r"(b));
    return d;
}


// 16-byte asynchronous global -> shared copy through L2 only; the L2 fetches
// the 64 bytes around it rather than a 128-byte line (scattered shards: same
// rate, half the DRAM bytes).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global.L2::64B [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- TMA bulk copy (global -> shared) completed on an mbarrier.
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                 : "=r"(ok)
                 : "r"(smem_u32(bar)), "r"(parity)
                 : "memory");
    return ok != 0;
}
// Bounded wait: false after `polls` polls (by default ~2^22: the copy never
// completed).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, int polls = 1 << 22) {
    for (int it = 0; it < polls; ++it)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

// Hint: bring the 128-byte line holding p into L2 (p must be a valid address).
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

template <int K_, int M_, int S_, int H_, int A_ = 0, int D_ = 0>
struct StripCfg {
    static constexpr int K = K_, M = M_, S = S_, H = H_, A = A_;
    // D > 0: dense batches of fixed-length records of at most D bytes, one
    // record per strip (DNA query); the sizes below are then maxima
    static constexpr int D = D_;
    static constexpr int BITS = A == 0 ? 2 : A == 1 ? 5 : 6;  // bits per symbol
    static constexpr int W = K - M + 1;                 // m-mer windows per k-mer; block length
    static constexpr int Z = K - S;                     // s-mers per k-mer minus one
    // blocks per strip (protein: ~110 k-mers so that four query CTAs fit an
    // SM; triplets: at most 60 per frame pass)
    static constexpr int NB = D > 0 ? (D + W - 1) / W : A == 2 ? 60 / W : A == 1 ? (110 + W - 1) / W
                                                           : (W >= 16) ? 8 : (128 + W - 1) / W;
    static constexpr int L = NB * W;                    // k-mers per thread
    static constexpr int NT = 128;                      // threads per CTA
    static constexpr int TILE = D > 0 ? NT * D : NT * L;  // k-mer positions per tile (multiple of 32)
    static constexpr int TILE_WORDS = TILE / 32;
    static constexpr int CODE_WORDS = (TILE + K + 96) / 16 + 4;  // 16 bases per word
    static constexpr int BIT_WORDS = (CODE_WORDS + 1) / 2 + 2;   // one bit per code index
    static constexpr int SW = 64 / H;                   // bit-slice width (Sec. IV-G)
    // query: staged shards per thread per block (triplets: two, so that four
    // query CTAs fit an SM)
    static constexpr int SLOTS = A == 0 && D == 0 ? 6 : A == 2 ? 2 : 4;
    // Triplets (A = 2): a tile covers BYTE_TILE = 3 * TILE bytes in three frame
    // passes; symbol c of pass f is the codon at byte T0 - OFF + f + 3c.
    static constexpr int BYTE_TILE = A == 2 ? 3 * TILE : TILE;
    static constexpr int OFF = A == 2 ? 48 : 16;        // bytes before T0 (16 symbols)
    static constexpr int CODE_SYMS = 16 * CODE_WORDS;   // symbols per tile (pass)
    // a tile's bytes, staged by one bulk copy
    static constexpr int RAW_BYTES = A == 2 ? ((3 * CODE_SYMS + 4 + 15) / 16) * 16 : 16 * CODE_WORDS;
    static constexpr int BYTE_WORDS = A == 2 ? RAW_BYTES / 32 + 2 : 1;  // byte-space boundary bitmap
    static constexpr int OUT_WORDS = BYTE_TILE / 32;    // answer words per tile
    static_assert(W >= 1 && W <= 32 && Z >= 0 && H >= 1 && H <= kMaxH, "parameters");
    static_assert(A == 0 || BITS * K <= 64, "a k-mer packs into one 64-bit word");
    static_assert(BYTE_TILE % 32 == 0, "tile must cover whole output words");
    static_assert(A != 2 || L <= 64, "a triplet strip's validity bits are read as one 64-bit window");
    static_assert(TILE % 32 == 0, "tile must cover whole output words");
};

template <int K, int M, int S, int H, int A = 0, int D = 0>
struct StripSmem {
    using C = StripCfg<K, M, S, H, A, D>;
    uint32_t codes[A == 0 ? C::CODE_WORDS : 1];  // DNA: 16 2-bit codes per word
    uint16_t bad16[2 * C::BIT_WORDS];   // bit per code index; read as uint32 words
    uint32_t starts[C::BIT_WORDS];      // record-start bit per code index
    uint32_t valid[C::TILE_WORDS + 2];  // validity bit per k-mer of the tile
    uint32_t outw[C::OUT_WORDS + 2];    // query answer bits of the tile
    // triplets: record boundaries by byte, the highest boundary at or below the
    // end of each byte word (relative to T0 - OFF, -1 if none in the tile), the
    // in-frame bit per symbol of the current pass, the last boundary <= T0 - OFF
    uint32_t bstarts[C::BYTE_WORDS];
    int lastb[C::BYTE_WORDS];
    uint32_t frame[A == 2 ? C::BIT_WORDS : 1];
    int64_t prev_start;
    int scan_tmp[4];
    uint32_t need_tmp[4];               // triplets: per warp, residues mod 3 of the boundaries
    uint2 onehot[64];                   // halves of 1 << p, p = 0 .. 63
    uint64_t raw_bar;                                   // completes the raw bulk copy
    int abort_flag;
    alignas(16) unsigned char raw[C::RAW_BYTES];        // the tile's sequence bytes (bulk copy)
    // protein: one 5-bit code per byte; triplets: one 6-bit codon code per symbol of the pass
    alignas(16) uint8_t pcode[A == 0 ? 16 : A == 1 ? C::RAW_BYTES : C::CODE_SYMS];
};


// The H bits of one s-mer hash as eight 32-bit halves (word w -> halves 2w, 2w+1),
// hash i in word i mod 4 (filters with hash-chosen sectors run the
// runtime-parameter kernels).
// kTable: the one-hot halves of a bit position come from a 64-entry shared
// table (tab[p] = halves of 1 << p), one shared load instead of a variable
// 64-bit shift on the ALU pipe (the query and the queued insert gain ~4 % and
// ~1 %; the direct insert on a cached filter loses ~3 % and keeps the shifts).
template <int H, bool kTable>
__device__ __forceinline__ void smer_halves(uint64_t hs, uint32_t m[8], const uint2 *tab) {
    constexpr int SW = 64 / H;
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = 0u;
#pragma unroll
    for (int i = 0; i < H; ++i) {
        uint32_t pos;
        if constexpr (SW >= 6) pos = (uint32_t)(hs >> (i * SW)) & 63u;
        else pos = (uint32_t)((hs * salt_of(i)) >> 58);
        if constexpr (kTable) {
            const uint2 one = tab[pos];
            m[2 * (i & 3)] |= one.x;
            m[2 * (i & 3) + 1] |= one.y;
        } else {
            const uint64_t one = 1ull << pos;
            m[2 * (i & 3)] |= (uint32_t)one;
            m[2 * (i & 3) + 1] |= (uint32_t)(one >> 32);
        }
    }
}

// FQ = 1 (DNA insert only): finished runs leave through the warp's run queue
// (queue_runs), one 32-byte request per run, instead of four 64-bit OR
// reductions from the run's lane.  The library takes it for filters several
// times larger than L2, where every run is a DRAM read-modify-write; it
// costs instructions where the filter is cached.
template <int K, int M, int S, int H, bool kQuery, int A = 0, int D = 0, int FQ = 0>
__global__ void __launch_bounds__(StripCfg<K, M, S, H, A, D>::NT) strip_kernel(LaunchArgs a) {
    using C = StripCfg<K, M, S, H, A, D>;
    constexpr int W = C::W, Z = C::Z, NB = C::NB, L = C::L, NT = C::NT, TILE = C::TILE;
    constexpr int R = C::SLOTS, BITS = C::BITS;
    constexpr int BT = C::BYTE_TILE, OFF = C::OFF, NPASS = A == 2 ? 3 : 1;
    constexpr int64_t kNone = INT64_MIN;
    constexpr uint64_t kMaskM = A == 0 ? 0ull : (1ull << (BITS * M)) - 1ull;
    constexpr uint64_t kMaskS = A == 0 ? 0ull : (1ull << (BITS * S)) - 1ull;
    __shared__ StripSmem<K, M, S, H, A, D> sm;
    // query: shards of the current block's run heads, [slot][half][thread]
    __shared__ __align__(16) uint4 slot_mem[kQuery ? R * 2 * NT : 1];
    // DNA insert with FQ = 1: per warp, a ring of finished runs (shard key,
    // eight half-words) that the warp drains four lanes per run
    constexpr bool kQueue = !kQuery && A == 0 && FQ;
    constexpr int QN = 128;
    __shared__ __align__(16) uint32_t fq_acc[kQueue ? (NT / 32) * QN * 8 : 1];
    __shared__ uint32_t fq_key[kQueue ? (NT / 32) * QN : 1];
    // protein and triplet insert: the cooperative flush's per-warp staging
    constexpr bool kCoopSmem = !kQuery && A != 0;
    __shared__ __align__(16) uint4 cs_acc[kCoopSmem ? (NT / 32) * 64 : 1];
    __shared__ uint32_t cs_key[kCoopSmem ? (NT / 32) * 32 : 1];

    if (*reinterpret_cast<volatile int *>(a.status) & kStatusBadOffsets) return;
    if (a.wait_test > 0) {
        // failure-detection test: a bounded wait that cannot succeed (an
        // mbarrier with one expected arrival that never comes, no copy
        // attached) gives up and is reported as the sticky timeout status
        if (threadIdx.x == 0) {
            mbar_init(&sm.raw_bar, 1);
            if (!mbar_wait(&sm.raw_bar, 0, a.wait_test)) atomicOr(a.status, kStatusTimeout);
        }
        return;
    }
    // dense batches: record r is bytes [r rlen, (r + 1) rlen), a tile holds NT
    // records; the geometry below is runtime there and the constants otherwise.
    // A CSR batch runs dense too when the offsets check found every record of
    // one length rlen (K <= rlen <= D) and its first offset is a multiple of 32
    // (tiles then start on answer-word boundaries, at records).
    int rlen = D > 0 ? (int)a.rec_len : 0;
    if (D > 0 && rlen == 0 && a.nonuniform != nullptr && *a.nonuniform == 0) {
        const int64_t o0 = a.offsets[0], len0 = a.offsets[1] - o0;
        if ((o0 & 31) == 0 && len0 >= K && len0 <= D) rlen = (int)len0;
    }
    const bool dense = D > 0 && rlen > 0;
    const int tile_pos = dense ? NT * rlen : BT;               // positions (bytes) per tile
    const int code_words = dense ? (tile_pos + K + 96) / 16 + 4 : C::CODE_WORDS;
    const int raw_bytes = dense ? 16 * code_words : C::RAW_BYTES;
    const int tile_words = dense ? tile_pos / 32 : C::TILE_WORDS;
    const int strip_len = dense ? rlen : L;
    const int nbl = dense ? (rlen - K + 1 + W - 1) / W : NB;  // blocks per strip
    const int64_t lo = D > 0 && a.rec_len > 0 ? 0 : a.offsets[0];
    const int64_t hi = D > 0 && a.rec_len > 0 ? a.n * (int64_t)rlen : a.offsets[a.n];
    if (hi <= lo) return;
    const int64_t base = lo & ~int64_t(31);
    const int64_t n_tiles = (hi - base + tile_pos - 1) / tile_pos;
    const int tid = threadIdx.x;
    const bool aligned = ((reinterpret_cast<uintptr_t>(a.seq)) & 15u) == 0;
    const uint32_t smask = (uint32_t)a.shard_mask;
    const uint64_t seed_m = a.seed, seed_s = ~a.seed;
    const uint32_t *bad32 = reinterpret_cast<const uint32_t *>(sm.bad16);

    // The bytes of a tile whose 16-aligned span lies inside [lo, hi) arrive by
    // one bulk copy (TMA) issued while the previous tile computes; other tiles
    // (the batch's edges, or an unaligned seq) load their bytes directly.
    auto bulk_ok = [&](int64_t tl) {
        const int64_t a0 = base + tl * tile_pos - OFF;
        return a.device_seq && aligned && a0 >= lo && a0 + raw_bytes <= hi;
    };
    if (tid == 0) {
        mbar_init(&sm.raw_bar, 1);
        sm.abort_flag = 0;
    }

    if ((kQuery || kQueue) && tid < 64)
        sm.onehot[tid] = make_uint2(tid < 32 ? 1u << tid : 0u, tid >= 32 ? 1u << (tid - 32) : 0u);
    __syncthreads();
    uint32_t raw_phase = 0;
    if (tid == 0 && blockIdx.x < n_tiles && bulk_ok(blockIdx.x))
        bulk_load(sm.raw, a.seq + (base + (int64_t)blockIdx.x * tile_pos - OFF), raw_bytes, &sm.raw_bar);

    for (int64_t tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
        const int64_t T0 = base + tile * tile_pos;
        const int64_t A0 = T0 - OFF;  // absolute position of code index 0 (triplets: of byte 0)
        const bool staged = bulk_ok(tile);
        // ---- phase 1 (warps 1..): bases -> codes + invalid bits.
        //      phase 1 (warp 0): record starts inside (T0, T0 + TILE + K - 1),
        //      from a search of the offsets, overlapping the others' encoding.
        if (tid < 32 && A == 2) {
            // triplets: every record boundary in (A0, A0 + RAW_BYTES) by byte,
            // and the last boundary at or below A0
            for (int w = tid; w < C::BYTE_WORDS; w += 32) sm.bstarts[w] = 0u;
            if (tid < 2) sm.valid[C::TILE_WORDS + tid] = 0u;
            const int64_t r0 = warp_find_boundary(a.offsets, a.n, A0, lo, hi, tid);
            if (tid == 0) sm.prev_start = r0 >= 1 ? a.offsets[r0 - 1] : kNone;
            __syncwarp();
            const int64_t lim = A0 + C::RAW_BYTES;
            bool more = true;
            for (int64_t rb = r0; more; rb += 32) {
                const int64_t r = rb + tid;
                const int64_t p = r <= a.n ? a.offsets[r] : lim;
                if (p > A0 && p < lim) atomicOr(&sm.bstarts[(p - A0) >> 5], 1u << ((p - A0) & 31));
                more = __shfl_sync(0xffffffffu, p, 31) < lim && rb + 32 <= a.n;
            }
        } else if (tid < 32 && dense) {
            // dense: record starts at T0 + j rlen (T0 is a multiple of rlen)
            for (int w = tid; w < C::BIT_WORDS; w += 32) sm.starts[w] = 0u;
            if (tid < 2) sm.valid[tile_words + tid] = 0u;
            __syncwarp();
            for (int j = tid + 1; j <= NT + 1; j += 32) {
                const int ci = 16 + j * rlen;
                if (ci < 16 + tile_pos + K - 1) atomicOr(&sm.starts[ci >> 5], 1u << (ci & 31));
            }
        } else if (tid < 32) {
            for (int w = tid; w < C::BIT_WORDS; w += 32) sm.starts[w] = 0u;
            if (tid < 2) sm.valid[C::TILE_WORDS + tid] = 0u;
            const int64_t r0 = warp_find_boundary(a.offsets, a.n, T0, lo, hi, tid);
            __syncwarp();
            const int64_t lim = T0 + TILE + K - 1;
            bool more = true;
            for (int64_t rb = r0; more; rb += 4 * 32) {
                int64_t p[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int64_t r = rb + tid + 32 * j;
                    p[j] = r <= a.n ? a.offsets[r] : lim;
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    if (p[j] < lim) {
                        const int ci = (int)(p[j] - A0);
                        atomicOr(&sm.starts[ci >> 5], 1u << (ci & 31));
                    }
                }
                more = __any_sync(0xffffffffu, p[3] < lim);
            }
        } else {
            if (kQuery)
                for (int w = tid - 32; w < C::OUT_WORDS + 2; w += NT - 32) sm.outw[w] = 0u;
            if (A == 2) {
                // triplets: the raw bytes are the front end's output (codons are
                // formed per frame pass below)
                if (staged) {
                    if (!mbar_wait(&sm.raw_bar, raw_phase)) sm.abort_flag = 1;
                } else {
                    for (int u = tid - 32; u < C::RAW_BYTES; u += NT - 32) {
                        const int64_t pp = A0 + u;
                        sm.raw[u] = (pp >= lo && pp < hi) ? a.seq[pp] : (unsigned char)0;
                    }
                }
            } else if (staged) {
                if (!mbar_wait(&sm.raw_bar, raw_phase)) sm.abort_flag = 1;
                for (int c = tid - 32; c < code_words; c += NT - 32) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(sm.raw + 16 * c);
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                    uint32_t bad;
                    if constexpr (A == 0) {
                        uint32_t code;
                        encode16(w, code, bad);
                        sm.codes[c] = code;
                    } else {
                        uint32_t o[4];
                        encode16_protein(w, o, bad);
                        *reinterpret_cast<uint4 *>(sm.pcode + 16 * c) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                    sm.bad16[c] = (uint16_t)bad;
                }
            } else {
                for (int c = tid - 32; c < code_words; c += NT - 32) {
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
                                const int64_t pp = p0 + 4 * q + b;
                                const uint32_t byte = (pp >= lo && pp < hi) ? (uint32_t)a.seq[pp] : 0u;
                                x |= byte << (8 * b);
                            }
                            w[q] = x;
                        }
                    }
                    uint32_t bad;
                    if constexpr (A == 0) {
                        uint32_t code;
                        encode16(w, code, bad);
                        sm.codes[c] = code;
                    } else {
                        uint32_t o[4];
                        encode16_protein(w, o, bad);
                        *reinterpret_cast<uint4 *>(sm.pcode + 16 * c) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                    sm.bad16[c] = (uint16_t)bad;
                }
            }
            if (A != 2)
                for (int c = code_words + tid - 32; c < 2 * C::BIT_WORDS; c += NT - 32) sm.bad16[c] = 0xFFFFu;
        }
        if (staged) raw_phase ^= 1u;
        if (__syncthreads_or(sm.abort_flag)) {
            if (tid == 0) atomicOr(a.status, kStatusTimeout);
            return;
        }
        // the raw buffer is free again (triplets: after the last frame pass's
        // symbols are formed): start the next tile's copy
        // A tile without a bulk copy (host memory read in place, the batch's
        // edges) gets its bytes prefetched into L2 instead, one 128-byte line
        // per thread and round, clipped to [lo, hi): its direct loads then
        // hit L2 rather than wait on the link.
        auto next_copy = [&]() {
            const int64_t nt = tile + gridDim.x;
            if (nt >= n_tiles) return;
            if (bulk_ok(nt)) {
                if (tid == 0) bulk_load(sm.raw, a.seq + (base + nt * tile_pos - OFF), raw_bytes, &sm.raw_bar);
                return;
            }
            const int64_t b0 = max(base + nt * tile_pos - OFF, lo);
            const int64_t b1 = min(base + nt * tile_pos - OFF + (int64_t)raw_bytes, hi);
            for (int64_t x = (b0 & ~int64_t(127)) + 128 * (int64_t)tid; x < b1; x += 128 * NT)
                prefetch_l2(a.seq + max(x, b0));
        };
        if constexpr (A != 2) next_copy();
        int prev_res = -1;  // triplets: (A0 - last boundary <= A0) mod 3, -1 if none
        if constexpr (A == 2) {
            // highest boundary at or below the end of each byte word (a block
            // max-scan; -1 = none since A0)
            constexpr int PER = (C::BYTE_WORDS + NT - 1) / NT;
            const int lane = tid & 31, warp = tid >> 5;
            int loc[PER];
            int run = -1;
            // a symbol of pass p (byte b = p + 3c) is in frame after a boundary at
            // byte lb iff p = lb mod 3; bit r of `res`: a boundary with lb mod 3 = r
            uint32_t res = 0u;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const int w = tid * PER + j;
                if (w < C::BYTE_WORDS) {
                    const uint32_t x = sm.bstarts[w];
                    if (x) {
                        run = 32 * w + 31 - __clz(x);
                        // bit i of word w is byte 32 w + i, = 2 w + i mod 3
                        const uint32_t cls = ((x & 0x49249249u) ? 1u : 0u) | ((x & 0x92492492u) ? 2u : 0u) |
                                             ((x & 0x24924924u) ? 4u : 0u);
                        const int sh = (2 * w) % 3;
                        res |= ((cls << sh) | (cls >> (3 - sh))) & 7u;
                    }
                }
                loc[j] = run;
            }
            res = __reduce_or_sync(0xffffffffu, res);
            if (lane == 0) sm.need_tmp[warp] = res;
            int incl = run;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, d);
                if (lane >= d) incl = v > incl ? v : incl;
            }
            if (lane == 31) sm.scan_tmp[warp] = incl;
            __syncthreads();
            int carry = -1;
            for (int q = 0; q < warp; ++q) carry = sm.scan_tmp[q] > carry ? sm.scan_tmp[q] : carry;
            const int up = __shfl_up_sync(0xffffffffu, incl, 1);
            if (lane > 0) carry = up > carry ? up : carry;
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const int w = tid * PER + j;
                if (w < C::BYTE_WORDS) sm.lastb[w] = loc[j] > carry ? loc[j] : carry;
            }
            if (sm.prev_start != kNone) prev_res = (int)((A0 - sm.prev_start) % 3);
            __syncthreads();
        }

        for (int pass = 0; pass < NPASS; ++pass) {
        if constexpr (A == 2) {
            // a pass none of whose symbols is in frame holds no valid k-mer and
            // is skipped (block-uniform): pass p is in frame after a boundary
            // at byte lb iff p = lb mod 3 (need_tmp), and before the tile's
            // first boundary iff p + prev_res = 0 mod 3
            const uint32_t need = sm.need_tmp[0] | sm.need_tmp[1] | sm.need_tmp[2] | sm.need_tmp[3] |
                                  (prev_res >= 0 ? 1u << ((3 - prev_res) % 3) : 0u);
            if (!((need >> pass) & 1u)) {
                if (pass == NPASS - 1) next_copy();
                continue;
            }
        }
        if constexpr (A == 2) {
            // ---- phase 2 (triplets): symbol c of this pass is the codon at byte
            // b = pass + 3c; invalid if a base is invalid or a record boundary
            // falls inside it; `starts` marks a boundary at b; `frame` marks b
            // in frame (the last boundary at or below b is a multiple of 3 back)
            const int lane = tid & 31;
            for (int c0 = (tid >> 5) * 32; c0 < 32 * C::BIT_WORDS; c0 += NT) {
                const int c = c0 + lane;
                uint32_t code = 63u;
                bool bad = true, at = false, fr = false;
                if (c < C::CODE_SYMS) {
                    const int b = pass + 3 * c;
                    const int x = base_code(sm.raw[b]), y = base_code(sm.raw[b + 1]), z = base_code(sm.raw[b + 2]);
                    const uint32_t wb = sm.bstarts[b >> 5];
                    const uint64_t two = (uint64_t)wb | ((uint64_t)sm.bstarts[(b >> 5) + 1] << 32);
                    const bool inner = ((two >> ((b & 31) + 1)) & 3ull) != 0;
                    bad = (x | y | z) < 0 || inner;
                    if (!bad) code = (uint32_t)(x * 16 + y * 4 + z);
                    at = (wb >> (b & 31)) & 1u;
                    const uint32_t below = wb & (0xFFFFFFFFu >> (31 - (b & 31)));
                    const int lb = below ? 32 * (b >> 5) + 31 - __clz(below)
                                         : ((b >> 5) > 0 ? sm.lastb[(b >> 5) - 1] : -1);
                    fr = lb >= 0 ? (b - lb) % 3 == 0 : (prev_res >= 0 && (b + prev_res) % 3 == 0);
                    sm.pcode[c] = (uint8_t)code;
                }
                const unsigned bw = __ballot_sync(0xffffffffu, bad);
                const unsigned aw = __ballot_sync(0xffffffffu, at);
                const unsigned fw = __ballot_sync(0xffffffffu, fr);
                if (lane == 0) {
                    reinterpret_cast<uint32_t *>(sm.bad16)[c0 >> 5] = bw;
                    sm.starts[c0 >> 5] = aw;
                    sm.frame[c0 >> 5] = fw;
                }
            }
            __syncthreads();
            if (pass == NPASS - 1) next_copy();
        }
        // ---- phase 3: validity bit per k-mer: no invalid base in its k bases,
        // no record start among its bases 1 .. k-1 (triplets: and in frame).
        for (int v = tid; v < tile_words; v += NT) {
            const uint64_t badw = bits64_at(bad32, 32 * v + 16);
            const uint64_t stw = bits64_at(sm.starts, 32 * v + 17);
            uint32_t ok = ~(window_or<K>(badw) | window_or<K - 1>(stw));
            if constexpr (A == 2) ok &= (uint32_t)bits64_at(sm.frame, 32 * v + 16);
            sm.valid[v] = ok;
        }
        __syncthreads();

        // ---- phase 4: strips
        const int kk0 = tid * strip_len;  // first k-mer of this thread (tile relative)
        // (triplets: the strip's first k-mer starts at byte T0 + pass + 3 kk0)
        const bool own = T0 + (A == 2 ? pass + 3 * kk0 : kk0) < hi;
        bool go = own;
        if constexpr (A == 2) {
            // a warp skips a frame pass in which none of its strips holds a
            // valid k-mer (inside one long record, two passes of three are out
            // of frame)
            // (every lane votes: a lane without a strip must not skip the vote)
            const bool has = own && (bits64_at(sm.valid, kk0) & ((1ull << L) - 1ull)) != 0;
            const bool any = __any_sync(0xffffffffu, has);
            go = own && any;
        }
        // the lanes that run a strip, from a vote of the whole warp (the
        // member mask of the cooperative flushes)
        const unsigned am = __ballot_sync(0xffffffffu, go);
        if (go) {
            // m-mer u of the strip starts at code index kk0 + 15 + u; the strip's
            // k-mers are u = 1 .. L (k-mer kk0 + u - 1 starts at code index kk0 + 16 + u - 1).
            uint64_t suf[W];
            uint32_t shard[W];
            uint32_t mk[Z + 1][8];
#pragma unroll
            for (int i = 0; i < W; ++i) {
                suf[i] = ~0ull;
                shard[i] = 0u;
            }
            // the first Z s-mers of the strip's first k-mer.  Protein: vb rolls
            // the s-mers (the last s symbols appended), va the m-mers.
            uint64_t va = 0, vb = 0;
            {
                if constexpr (A == 0) {
                    uint32_t wv[4];
                    codes64_at(sm.codes, kk0 + 16, wv);
#pragma unroll
                    for (int z = 0; z < Z; ++z)
                        smer_halves<H, kQuery || kQueue>(hash_smer(win_value(wv, z, S), seed_s), mk[z + 1], sm.onehot);
                } else {
#pragma unroll
                    for (int i = 0; i < S - 1; ++i) vb = (vb << BITS) | sm.pcode[kk0 + 16 + i];
#pragma unroll
                    for (int z = 0; z < Z; ++z) {
                        vb = (vb << BITS) | sm.pcode[kk0 + 16 + z + S - 1];
                        smer_halves<H, kQuery || kQueue>(hash_smer(vb & kMaskS, seed_s), mk[z + 1], sm.onehot);
                    }
#pragma unroll
                    for (int i = 0; i < M - 1; ++i) va = (va << BITS) | sm.pcode[kk0 + 15 + i];
                }
#pragma unroll
                for (int j = 0; j < 8; ++j) mk[0][j] = 0u;
            }
            // run / answer state.  Insert keys a k-mer's run by its shard with bit
            // 31 set when the k-mer is invalid (shards are < 2^31 here), so an
            // invalid k-mer never matches a valid run and a run is flushed only
            // if its key is valid.
            uint32_t cur_key = 0x80000000u;
            uint32_t acc[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) acc[j] = 0u;
            uint64_t F0 = 0, F1 = 0, F2 = 0, F3 = 0;
            uint64_t *const words = a.words;
            int q_head = 0, q_tail = 0;  // DNA insert: the warp's run queue (warp-uniform)

#pragma unroll 1
            for (int blk = 0; blk <= nbl; ++blk) {
                // -- pass A: m-mers u = blk*W .. blk*W + W-1; emits the keys of
                //    k-mers u = (blk-1)*W + 1 .. blk*W (the strip's block blk-1).
                //    Query: every run head's shard is copied to a slot (cp.async)
                //    and flagged in `heads`.
                int nh = 0;
                uint32_t heads = 0;
                const uint32_t last_before = shard[W - 1];

                const int kb = kk0 + (blk - 1) * W;
                uint64_t vwin = 0;
                if (blk > 0) vwin = bits64_at(sm.valid, kb);
                {
                    uint32_t wv[4];
                    if constexpr (A == 0) codes64_at(sm.codes, kk0 + 15 + blk * W, wv);
                    uint64_t h[W];
                    uint64_t pre = ~0ull;
#pragma unroll
                    for (int i = 0; i < W; ++i) {
                        uint64_t mv;
                        if constexpr (A == 0) {
                            mv = win_value(wv, i, M);
                        } else {
                            va = (va << BITS) | sm.pcode[kk0 + 15 + blk * W + i + M - 1];
                            mv = va & kMaskM;
                        }
                        h[i] = hash_minimizer(mv, seed_m);
                        pre = h[i] < pre ? h[i] : pre;
                        if (i < W - 1) {
                            const uint64_t mu = suf[i + 1] < pre ? suf[i + 1] : pre;
                            shard[i] = (uint32_t)mu & smask;
                            if (kQuery && blk > 0) {
                                const bool head = (i == 0) ? (blk == 1 || shard[0] != last_before)
                                                           : (shard[i] != shard[i - 1]);
                                if (head) {
                                    heads |= 1u << i;
                                    const uint64_t *src = words + (uint64_t)shard[i] * 4;
                                    if (nh < R) {
                                        cp_async16(smem_u32(&slot_mem[(nh * 2 + 0) * NT + tid]), src);
                                        cp_async16(smem_u32(&slot_mem[(nh * 2 + 1) * NT + tid]), src + 2);
                                    } else {
                                        prefetch_l2(src);
                                    }
                                    ++nh;
                                }
                            }
                        }
                    }
                    if (kQuery) cp_async_commit();
                    suf[W - 1] = h[W - 1];
#pragma unroll
                    for (int i = W - 2; i >= 0; --i) suf[i] = h[i] < suf[i + 1] ? h[i] : suf[i + 1];
                    shard[W - 1] = (uint32_t)suf[0] & smask;
                    if (kQuery && blk > 0) {
                        const bool head = (W == 1) ? (blk == 1 || shard[0] != last_before)
                                                   : (shard[W - 1] != shard[W > 1 ? W - 2 : 0]);
                        if (head) {
                            heads |= 1u << (W - 1);
                            const uint64_t *src = words + (uint64_t)shard[W - 1] * 4;
                            if (nh < R) {
                                cp_async16(smem_u32(&slot_mem[(nh * 2 + 0) * NT + tid]), src);
                                cp_async16(smem_u32(&slot_mem[(nh * 2 + 1) * NT + tid]), src + 2);
                            } else {
                                prefetch_l2(src);
                            }
                        }
                    }
                    if (kQuery) cp_async_commit();
                }
                if (blk == 0) continue;
                // -- pass B: k-mers kk = kb + i; the newest s-mer of k-mer kk starts at
                //    code index kk + 16 + Z.
                {
                    uint32_t wv[4];
                    if constexpr (A == 0) codes64_at(sm.codes, kb + 16 + Z, wv);
                    uint32_t present = 0;
                    int nb = 0;
                    if (kQuery) cp_async_wait<1>();
#pragma unroll
                    for (int i = 0; i < W; ++i) {
#pragma unroll
                        for (int z = 0; z < Z; ++z)
#pragma unroll
                            for (int j = 0; j < 8; ++j) mk[z][j] = mk[z + 1][j];
                        uint64_t sv;
                        if constexpr (A == 0) {
                            sv = win_value(wv, i, S);
                        } else {
                            vb = (vb << BITS) | sm.pcode[kb + 16 + Z + i + S - 1];
                            sv = vb & kMaskS;
                        }
                        smer_halves<H, kQuery || kQueue>(hash_smer(sv, seed_s), mk[Z], sm.onehot);
                        // OR of the k-mer's older s-mers (its newest is mk[Z])
                        uint32_t older[8];
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            uint32_t x = 0u;
#pragma unroll
                            for (int z = 0; z < Z; ++z) x |= mk[z][j];
                            older[j] = x;
                        }
                        if (!kQuery) {
                            const uint32_t key = shard[i] | ((((uint32_t)(vwin >> i)) & 1u) ^ 1u) << 31;
                            // DNA (runs of ~(w+1)/2 = 8.5 k-mers): each lane flushes its own
                            // runs; protein (runs of ~3): the warp flushes cooperatively
                            if constexpr (kQueue) {
                                const bool fl = key != cur_key && !(cur_key >> 31);
                                if (am == 0xffffffffu)
                                    queue_runs<H, QN>(fq_acc + (tid >> 5) * QN * 8, fq_key + (tid >> 5) * QN, q_head,
                                                      q_tail, fl, cur_key, acc, tid & 31, 8, words);
                                else if (fl)
                                    flush_run<H>(words + (uint64_t)cur_key * 4, acc);
                            } else if constexpr (A == 0) {
                                if (key != cur_key && !(cur_key >> 31)) flush_run<H>(words + (uint64_t)cur_key * 4, acc);
                            } else {
                                flush_coop<H>(words, cur_key, acc, key != cur_key && !(cur_key >> 31), am,
                                              cs_key + (tid >> 5) * 32, cs_acc + (tid >> 5) * 64);
                            }
                            const uint32_t same = key == cur_key ? 1u : 0u;
#pragma unroll
                            for (int j = 0; j < 8; ++j) acc[j] = keep_if(acc[j], same) | older[j] | mk[Z][j];
                            cur_key = key;
                        } else {
                            if (i == W - 1) cp_async_wait<0>();
                            if ((heads >> i) & 1u) {
                                const int sl = nb < R ? nb : R - 1;
                                head_shard(F0, F1, F2, F3, smem_u32(&slot_mem[(sl * 2 + 0) * NT + tid]),
                                           smem_u32(&slot_mem[(sl * 2 + 1) * NT + tid]),
                                           words + (uint64_t)shard[i] * 4, nb < R);
                                ++nb;
                            }
                            const uint32_t f[8] = {(uint32_t)F0, (uint32_t)(F0 >> 32), (uint32_t)F1,
                                                   (uint32_t)(F1 >> 32), (uint32_t)F2, (uint32_t)(F2 >> 32),
                                                   (uint32_t)F3, (uint32_t)(F3 >> 32)};
                            uint32_t miss = 0u;
#pragma unroll
                            for (int j = 0; j < 8; ++j) miss |= (older[j] | mk[Z][j]) & ~f[j];
                            present |= (miss == 0u ? 1u : 0u) << i;
                        }
                    }
                    // only valid k-mers answer (one AND for the block)
                    if (kQuery) present &= (uint32_t)vwin & (W >= 32 ? 0xFFFFFFFFu : ((1u << W) - 1u));
                    if (kQuery && present) {
                        if constexpr (A == 2) {
                            // k-mer kb + i starts at tile byte pass + 3 (kb + i)
                            for (uint32_t pm = present; pm; pm &= pm - 1u) {
                                const int rb = pass + 3 * (kb + __ffs(pm) - 1);
                                atomicOr(&sm.outw[rb >> 5], 1u << (rb & 31));
                            }
                        } else {
                            const int wi = kb >> 5, sh = kb & 31;
                            atomicOr(&sm.outw[wi], present << sh);
                            if (sh + W > 32) atomicOr(&sm.outw[wi + 1], (uint32_t)((uint64_t)present >> (32 - sh)));
                        }
                    }
                }
            }
            if constexpr (!kQuery) {
                if constexpr (kQueue) {
                    // the strip's last runs, then everything still queued
                    if (am == 0xffffffffu)
                        queue_runs<H, QN>(fq_acc + (tid >> 5) * QN * 8, fq_key + (tid >> 5) * QN, q_head, q_tail,
                                          !(cur_key >> 31), cur_key, acc, tid & 31, 1, words);
                    else if (!(cur_key >> 31))
                        flush_run<H>(words + (uint64_t)cur_key * 4, acc);
                } else if constexpr (A == 0) {
                    if (!(cur_key >> 31)) flush_run<H>(words + (uint64_t)cur_key * 4, acc);
                } else {
                    flush_coop<H>(words, cur_key, acc, !(cur_key >> 31), am, cs_key + (tid >> 5) * 32,
                                  cs_acc + (tid >> 5) * 64);
                }
            }
        }
        __syncthreads();
        }  // frame passes
        if (kQuery) {
            const int64_t w_lo = lo >> 5, w_hi = min((hi + 31) >> 5, a.out_words_end);
            for (int w = tid; w < (dense ? tile_words : C::OUT_WORDS); w += NT) {
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

template <int K, int M, int S, int H, int A = 0>
inline StripEntry strip_entry() {
    return StripEntry{K, M, S, H, reinterpret_cast<const void *>(&strip_kernel<K, M, S, H, false, A>),
                      reinterpret_cast<const void *>(&strip_kernel<K, M, S, H, true, A>),
                      StripCfg<K, M, S, H, A>::NT};
}

}  // namespace sbf
