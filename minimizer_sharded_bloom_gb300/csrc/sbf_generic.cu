// sbf_generic.cu -- runtime-parameter SBF kernels (any 1 <= m, s <= k <= 32,
// 1 <= H <= 32; CSR batches or dense batches of fixed-length records), used
// for (k, m, s, H) combinations that have no compile-time specialised kernel.
// One thread per k-mer position, following the paper's Algorithm 1 (insert)
// and Algorithm 2 (query) directly: pack the k-mer, take the minimum minimizer
// hash over its k-m+1 m-mers, OR or test the bits of its k-s+1 s-mers
// ("cuSBF", Sec. IV-D, IV-E).
//
// Work layout: a grid-stride loop over 32-position chunks aligned to absolute
// position multiples of 32, one warp per chunk, so that each query answer word
// is produced by exactly one warp with one __ballot_sync.
#include "sbf_device.cuh"
#include "sbf_kernels.h"

namespace sbf {
namespace {

template <bool kQuery>
__global__ void __launch_bounds__(256) generic_kernel(LaunchArgs a) {
    if (*reinterpret_cast<volatile int *>(a.status) & kStatusBadOffsets) return;
    const int64_t lo = a.rec_len ? 0 : a.offsets[0], hi = a.rec_len ? a.n * a.rec_len : a.offsets[a.n];
    if (hi <= lo) return;
    const int lane = threadIdx.x & 31;
    const int64_t warp = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) >> 5;
    const int64_t n_warps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const uint64_t mask_m = low_mask(a.m), mask_s = low_mask(a.s);
    const uint64_t seed_s = ~a.seed;
    for (int64_t w0 = (lo & ~int64_t(31)) + warp * 32; w0 < hi; w0 += n_warps * 32) {
        const int64_t g = w0 + lane;
        bool valid = false;
        uint64_t shard = 0, K[4] = {0, 0, 0, 0};
        if (g >= lo && g < hi) {
            // the end of the record holding g (first r with offsets[r + 1] > g)
            int64_t rec_end;
            if (a.rec_len) {
                rec_end = (g / a.rec_len + 1) * a.rec_len;
            } else {
                int64_t r_lo = 0, r_hi = a.n - 1;
                while (r_lo < r_hi) {
                    const int64_t mid = r_lo + ((r_hi - r_lo) >> 1);
                    if (a.offsets[mid + 1] > g) r_hi = mid; else r_lo = mid + 1;
                }
                rec_end = a.offsets[r_lo + 1];
            }
            if (g + a.k <= rec_end) {
                uint64_t kv = 0;
                bool ok = true;
                for (int i = 0; i < a.k; ++i) {
                    const int c = base_code(a.seq[g + i]);
                    ok &= c >= 0;
                    kv = (kv << 2) | (uint64_t)(c & 3);
                }
                if (ok) {
                    uint64_t mu = ~0ull;
                    for (int i = 0; i <= a.k - a.m; ++i) {
                        const uint64_t x = (kv >> (2 * (a.k - a.m - i))) & mask_m;
                        const uint64_t h = hash_minimizer(x, a.seed);
                        mu = h < mu ? h : mu;
                    }
                    shard = mu & a.shard_mask;
                    for (int j = 0; j <= a.k - a.s; ++j) {
                        const uint64_t y = (kv >> (2 * (a.k - a.s - j))) & mask_s;
                        smer_bits_runtime(hash_smer(y, seed_s), a.H, K, a.sectors);
                    }
                    valid = true;
                }
            }
        }
        if (kQuery) {
            bool present = false;
            if (valid) {
                const uint64_t *F = a.words + shard * 4;
                present = ((K[0] & ~__ldg(F + 0)) | (K[1] & ~__ldg(F + 1)) |
                           (K[2] & ~__ldg(F + 2)) | (K[3] & ~__ldg(F + 3))) == 0;
            }
            const unsigned bits = __ballot_sync(0xffffffffu, present);
            if (lane == 0 && (w0 >> 5) < a.out_words_end) a.out[w0 >> 5] = bits;
        } else if (valid) {
            uint64_t *F = a.words + shard * 4;
#pragma unroll
            for (int w = 0; w < 4; ++w)
                if (K[w]) atomicOr(reinterpret_cast<unsigned long long *>(F + w), K[w]);
        }
    }
}

}  // namespace

const void *generic_insert_kernel() { return reinterpret_cast<const void *>(&generic_kernel<false>); }
const void *generic_query_kernel() { return reinterpret_cast<const void *>(&generic_kernel<true>); }

// One thread per offsets pair; sets the sticky status on a decreasing pair or
// a negative first offset.  With `nonuniform` (zeroed by the caller), also
// flags a record whose length differs from the first record's.
__global__ void check_offsets_kernel(const int64_t *off, int64_t n, int *status, int *nonuniform) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t len0 = off[1] - off[0];
    bool bad = false, uneven = false;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t d = off[i + 1] - off[i];
        bad |= d < 0;
        uneven |= d != len0;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) bad |= off[0] < 0;
    const bool any_bad = __any_sync(0xffffffffu, bad);
    const bool any_uneven = __any_sync(0xffffffffu, uneven);
    if ((threadIdx.x & 31) == 0) {
        if (any_bad) atomicOr(status, kStatusBadOffsets);
        if (any_uneven && nonuniform) atomicOr(nonuniform, 1);
    }
}

}  // namespace sbf
