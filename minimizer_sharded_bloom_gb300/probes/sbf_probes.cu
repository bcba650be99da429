// sbf_probes.cu -- micro-benchmarks of the ceilings that bound the Super Bloom
// filter kernels on the GPU they run on (declared in include/sbf_probes.h).
//
// The insert on a filter larger than L2 is bound by scattered 32-byte
// read-modify-writes of its shards, one per run of k-mers that share a
// minimizer; the query by scattered 32-byte shard reads and by its integer
// instruction mix ("cuSBF", Sec. IV-D/E, Sec. V-F and Fig. 7).  These kernels
// measure each of those alone: no k-mer work, rows drawn by a counter-based
// generator (no index array to read).
#include <cuda_runtime.h>

#include <cstdint>

#include "sbf_probes.h"

namespace {

// SplitMix64's output function (Steele, Lea, Flood 2014), used as a
// counter-based generator of row indices.
__device__ __forceinline__ uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

constexpr int kAluSteps = 8;   // steps per round, unrolled
constexpr int kAluChains = 8;  // independent chains per thread

template <int KIND>
__device__ __forceinline__ void alu_step(uint32_t &x, uint32_t &y, uint32_t &z) {
    if constexpr (KIND == 0) {
        // LOP3, funnel shift, compare + select, min
        asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(x) : "r"(y), "r"(z));
        asm volatile("shf.l.wrap.b32 %0, %0, %1, 7;" : "+r"(y) : "r"(x));
        asm volatile("{ .reg .pred p; setp.lt.u32 p, %0, 0x9E3779B9; selp.b32 %1, %2, %1, p; }"
                     : "+r"(x), "+r"(z) : "r"(y));
        asm volatile("min.u32 %0, %0, %1;" : "+r"(x) : "r"(z));
    } else if constexpr (KIND == 1) {
        asm volatile("lop3.b32 %0, %0, %1, %2, 0x96;" : "+r"(x) : "r"(y), "r"(z));
        asm volatile("lop3.b32 %0, %0, %1, %2, 0xE8;" : "+r"(y) : "r"(z), "r"(x));
        asm volatile("lop3.b32 %0, %0, %1, %2, 0x6A;" : "+r"(z) : "r"(x), "r"(y));
    } else if constexpr (KIND == 2) {
        asm volatile("shf.l.wrap.b32 %0, %0, %1, 5;" : "+r"(x) : "r"(y));
        asm volatile("shf.l.wrap.b32 %0, %0, %1, 11;" : "+r"(y) : "r"(z));
        asm volatile("shf.l.wrap.b32 %0, %0, %1, 17;" : "+r"(z) : "r"(x));
    } else if constexpr (KIND == 3) {
        asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(x) : "r"(y), "r"(z));
        asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(y) : "r"(z), "r"(x));
        asm volatile("mad.lo.u32 %0, %0, %1, %2;" : "+r"(z) : "r"(x), "r"(y));
    } else {
        // 64-bit unsigned minimum of (x:y) and (z:x), three per step
        asm volatile("{ .reg .b64 a, b; mov.b64 a, {%0, %1}; mov.b64 b, {%2, %0}; min.u64 a, a, b;"
                     " mov.b64 {%0, %1}, a; }" : "+r"(x), "+r"(y) : "r"(z));
        asm volatile("{ .reg .b64 a, b; mov.b64 a, {%0, %1}; mov.b64 b, {%2, %1}; min.u64 a, a, b;"
                     " mov.b64 {%0, %1}, a; }" : "+r"(y), "+r"(z) : "r"(x));
        asm volatile("{ .reg .b64 a, b; mov.b64 a, {%0, %1}; mov.b64 b, {%1, %2}; min.u64 a, a, b;"
                     " mov.b64 {%0, %1}, a; }" : "+r"(z), "+r"(x) : "r"(y));
    }
}

constexpr int alu_ops_per_step(int kind) { return kind == 0 ? 5 : 3; }

template <int KIND>
__global__ void __launch_bounds__(1024) probe_alu_kernel(int iters, uint32_t *sink) {
    const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    uint32_t x[kAluChains], y[kAluChains], z[kAluChains];
#pragma unroll
    for (int c = 0; c < kAluChains; ++c) {
        x[c] = t * 0x9E3779B9u + (uint32_t)c;
        y[c] = (t ^ ((uint32_t)c * 0x85EBCA6Bu)) | 1u;
        z[c] = t + 0x27D4EB2Fu * (uint32_t)(c + 1);
    }
#pragma unroll 1
    for (int it = 0; it < iters; ++it) {
#pragma unroll
        for (int u = 0; u < kAluSteps; ++u)
#pragma unroll
            for (int c = 0; c < kAluChains; ++c) alu_step<KIND>(x[c], y[c], z[c]);
    }
    uint32_t r = 0;
#pragma unroll
    for (int c = 0; c < kAluChains; ++c) r ^= x[c] + y[c] + z[c];
    sink[t] = r;
}

template <int MODE>
__global__ void __launch_bounds__(1024) probe_rmw_kernel(uint64_t *buf, uint64_t row_mask, int64_t n_updates,
                                                         uint64_t seed) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if constexpr (MODE == 3) {
        // each thread makes one row per round and queues it (row, four words)
        // in its warp's shared-memory area; the warp then drains the 32 rows
        // with lane l writing word l & 3 of row 8 t + (l >> 2) in trip t
        __shared__ uint64_t q_word[32][32][4];
        __shared__ uint64_t q_row[32][32];
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        for (int64_t u0 = tid - lane; u0 < n_updates; u0 += stride) {
            const int64_t u = u0 + lane;
            const bool have = u < n_updates;
            const uint64_t h = mix64(seed + (uint64_t)u);
#pragma unroll
            for (int w = 0; w < 4; ++w) q_word[warp][lane][w] = have ? 1ull << ((h >> (34 + 6 * w)) & 63u) : 0ull;
            q_row[warp][lane] = h & row_mask;
            __syncwarp();
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int e = 8 * t + (lane >> 2), w = lane & 3;
                const uint64_t v = q_word[warp][e][w];
                if (v)
                    asm volatile("red.global.or.b64 [%0], %1;" ::"l"(buf + q_row[warp][e] * 4 + w), "l"(v) : "memory");
            }
            __syncwarp();
        }
    } else if constexpr (MODE == 1) {
        // four consecutive lanes per row, one word each
        for (int64_t t = tid; t < 4 * n_updates; t += stride) {
            const uint64_t h = mix64(seed + (uint64_t)(t >> 2));
            const int w = (int)(t & 3);
            const uint64_t v = 1ull << ((h >> (34 + 6 * w)) & 63u);
            asm volatile("red.global.or.b64 [%0], %1;" ::"l"(buf + (h & row_mask) * 4 + w), "l"(v) : "memory");
        }
    } else {
        for (int64_t u = tid; u < n_updates; u += stride) {
            const uint64_t h = mix64(seed + (uint64_t)u);
            uint64_t *row = buf + (h & row_mask) * 4;
            uint64_t v[4];
#pragma unroll
            for (int w = 0; w < 4; ++w) v[w] = 1ull << ((h >> (34 + 6 * w)) & 63u);
            if constexpr (MODE == 0) {
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    asm volatile("red.global.or.b64 [%0], %1;" ::"l"(row + w), "l"(v[w]) : "memory");
            } else {
                uint64_t a, b, c, d;
                asm volatile("ld.global.v4.u64 {%0, %1, %2, %3}, [%4];"
                             : "=l"(a), "=l"(b), "=l"(c), "=l"(d)
                             : "l"(row));
                asm volatile("st.global.v4.u64 [%0], {%1, %2, %3, %4};" ::"l"(row), "l"(a | v[0]), "l"(b | v[1]),
                             "l"(c | v[2]), "l"(d | v[3])
                             : "memory");
            }
        }
    }
}

constexpr int kReadsInFlight = 8;

template <int MODE>
__device__ __forceinline__ void load_row(const uint64_t *p, uint64_t &a, uint64_t &b, uint64_t &c, uint64_t &d) {
    if constexpr (MODE == 0)
        asm volatile("ld.global.nc.v4.u64 {%0, %1, %2, %3}, [%4];" : "=l"(a), "=l"(b), "=l"(c), "=l"(d) : "l"(p));
    else if constexpr (MODE == 1)
        asm volatile("ld.global.nc.L2::64B.v4.u64 {%0, %1, %2, %3}, [%4];"
                     : "=l"(a), "=l"(b), "=l"(c), "=l"(d)
                     : "l"(p));
    else if constexpr (MODE == 2)
        asm volatile("ld.global.nc.L2::128B.v4.u64 {%0, %1, %2, %3}, [%4];"
                     : "=l"(a), "=l"(b), "=l"(c), "=l"(d)
                     : "l"(p));
    else
        asm volatile("ld.global.nc.L2::256B.v4.u64 {%0, %1, %2, %3}, [%4];"
                     : "=l"(a), "=l"(b), "=l"(c), "=l"(d)
                     : "l"(p));
}

template <int MODE>
__device__ __forceinline__ void cp_row(uint32_t dst, const uint64_t *p) {
    if constexpr (MODE == 4) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(p) : "memory");
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 16), "l"(p + 2) : "memory");
    } else {
        asm volatile("cp.async.cg.shared.global.L2::64B [%0], [%1], 16;" ::"r"(dst), "l"(p) : "memory");
        asm volatile("cp.async.cg.shared.global.L2::64B [%0], [%1], 16;" ::"r"(dst + 16), "l"(p + 2) : "memory");
    }
}

template <int MODE>
__global__ void __launch_bounds__(256) probe_read_kernel(const uint64_t *buf, uint64_t row_mask, int64_t n_reads,
                                                          uint64_t seed, uint64_t *sink) {
    extern __shared__ __align__(16) unsigned char slots[];  // cp.async modes: kReadsInFlight x 32 B per thread
    const int64_t stride = (int64_t)gridDim.x * blockDim.x * kReadsInFlight;
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    uint64_t acc = 0;
    uint32_t phase = 0;
    if constexpr (MODE == 6) {
        uint64_t *bars = reinterpret_cast<uint64_t *>(slots + blockDim.x * kReadsInFlight * 32);
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(
                         static_cast<uint32_t>(__cvta_generic_to_shared(bars + threadIdx.x)))
                     : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
#pragma unroll 1
    for (int64_t base = tid * kReadsInFlight; base < n_reads; base += stride) {
        if constexpr (MODE <= 3) {
            uint64_t v[kReadsInFlight][4];
#pragma unroll
            for (int j = 0; j < kReadsInFlight; ++j) {
                const uint64_t h = mix64(seed + (uint64_t)(base + j));
                if (base + j < n_reads) {
                    load_row<MODE>(buf + (h & row_mask) * 4, v[j][0], v[j][1], v[j][2], v[j][3]);
                } else {
                    v[j][0] = v[j][1] = v[j][2] = v[j][3] = 0;
                }
            }
#pragma unroll
            for (int j = 0; j < kReadsInFlight; ++j) acc ^= v[j][0] ^ v[j][1] ^ v[j][2] ^ v[j][3];
        } else if constexpr (MODE == 6) {
            // one 32-byte bulk copy (TMA) per row into this thread's slots,
            // completed on this thread's own mbarrier
            uint64_t *bars = reinterpret_cast<uint64_t *>(slots + blockDim.x * kReadsInFlight * 32);
            const uint32_t bar = static_cast<uint32_t>(__cvta_generic_to_shared(bars + threadIdx.x));
            const uint32_t s0 = static_cast<uint32_t>(__cvta_generic_to_shared(slots)) +
                                threadIdx.x * kReadsInFlight * 32u;
            int cnt = 0;
#pragma unroll
            for (int j = 0; j < kReadsInFlight; ++j) cnt += base + j < n_reads;
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(32 * cnt)
                         : "memory");
#pragma unroll
            for (int j = 0; j < kReadsInFlight; ++j) {
                const uint64_t h = mix64(seed + (uint64_t)(base + j));
                if (base + j < n_reads)
                    asm volatile(
                        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 32, [%2];" ::"r"(
                            s0 + 32u * j),
                        "l"(buf + (h & row_mask) * 4), "r"(bar)
                        : "memory");
            }
            bool done = false;
            for (int it = 0; it < (1 << 22) && !done; ++it) {
                uint32_t ok;
                asm volatile(
                    "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
                    : "=r"(ok)
                    : "r"(bar), "r"(phase)
                    : "memory");
                done = ok != 0;
            }
            if (!done) {
                // the copies never completed: leave a marker and stop
                sink[tid] = ~0ull;
                return;
            }
            phase ^= 1u;
            const uint4 *mine = reinterpret_cast<const uint4 *>(slots + threadIdx.x * kReadsInFlight * 32);
#pragma unroll
            for (int j = 0; j < kReadsInFlight; ++j) {
                if (base + j < n_reads) {
                    const uint4 lo = mine[2 * j], hi = mine[2 * j + 1];
                    acc ^= ((uint64_t)(lo.x ^ hi.x) << 32) ^ (lo.y ^ hi.y) ^ lo.z ^ hi.z ^ lo.w ^ hi.w;
                }
            }
        } else {
            const uint32_t s0 = static_cast<uint32_t>(__cvta_generic_to_shared(slots)) +
                                threadIdx.x * kReadsInFlight * 32u;
#pragma unroll
            for (int j = 0; j < kReadsInFlight; ++j) {
                const uint64_t h = mix64(seed + (uint64_t)(base + j));
                if (base + j < n_reads) cp_row<MODE>(s0 + 32u * j, buf + (h & row_mask) * 4);
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
            asm volatile("cp.async.wait_group 0;" ::: "memory");
            const uint4 *mine = reinterpret_cast<const uint4 *>(slots + threadIdx.x * kReadsInFlight * 32);
#pragma unroll
            for (int j = 0; j < kReadsInFlight; ++j) {
                if (base + j < n_reads) {
                    const uint4 lo = mine[2 * j], hi = mine[2 * j + 1];
                    acc ^= ((uint64_t)(lo.x ^ hi.x) << 32) ^ (lo.y ^ hi.y) ^ lo.z ^ hi.z ^ lo.w ^ hi.w;
                }
            }
        }
    }
    sink[tid] = acc;
}

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

bool pow2(uint64_t x) { return x && !(x & (x - 1)); }

int launched() { return cudaGetLastError() == cudaSuccess ? 0 : -2; }

}  // namespace

extern "C" {

int sbf_probe_sm_count(int *sms) {
    if (!sms) return -1;
    int dev = 0;
    cudaDeviceProp p;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaGetDeviceProperties(&p, dev) != cudaSuccess) return -2;
    *sms = p.multiProcessorCount;
    return 0;
}

int sbf_probe_alu(int kind, int iters, int blocks, int threads, uint32_t *sink, void *stream, double *ops) {
    if (kind < 0 || kind > 4 || iters < 1 || blocks < 1 || threads < 32 || threads > 1024 || !sink) return -1;
    cudaStream_t st = as_stream(stream);
    switch (kind) {
        case 0: probe_alu_kernel<0><<<blocks, threads, 0, st>>>(iters, sink); break;
        case 1: probe_alu_kernel<1><<<blocks, threads, 0, st>>>(iters, sink); break;
        case 2: probe_alu_kernel<2><<<blocks, threads, 0, st>>>(iters, sink); break;
        case 3: probe_alu_kernel<3><<<blocks, threads, 0, st>>>(iters, sink); break;
        default: probe_alu_kernel<4><<<blocks, threads, 0, st>>>(iters, sink); break;
    }
    if (ops)
        *ops = (double)blocks * threads * (double)iters * kAluSteps * kAluChains * alu_ops_per_step(kind);
    return launched();
}

int sbf_probe_rmw(int mode, uint64_t *buf, uint64_t n_rows, int64_t n_updates, uint64_t seed, int blocks,
                  int threads, void *stream) {
    if (mode < 0 || mode > 3 || !buf || !pow2(n_rows) || n_updates < 0 || blocks < 1 || threads < 32 ||
        threads > 1024 || (mode == 3 && threads % 32))
        return -1;
    cudaStream_t st = as_stream(stream);
    const uint64_t mask = n_rows - 1;
    switch (mode) {
        case 0: probe_rmw_kernel<0><<<blocks, threads, 0, st>>>(buf, mask, n_updates, seed); break;
        case 1: probe_rmw_kernel<1><<<blocks, threads, 0, st>>>(buf, mask, n_updates, seed); break;
        case 3: probe_rmw_kernel<3><<<blocks, threads, 0, st>>>(buf, mask, n_updates, seed); break;
        default: probe_rmw_kernel<2><<<blocks, threads, 0, st>>>(buf, mask, n_updates, seed); break;
    }
    return launched();
}

int sbf_probe_read(int mode, const uint64_t *buf, uint64_t n_rows, int64_t n_reads, uint64_t seed, int blocks,
                   int threads, uint64_t *sink, void *stream) {
    if (mode < 0 || mode > 6 || !buf || !sink || !pow2(n_rows) || n_reads < 0 || blocks < 1 || threads < 32 ||
        threads > 256)
        return -1;
    cudaStream_t st = as_stream(stream);
    const uint64_t mask = n_rows - 1;
    const size_t smem = mode >= 4 ? (size_t)threads * (kReadsInFlight * 32 + 8) : 0;
    if (smem > 48 * 1024) {
        const void *fn = mode == 4   ? reinterpret_cast<const void *>(&probe_read_kernel<4>)
                         : mode == 5 ? reinterpret_cast<const void *>(&probe_read_kernel<5>)
                                     : reinterpret_cast<const void *>(&probe_read_kernel<6>);
        if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
            return -2;
    }
    switch (mode) {
        case 0: probe_read_kernel<0><<<blocks, threads, 0, st>>>(buf, mask, n_reads, seed, sink); break;
        case 1: probe_read_kernel<1><<<blocks, threads, 0, st>>>(buf, mask, n_reads, seed, sink); break;
        case 2: probe_read_kernel<2><<<blocks, threads, 0, st>>>(buf, mask, n_reads, seed, sink); break;
        case 3: probe_read_kernel<3><<<blocks, threads, 0, st>>>(buf, mask, n_reads, seed, sink); break;
        case 4: probe_read_kernel<4><<<blocks, threads, smem, st>>>(buf, mask, n_reads, seed, sink); break;
        case 6: probe_read_kernel<6><<<blocks, threads, smem, st>>>(buf, mask, n_reads, seed, sink); break;
        default: probe_read_kernel<5><<<blocks, threads, smem, st>>>(buf, mask, n_reads, seed, sink); break;
    }
    return launched();
}

}  // extern "C"
