// sbf_noalloc.cu -- a host-facing query that allocates nothing.
//
// sbf_query_host stages its batch through device buffers that it allocates
// (and grows) with cudaMalloc.  Some callers cannot allocate device memory at
// call time: code running under an allocator that owns the whole device (a
// framework's caching allocator, a fixed memory budget), or loops where the
// implicit device synchronisation of cudaMalloc / cudaFree is not acceptable.
// sbf_query_host_noalloc serves them: it stages the batch through one
// file-scope __device__ array of fixed size instead.
//
// The array exists once per device that loads this library and stays
// allocated until the process exits.  Every call shares it and it keeps the
// previous call's contents.  The query kernel reads only the bytes and offsets
// copied in by the same call, and when it runs it writes every answer word
// that is copied back.  It does not run when the filter's sticky status is
// already set (malformed offsets of an earlier call not yet reported, or a
// bounded device wait that gave up): the staged answer words then hold an
// earlier call's contents.  So the call ends like sbf_query_host, by reading
// and clearing the status, and returns its error instead of those words'
// meaning.  Calls whose work overlaps on the GPU (for example on two streams)
// race on the array.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "sbf_internal.h"

namespace {

constexpr int64_t kMaxPositions = int64_t(1) << 24;  // offsets[n] - offsets[0]
constexpr int64_t kMaxRecords = int64_t(1) << 20;    // n
constexpr int64_t kSeqBytes = kMaxPositions + 64;
constexpr int64_t kOffBytes = (kMaxRecords + 1) * 8;
constexpr int64_t kOutBytes = (kMaxPositions / 32 + 8) * 4;
constexpr int64_t kOffAt = (kSeqBytes + 255) & ~int64_t(255);
constexpr int64_t kOutAt = (kOffAt + kOffBytes + 255) & ~int64_t(255);
constexpr int64_t kFlagAt = (kOutAt + kOutBytes + 255) & ~int64_t(255);
constexpr int64_t kScratchBytes = kFlagAt + 256;

// ~26 MiB: the sequence bytes, then the offsets, then the answer words, then
// the query's uniform-batch flag word.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
char *g_scratch_addr[kMaxDevices] = {};

// Device address of g_scratch on `dev` (the current device), looked up once
// per device.  In host code g_scratch names a host-side stand-in, never the
// device memory, so the address must come from cudaGetSymbolAddress.
int scratch_on(int dev, char **out) {
    if (dev < 0 || dev >= kMaxDevices) return sbf::set_error(SBF_ERR_INVALID_ARG, "device index %d too large", dev);
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || !p)
            return sbf::set_error(SBF_ERR_CUDA, "cudaGetSymbolAddress of the staging array: %s", cudaGetErrorString(e));
        g_scratch_addr[dev] = static_cast<char *>(p);
    }
    *out = g_scratch_addr[dev];
    return SBF_OK;
}

}  // namespace

extern "C" int sbf_query_host_noalloc(const sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n,
                                      uint32_t *out_bits, void *stream) {
    using sbf::set_error;
    if (!f || !seq || !offsets || !out_bits || n < 0)
        return set_error(SBF_ERR_INVALID_ARG, "sbf_query_host_noalloc: bad arguments");
    if (n == 0) return SBF_OK;
    if (n > kMaxRecords)
        return set_error(SBF_ERR_INVALID_ARG, "sbf_query_host_noalloc: %lld records exceed the maximum of %lld",
                         (long long)n, (long long)kMaxRecords);
    if (offsets[0] < 0) return set_error(SBF_ERR_BAD_OFFSETS, "offsets[0] < 0");
    for (int64_t r = 0; r < n; ++r)
        if (offsets[r + 1] < offsets[r])
            return set_error(SBF_ERR_BAD_OFFSETS, "offsets decrease at record %lld", (long long)r);
    const int64_t lo = offsets[0], hi = offsets[n];
    if (hi - lo > kMaxPositions)
        return set_error(SBF_ERR_INVALID_ARG, "sbf_query_host_noalloc: %lld positions exceed the maximum of %lld",
                         (long long)(hi - lo), (long long)kMaxPositions);
    if (hi == lo) return SBF_OK;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != f->device)
        return set_error(SBF_ERR_INVALID_ARG, "the filter's device is not current");
    char *base = nullptr;
    if (int rc = scratch_on(dev, &base)) return rc;

    // Position g of the batch lives at byte g - cs of the staged sequence and
    // its answer bit in word (g >> 5) - (cs >> 5) of the staged answers; cs is
    // offsets[0] rounded down to a multiple of 32.  The kernel is handed
    // pointers biased by cs so that it indexes with the caller's offsets.
    const int64_t cs = lo & ~int64_t(31);
    char *d_seq = base;
    int64_t *d_off = reinterpret_cast<int64_t *>(base + kOffAt);
    uint32_t *d_out = reinterpret_cast<uint32_t *>(base + kOutAt);
    const char *k_seq = reinterpret_cast<const char *>(reinterpret_cast<uintptr_t>(d_seq) - (uintptr_t)cs);
    uint32_t *k_out = reinterpret_cast<uint32_t *>(reinterpret_cast<uintptr_t>(d_out) - (uintptr_t)(cs >> 5) * 4);
    const int64_t words = (hi - cs + 31) / 32;

    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(d_seq + (lo - cs), seq + lo, (size_t)(hi - lo), cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(d_off, offsets, sizeof(int64_t) * (size_t)(n + 1), cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return set_error(SBF_ERR_CUDA, "host-to-device copy: %s", cudaGetErrorString(e));
    int *d_flag = reinterpret_cast<int *>(base + kFlagAt);
    if (int rc = sbf::launch_query(f, k_seq, d_off, n, k_out, stream, true, d_flag)) return rc;
    e = cudaMemcpyAsync(out_bits + (cs >> 5), d_out, sizeof(uint32_t) * (size_t)words, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return set_error(SBF_ERR_CUDA, "sbf_query_host_noalloc: %s", cudaGetErrorString(e));
    // a set status means the kernel skipped its work and the copied words are
    // stale: report it (and clear it) as sbf_query_host does; this reads one
    // int with cudaMemcpy and allocates nothing
    return sbf_get_status(const_cast<sbf_filter *>(f), stream);
}
