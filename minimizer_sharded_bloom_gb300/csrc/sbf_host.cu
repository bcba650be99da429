// sbf_host.cu -- host-facing insert/query ("cuSBF", Sec. IV-A: host-facing
// entry points synchronize; Sec. IV-G "Host FASTX staging": overlap pinned
// staging and host-to-device copies with kernels on alternating streams).
//
// The CSR batch is cut into chunks of output positions [cs, ce) (cs, ce
// multiples of 32 except at the very end).  A chunk ships the bytes
// [max(cs, offsets[0]), min(ce + kb - 1, offsets[n])) (kb = bytes of one
// k-mer) and its records clipped to that range, so every k-mer that starts in
// [cs, ce) sees exactly its own bytes; k-mers starting at or after ce fall off
// the clipped end and are invalid in that chunk.  A record clipped at the
// chunk's start keeps its symbol frame (DNA triplets).  Chunk c runs on slot c & 1 (a stream, device buffers
// and pinned buffers, all kept in the filter between calls); the host prepares
// chunk c+1 while the GPU works on chunk c.  Host buffers that are already
// page-locked are copied from (and to) directly; pageable ones go through the
// pinned staging buffers.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "sbf_internal.h"

namespace {

struct Slot {
    cudaStream_t stream = nullptr;
    char *d_seq = nullptr;
    int64_t *d_off = nullptr;
    uint32_t *d_out = nullptr;
    char *h_seq = nullptr;      // pinned staging for pageable sequence input
    int64_t *h_off = nullptr;   // pinned chunk-local offsets
    uint32_t *h_out = nullptr;  // pinned staging for pageable output
    int64_t cap_dseq = 0, cap_doff = 0, cap_dout = 0;
    int64_t cap_hseq = 0, cap_hoff = 0, cap_hout = 0;
    uint32_t *pend_dst = nullptr;  // pageable destination of a finished query chunk
    int64_t pend_words = 0;
};

struct Stager {
    Slot slot[2];
};

template <typename T>
cudaError_t grow_dev(T *&p, int64_t &cap, int64_t need) {
    if (need <= cap) return cudaSuccess;
    cudaFree(p);
    p = nullptr;
    cap = 0;
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&p), sizeof(T) * (size_t)need);
    if (e == cudaSuccess) cap = need;
    return e;
}

template <typename T>
cudaError_t grow_pinned(T *&p, int64_t &cap, int64_t need) {
    if (need <= cap) return cudaSuccess;
    cudaFreeHost(p);
    p = nullptr;
    cap = 0;
    cudaError_t e = cudaMallocHost(reinterpret_cast<void **>(&p), sizeof(T) * (size_t)need);
    if (e == cudaSuccess) cap = need;
    return e;
}

cudaError_t prepare(Slot &s, int64_t seq_bytes, int64_t n_off, int64_t out_words, bool stage_seq,
                    bool stage_out) {
    cudaError_t e = cudaSuccess;
    if (!s.stream) e = cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = grow_dev(s.d_seq, s.cap_dseq, std::max<int64_t>(seq_bytes, 16));
    if (e == cudaSuccess) e = grow_dev(s.d_off, s.cap_doff, std::max<int64_t>(n_off, 2));
    if (e == cudaSuccess && out_words) e = grow_dev(s.d_out, s.cap_dout, out_words);
    if (e == cudaSuccess && stage_seq) e = grow_pinned(s.h_seq, s.cap_hseq, seq_bytes);
    if (e == cudaSuccess) e = grow_pinned(s.h_off, s.cap_hoff, std::max<int64_t>(n_off, 2));
    if (e == cudaSuccess && stage_out) e = grow_pinned(s.h_out, s.cap_hout, out_words);
    return e;
}

// 1 = page-locked host memory, 0 = pageable host memory, -1 = not host memory.
int host_kind(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    if (a.type == cudaMemoryTypeHost) return 1;
    if (a.type == cudaMemoryTypeUnregistered) return 0;
    return -1;
}

// Device alias of host pointer p when kernels can read and write it in place:
// page-locked memory (its mapped address), or pageable memory on a device that
// accesses host memory through the host page tables (e.g. over NVLink-C2C).
// Returns nullptr when p must be staged.
const void *device_alias(const void *p, int dev) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    if (a.type == cudaMemoryTypeHost) return a.devicePointer ? a.devicePointer : p;
    if (a.type == cudaMemoryTypeUnregistered) {
        int pageable = 0;
        if (cudaDeviceGetAttribute(&pageable, cudaDevAttrPageableMemoryAccess, dev) == cudaSuccess && pageable)
            return p;
    }
    return nullptr;
}

// Read (and for query write) the host buffers in place: one launch, no copies.
// Returns 1 when done this way, 0 when the buffers are not device-accessible.
int run_in_place(sbf_filter *f, const char *seq, const int64_t *off, int64_t n, uint32_t *out_bits,
                 void *user_stream, bool query, int *rc) {
    const int64_t lo = off[0], hi = off[n];
    const void *s_al = device_alias(seq + lo, f->device);
    const void *o_al = device_alias(off, f->device);
    const void *q_al = query ? device_alias(out_bits + (lo >> 5), f->device) : nullptr;
    if (!s_al || !o_al || (query && !q_al)) return 0;
    // the aliases of the buffers' first used elements, re-biased to index with the caller's offsets
    const char *dseq = reinterpret_cast<const char *>(reinterpret_cast<uintptr_t>(s_al) - (uintptr_t)lo);
    const int64_t *doff = static_cast<const int64_t *>(o_al);
    uint32_t *dout = query ? reinterpret_cast<uint32_t *>(reinterpret_cast<uintptr_t>(q_al) -
                                                           (uintptr_t)(lo >> 5) * sizeof(uint32_t))
                           : nullptr;
    *rc = query ? sbf::launch_query(f, dseq, doff, n, dout, user_stream, false)
                : sbf::launch_insert(f, dseq, doff, n, user_stream, false);
    if (*rc == SBF_OK) {
        cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(user_stream));
        if (e != cudaSuccess) *rc = sbf::set_error(SBF_ERR_CUDA, "host call: %s", cudaGetErrorString(e));
    }
    if (*rc == SBF_OK) *rc = sbf_get_status(f, user_stream);
    return 1;
}

// First record r with offsets[r + 1] > g.
int64_t record_at(const int64_t *off, int64_t n, int64_t g) {
    int64_t lo = 0, hi = n - 1;
    while (lo < hi) {
        const int64_t mid = lo + (hi - lo) / 2;
        if (off[mid + 1] > g) hi = mid; else lo = mid + 1;
    }
    return lo;
}

int run_host(sbf_filter *f, const char *seq, const int64_t *off, int64_t n, uint32_t *out_bits,
             void *user_stream, bool query) {
    using sbf::set_error;
    if (!f || !seq || !off || n < 0 || (query && !out_bits))
        return set_error(SBF_ERR_INVALID_ARG, "host call: bad arguments");
    if (n == 0) return SBF_OK;
    if (off[0] < 0) return set_error(SBF_ERR_BAD_OFFSETS, "offsets[0] < 0");
    // The whole-array check runs on the host only where the host needs valid
    // offsets (an empty range, the staged path's chunking); in place, the
    // device check kernel covers them and sbf_get_status reports them.
    auto host_check = [&]() -> int {
        for (int64_t r = 0; r < n; ++r)
            if (off[r + 1] < off[r])
                return set_error(SBF_ERR_BAD_OFFSETS, "offsets decrease at record %lld", (long long)r);
        return SBF_OK;
    };
    const int64_t lo = off[0], hi = off[n];
    if (hi <= lo) return host_check();
    const int seq_kind = host_kind(seq + lo);
    const int out_kind = query ? host_kind(out_bits + (lo >> 5)) : 0;
    if (seq_kind < 0 || out_kind < 0 || host_kind(off) < 0)
        return set_error(SBF_ERR_INVALID_ARG, "host call given a device pointer; use sbf_insert/sbf_query");
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != f->device)
        return set_error(SBF_ERR_INVALID_ARG, "the filter's device is not current");
    if (f->host_mode == 0) {
        int rc = SBF_OK;
        if (run_in_place(f, seq, off, n, out_bits, user_stream, query, &rc)) return rc;
    }
    if (int rc = host_check()) return rc;
    if (!f->stager) f->stager = new Stager;
    Stager &st = *static_cast<Stager *>(f->stager);

    cudaEvent_t ready;
    if (cudaEventCreateWithFlags(&ready, cudaEventDisableTiming) != cudaSuccess)
        return set_error(SBF_ERR_CUDA, "cudaEventCreate");
    cudaEventRecord(ready, reinterpret_cast<cudaStream_t>(user_stream));

    int rc = SBF_OK;
    int64_t cs = lo & ~int64_t(31);
    for (int64_t c = 0; cs < hi && rc == SBF_OK; ++c) {
        const int64_t ce = std::min<int64_t>(cs + f->host_chunk, hi);
        const int64_t data_lo = std::max<int64_t>(cs, lo);
        const int64_t data_hi = std::min<int64_t>(ce + sbf::kmer_bytes(f) - 1, hi);
        const int64_t r0 = record_at(off, n, data_lo);
        const int64_t r1 = record_at(off, n, data_hi - 1) + 1;
        const int64_t n_loc = r1 - r0;
        // A record clipped at data_lo keeps its symbol frame: its chunk-local
        // start moves up to its next symbol boundary (triplets; the bytes
        // skipped start no symbol of the record).
        const int sb = sbf::symbol_bytes(f->alphabet);
        const int64_t first_lo = off[r0] < data_lo ? data_lo + (sb - (data_lo - off[r0]) % sb) % sb : data_lo;
        const int64_t dev_words = (data_hi - cs + 31) / 32 + 1;  // what the kernel writes
        const int64_t words = (ce - cs + 31) / 32;                // what this chunk returns
        Slot &s = st.slot[c & 1];
        if (s.stream) {
            if (cudaStreamSynchronize(s.stream) != cudaSuccess) {
                rc = set_error(SBF_ERR_CUDA, "staging stream failed");
                break;
            }
            if (s.pend_dst) std::memcpy(s.pend_dst, s.h_out, sizeof(uint32_t) * (size_t)s.pend_words);
            s.pend_dst = nullptr;
        }
        if (prepare(s, data_hi - cs, n_loc + 1, query ? dev_words : 0, seq_kind == 0,
                    query && out_kind == 0) != cudaSuccess) {
            cudaGetLastError();
            rc = set_error(SBF_ERR_OOM, "staging buffers could not be allocated");
            break;
        }
        cudaStreamWaitEvent(s.stream, ready, 0);
        for (int64_t r = 0; r <= n_loc; ++r)
            s.h_off[r] = std::min<int64_t>(std::max<int64_t>(off[r0 + r], data_lo), data_hi) - cs;
        // (a record that ends before that boundary is left empty)
        s.h_off[0] = std::min<int64_t>(first_lo - cs, s.h_off[1]);
        const char *src = seq + data_lo;
        char *dst = s.d_seq + (data_lo - cs);
        if (seq_kind == 0) {
            std::memcpy(s.h_seq + (data_lo - cs), src, (size_t)(data_hi - data_lo));
            src = s.h_seq + (data_lo - cs);
        }
        cudaError_t e = cudaMemcpyAsync(dst, src, (size_t)(data_hi - data_lo), cudaMemcpyHostToDevice, s.stream);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(s.d_off, s.h_off, sizeof(int64_t) * (size_t)(n_loc + 1), cudaMemcpyHostToDevice,
                                s.stream);
        if (e != cudaSuccess) {
            rc = set_error(SBF_ERR_CUDA, "host-to-device copy: %s", cudaGetErrorString(e));
            break;
        }
        if (query) {
            rc = sbf_query(f, s.d_seq, s.d_off, n_loc, s.d_out, s.stream);
            if (rc != SBF_OK) break;
            uint32_t *final_dst = out_bits + (cs >> 5);
            uint32_t *land = out_kind == 1 ? final_dst : s.h_out;
            e = cudaMemcpyAsync(land, s.d_out, sizeof(uint32_t) * (size_t)words, cudaMemcpyDeviceToHost, s.stream);
            if (e != cudaSuccess) {
                rc = set_error(SBF_ERR_CUDA, "device-to-host copy: %s", cudaGetErrorString(e));
                break;
            }
            if (out_kind == 0) {
                s.pend_dst = final_dst;
                s.pend_words = words;
            }
        } else {
            rc = sbf_insert(f, s.d_seq, s.d_off, n_loc, s.stream);
            if (rc != SBF_OK) break;
        }
        cs = ce;
    }
    for (Slot &s : st.slot) {
        if (!s.stream) continue;
        if (cudaStreamSynchronize(s.stream) != cudaSuccess && rc == SBF_OK)
            rc = set_error(SBF_ERR_CUDA, "staging stream failed");
        if (s.pend_dst && rc == SBF_OK) std::memcpy(s.pend_dst, s.h_out, sizeof(uint32_t) * (size_t)s.pend_words);
        s.pend_dst = nullptr;
    }
    cudaEventDestroy(ready);
    if (rc == SBF_OK) {
        // the device check of the chunk offsets could only have failed if the host check missed it
        rc = sbf_get_status(f, nullptr);
    }
    return rc;
}

}  // namespace

void sbf::destroy_stager(void *p) {
    if (!p) return;
    Stager *st = static_cast<Stager *>(p);
    for (Slot &s : st->slot) {
        if (s.stream) cudaStreamSynchronize(s.stream);
        cudaFree(s.d_seq);
        cudaFree(s.d_off);
        cudaFree(s.d_out);
        cudaFreeHost(s.h_seq);
        cudaFreeHost(s.h_off);
        cudaFreeHost(s.h_out);
        if (s.stream) cudaStreamDestroy(s.stream);
    }
    delete st;
}

extern "C" {

int sbf_set_host_mode(sbf_filter *f, int mode) {
    if (!f || mode < 0 || mode > 1) return sbf::set_error(SBF_ERR_INVALID_ARG, "sbf_set_host_mode: mode is 0 or 1");
    f->host_mode = mode;
    return SBF_OK;
}

int sbf_set_host_chunk(sbf_filter *f, int64_t positions) {
    if (!f || positions < 32) return sbf::set_error(SBF_ERR_INVALID_ARG, "sbf_set_host_chunk: need >= 32 positions");
    f->host_chunk = positions & ~int64_t(31);
    return SBF_OK;
}

int sbf_insert_host(sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n, void *stream) {
    return run_host(f, seq, offsets, n, nullptr, stream, false);
}

int sbf_query_host(const sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n,
                   uint32_t *out_bits, void *stream) {
    return run_host(const_cast<sbf_filter *>(f), seq, offsets, n, out_bits, stream, true);
}

}  // extern "C"
