// sbf_host.cu -- host-facing insert/query ("cuSBF", Sec. IV-A: host-facing
// entry points synchronize; Sec. IV-G "Host FASTX staging": overlap pinned
// staging and host-to-device copies with kernels on alternating streams).
//
// In place: where the device can read (and write) the caller's buffers, one
// launch reads them directly.  Staged: the CSR batch is cut into chunks of
// positions [cs, ce) (multiples of 32 except at the very end).  A chunk ends at
// a record start on a 32-position boundary when one is near ce: its records
// are whole.  Otherwise it ends at ce itself and ships the bytes up to
// min(ce + kb - 1, offsets[n]) (kb = bytes of one k-mer) with its last record
// clipped there; every k-mer starting in [cs, ce) sees exactly its own bytes,
// and the answer words from ce >> 5 on are left to the next chunk.  A record
// clipped at a chunk's start keeps its symbol frame (DNA triplets).  The
// kernels index absolute positions: a chunk's offsets are the caller's, as
// they are, with both ends clipped, and its staged bytes are addressed through
// a pointer biased by cs, so the host never rewrites the offsets (a chunk's
// two clipped ends are written on the device).  Chunk c runs on slot c mod 4
// (a stream, device buffers and pinned buffers, all kept in the filter
// between calls).  Host buffers that are already page-locked are copied from
// directly; pageable ones go through the pinned staging buffers.  Answers go
// straight to the caller's buffer where the device can write it.  When no
// pinned staging buffer is in play, every chunk is enqueued at once and the
// host waits once; otherwise it waits for a slot before reusing its buffers.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "sbf_chunks.h"
#include "sbf_internal.h"

namespace {

struct Slot {
    cudaStream_t stream = nullptr;
    char *d_seq = nullptr;
    int64_t *d_off = nullptr;
    uint32_t *d_out = nullptr;
    int *d_flag = nullptr;      // the query's uniform-batch flag word (one per slot: no allocation per chunk)
    char *h_seq = nullptr;      // pinned staging for pageable sequence input
    int64_t *h_off = nullptr;   // pinned chunk-local offsets
    uint32_t *h_out = nullptr;  // pinned staging for pageable output
    int64_t cap_dseq = 0, cap_doff = 0, cap_dout = 0;
    int64_t cap_hseq = 0, cap_hoff = 0, cap_hout = 0;
    uint32_t *pend_dst = nullptr;  // pageable destination of a finished query chunk
    int64_t pend_words = 0;
};

constexpr int kSlots = 8;

struct Stager {
    // kSlots slots: a chunk's copy waits only for the chunk kSlots back,
    // which leaves the copy engine slack when copies and kernels take about
    // as long, and keeps the batch's small last chunks from waiting on the
    // kernels of its large middle ones
    Slot slot[kSlots];
    int64_t *d_all_off = nullptr;  // the whole offsets array of a call, on the device
    int64_t cap_all_off = 0;
    int *d_call_flag = nullptr;    // its uniformity flag (from the one check of the call)
};

// Offsets arrays up to this many entries (256 MiB) go to the device whole.
constexpr int64_t kAllOffMax = int64_t(1) << 25;

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

cudaError_t prepare(Slot &s, int64_t seq_bytes, int64_t n_off, int64_t n_off_host, int64_t out_words,
                    bool stage_seq, bool stage_out) {
    cudaError_t e = cudaSuccess;
    if (!s.stream) e = cudaStreamCreateWithFlags(&s.stream, cudaStreamNonBlocking);
    if (e == cudaSuccess && !s.d_flag) e = cudaMalloc(reinterpret_cast<void **>(&s.d_flag), sizeof(int));
    if (e == cudaSuccess) e = grow_dev(s.d_seq, s.cap_dseq, std::max<int64_t>(seq_bytes, 16));
    if (e == cudaSuccess) e = grow_dev(s.d_off, s.cap_doff, std::max<int64_t>(n_off, 2));
    if (e == cudaSuccess && out_words) e = grow_dev(s.d_out, s.cap_dout, out_words);
    if (e == cudaSuccess && stage_seq) e = grow_pinned(s.h_seq, s.cap_hseq, seq_bytes);
    if (e == cudaSuccess) e = grow_pinned(s.h_off, s.cap_hoff, std::max<int64_t>(n_off_host, 2));
    if (e == cudaSuccess && stage_out) e = grow_pinned(s.h_out, s.cap_hout, out_words);
    return e;
}

// The two clipped ends of a chunk's device offsets, written on the device so
// that no host buffer has to outlive the call's enqueueing.
__global__ void patch_ends_kernel(int64_t *off, int64_t n_loc, int64_t first, int64_t last) {
    if (threadIdx.x == 0) off[0] = first;
    if (threadIdx.x == 1) off[n_loc] = last;
}

cudaError_t patch_ends(int64_t *off, int64_t n_loc, int64_t first, int64_t last, cudaStream_t st) {
    patch_ends_kernel<<<1, 32, 0, st>>>(off, n_loc, first, last);
    return cudaGetLastError();
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
    const int64_t lo = off[0];
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
    // In place (no copies) where the device reads the buffers itself: always
    // in mode 2; in mode 0 only for a pageable sequence.  A page-locked one is
    // staged: the copy engine moves it over the host link faster than the
    // kernel's own loads, and the chunks keep a batch of equal-length reads
    // dense.  (A pageable sequence would need a host copy into pinned memory.)
    const bool stage_first = f->host_mode == 1 || (f->host_mode == 0 && seq_kind == 1);
    if (!stage_first) {
        int rc = SBF_OK;
        if (run_in_place(f, seq, off, n, out_bits, user_stream, query, &rc)) return rc;
    }
    // Staged.  The offsets are checked once before any chunk's kernel runs:
    // on a device copy of the whole array (queries, below), on the device
    // reading them in place, or else on the host.  A bad array sets the
    // sticky status, and every chunk's kernel then returns at once.
    const int64_t *off_dev = static_cast<const int64_t *>(device_alias(off, f->device));
    // answers go straight to the caller's buffer where the device can write it
    uint32_t *out_dev = nullptr;
    if (query) {
        if (const void *q = device_alias(out_bits + (lo >> 5), f->device))
            out_dev = reinterpret_cast<uint32_t *>(reinterpret_cast<uintptr_t>(q) -
                                                   (uintptr_t)(lo >> 5) * sizeof(uint32_t));
    }
    const bool off_pinned = host_kind(off) == 1;
    if (!f->stager) f->stager = new Stager;
    Stager &st = *static_cast<Stager *>(f->stager);
    // For a query, where it fits, the whole offsets array crosses the host
    // link once: one copy to the device, one check there (which also finds
    // whether every record has one length), and chunks whose two ends are
    // record starts index that copy directly, with no check of their own.
    // (Measured on the 1 Gbp insert this was slower, 7.3 against 6.1 ms, so
    // an insert ships each chunk's slice and checks it.)
    bool all_off = query && n + 1 <= kAllOffMax;
    if (all_off) {
        cudaError_t e = grow_dev(st.d_all_off, st.cap_all_off, n + 1);
        if (e == cudaSuccess && !st.d_call_flag) e = cudaMalloc(reinterpret_cast<void **>(&st.d_call_flag), sizeof(int));
        if (e != cudaSuccess) {
            cudaGetLastError();
            all_off = false;
        }
    }
    if (!all_off && !off_dev)
        if (int rc = host_check()) return rc;

    // Copies wait for the caller's earlier work (ready); kernels also for the
    // offsets check (checked), which thus overlaps the first copies.
    cudaEvent_t ready, checked;
    if (cudaEventCreateWithFlags(&ready, cudaEventDisableTiming) != cudaSuccess)
        return set_error(SBF_ERR_CUDA, "cudaEventCreate");
    if (cudaEventCreateWithFlags(&checked, cudaEventDisableTiming) != cudaSuccess) {
        cudaEventDestroy(ready);
        return set_error(SBF_ERR_CUDA, "cudaEventCreate");
    }
    cudaEventRecord(ready, reinterpret_cast<cudaStream_t>(user_stream));
    int *call_flag = query && f->query_detects_dense ? st.d_call_flag : nullptr;
    int crc = SBF_OK;
    if (all_off) {
        cudaError_t e = cudaMemcpyAsync(st.d_all_off, off, sizeof(int64_t) * (size_t)(n + 1), cudaMemcpyHostToDevice,
                                        reinterpret_cast<cudaStream_t>(user_stream));
        crc = e == cudaSuccess ? sbf::launch_offsets_check(f, st.d_all_off, n, user_stream, call_flag)
                               : set_error(SBF_ERR_CUDA, "offsets copy: %s", cudaGetErrorString(e));
    } else if (off_dev) {
        crc = sbf::launch_offsets_check(f, off_dev, n, user_stream);
    }
    if (crc != SBF_OK) {
        cudaEventDestroy(ready);
        cudaEventDestroy(checked);
        return crc;
    }
    cudaEventRecord(checked, reinterpret_cast<cudaStream_t>(user_stream));

    // With page-locked input, offsets the device reads whole or page-locked,
    // and answers the device writes in place, no host buffer is reused from
    // chunk to chunk: every chunk is enqueued at once (a slot's stream orders
    // its device buffers) and the host waits once at the end, so a host
    // thread that is descheduled mid-call does not leave the GPU idle.
    // Otherwise a slot's pinned staging buffers are reused four chunks on,
    // after a wait for that slot.
    const bool host_staging = seq_kind == 0 || (query && !out_dev) || (!all_off && !off_pinned);
    const int64_t kb = sbf::kmer_bytes(f);
    // the chunks and their clipped ends (sbf_chunks.h); a query's chunks also
    // shrink towards the batch's end, an insert's do not (its kernels take
    // longer than its copies, and small launches of its random updates cost
    // throughput)
    sbf::ChunkPlan plan(off, n, f->host_chunk, kb, sbf::symbol_bytes(f->alphabet), query);
    const int64_t chunk_max = plan.chunk_max();
    // the most records any chunk holds: every slot's offsets buffer is sized
    // for it before the first chunk, so no buffer grows (and frees) while
    // earlier chunks are in flight (plain host arithmetic over the plan)
    int64_t max_recs = 1;
    {
        sbf::ChunkPlan pre(off, n, f->host_chunk, sbf::kmer_bytes(f), sbf::symbol_bytes(f->alphabet), query);
        sbf::Chunk c0;
        while (pre.next(c0))
            if (!c0.empty) max_recs = std::max<int64_t>(max_recs, c0.r1 - c0.r0);
    }
    int rc = SBF_OK;
    sbf::Chunk ch;
    for (int64_t c = 0; rc == SBF_OK && plan.next(ch); ++c) {
        if (ch.empty) continue;  // only with offsets the check rejects
        const int64_t cs = ch.cs, ce = ch.ce, data_lo = ch.data_lo, data_hi = ch.data_hi;
        const int64_t r0 = ch.r0, r1 = ch.r1, first = ch.first, last = ch.last;
        const int64_t n_loc = r1 - r0;
        const int64_t dev_words = (data_hi - cs + 31) / 32 + 1;  // what the kernel may write
        const int64_t words = (ce - cs + 31) / 32;                // what this chunk returns
        Slot &s = st.slot[c % kSlots];
        if (s.stream && host_staging) {
            if (cudaStreamSynchronize(s.stream) != cudaSuccess) {
                rc = set_error(SBF_ERR_CUDA, "staging stream failed");
                break;
            }
            if (s.pend_dst) std::memcpy(s.pend_dst, s.h_out, sizeof(uint32_t) * (size_t)s.pend_words);
            s.pend_dst = nullptr;
        }
        const bool stage_out = query && !out_dev;
        // sized for the largest chunk at once: growing a buffer mid-call would
        // free it, which waits for the whole device
        const int64_t max_bytes = std::max<int64_t>(data_hi - cs, chunk_max + kb);
        if (prepare(s, max_bytes, max_recs + 1, (all_off || off_pinned) ? 2 : max_recs + 1,
                    stage_out ? std::max<int64_t>(dev_words, (max_bytes + 31) / 32 + 1) : 0, seq_kind == 0,
                    stage_out) != cudaSuccess) {
            cudaGetLastError();
            rc = set_error(SBF_ERR_OOM, "staging buffers could not be allocated");
            break;
        }
        cudaStreamWaitEvent(s.stream, ready, 0);
        const char *src = seq + data_lo;
        char *dst = s.d_seq + (data_lo - cs);
        if (seq_kind == 0) {
            std::memcpy(s.h_seq + (data_lo - cs), src, (size_t)(data_hi - data_lo));
            src = s.h_seq + (data_lo - cs);
        }
        cudaError_t e = cudaMemcpyAsync(dst, src, (size_t)(data_hi - data_lo), cudaMemcpyHostToDevice, s.stream);
        const size_t off_bytes = sizeof(int64_t) * (size_t)(n_loc + 1);
        // both ends at record starts: the caller's slice as it is
        const bool whole = ch.whole;
        const int64_t *k_off = s.d_off;
        if (all_off) {
            // from the device copy of the whole array (written before `checked`)
            if (e == cudaSuccess) e = cudaStreamWaitEvent(s.stream, checked, 0);
            if (whole) {
                k_off = st.d_all_off + r0;
            } else {
                if (e == cudaSuccess)
                    e = cudaMemcpyAsync(s.d_off, st.d_all_off + r0, off_bytes, cudaMemcpyDeviceToDevice, s.stream);
                if (e == cudaSuccess) e = patch_ends(s.d_off, n_loc, first, last, s.stream);
            }
        } else if (off_pinned) {
            // the slice straight from the caller's page-locked array, then the two ends
            if (e == cudaSuccess) e = cudaMemcpyAsync(s.d_off, off + r0, off_bytes, cudaMemcpyHostToDevice, s.stream);
            if (e == cudaSuccess) e = patch_ends(s.d_off, n_loc, first, last, s.stream);
        } else {
            std::memcpy(s.h_off, off + r0, off_bytes);
            s.h_off[0] = first;
            s.h_off[n_loc] = last;
            if (e == cudaSuccess) e = cudaMemcpyAsync(s.d_off, s.h_off, off_bytes, cudaMemcpyHostToDevice, s.stream);
        }
        if (e != cudaSuccess) {
            rc = set_error(SBF_ERR_CUDA, "host-to-device copy: %s", cudaGetErrorString(e));
            break;
        }
        cudaStreamWaitEvent(s.stream, checked, 0);
        // the kernel indexes absolute positions: the staged bytes sit at d_seq + (g - cs)
        const char *k_seq = reinterpret_cast<const char *>(reinterpret_cast<uintptr_t>(s.d_seq) - (uintptr_t)cs);
        if (query) {
            uint32_t *k_out = out_dev ? out_dev
                                      : reinterpret_cast<uint32_t *>(reinterpret_cast<uintptr_t>(s.d_out) -
                                                                     (uintptr_t)(cs >> 5) * sizeof(uint32_t));
            // a chunk cut inside a record leaves the words from ce on to the next chunk.
            // Checked whole: a whole chunk takes the call's uniformity flag (a
            // uniform batch gives uniform whole chunks), a cut one none (CSR).
            if (all_off)
                rc = sbf::launch_query(f, k_seq, k_off, n_loc, k_out, s.stream, true, whole ? call_flag : nullptr,
                                       ch.final ? INT64_MAX : (ce >> 5), false);
            else
                rc = sbf::launch_query(f, k_seq, k_off, n_loc, k_out, s.stream, true, s.d_flag,
                                       ch.final ? INT64_MAX : (ce >> 5));
            if (rc != SBF_OK) break;
            if (stage_out) {
                e = cudaMemcpyAsync(s.h_out, s.d_out, sizeof(uint32_t) * (size_t)words, cudaMemcpyDeviceToHost,
                                    s.stream);
                if (e != cudaSuccess) {
                    rc = set_error(SBF_ERR_CUDA, "device-to-host copy: %s", cudaGetErrorString(e));
                    break;
                }
                s.pend_dst = out_bits + (cs >> 5);
                s.pend_words = words;
            }
        } else {
            rc = sbf::launch_insert(f, k_seq, k_off, n_loc, s.stream, true, !all_off);
            if (rc != SBF_OK) break;
        }
    }
    for (Slot &s : st.slot) {
        if (!s.stream) continue;
        if (cudaStreamSynchronize(s.stream) != cudaSuccess && rc == SBF_OK)
            rc = set_error(SBF_ERR_CUDA, "staging stream failed");
        if (s.pend_dst && rc == SBF_OK) std::memcpy(s.pend_dst, s.h_out, sizeof(uint32_t) * (size_t)s.pend_words);
        s.pend_dst = nullptr;
    }
    cudaEventDestroy(ready);
    cudaEventDestroy(checked);
    if (rc == SBF_OK) rc = sbf_get_status(f, user_stream);
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
        cudaFree(s.d_flag);
        cudaFreeHost(s.h_seq);
        cudaFreeHost(s.h_off);
        cudaFreeHost(s.h_out);
        if (s.stream) cudaStreamDestroy(s.stream);
    }
    cudaFree(st->d_all_off);
    cudaFree(st->d_call_flag);
    delete st;
}

extern "C" {

int sbf_set_host_mode(sbf_filter *f, int mode) {
    if (!f || mode < 0 || mode > 2) return sbf::set_error(SBF_ERR_INVALID_ARG, "sbf_set_host_mode: mode is 0, 1 or 2");
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
