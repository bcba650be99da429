// sbf_api.cu -- the C ABI of libsbf (declared in include/sbf.h).
//
// Argument checking, filter allocation, kernel selection (compile-time
// specialised strip kernel when one exists for (k, m, s, H), else the
// runtime-parameter kernel) and launch.  Device-facing calls enqueue on the
// caller's stream and return; the host-facing calls stage CSR batches through
// pinned buffers on two streams.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "sbf_internal.h"
#include "sbf_kernels.h"
#include "sbf_registry.h"

namespace sbf {
extern const StripEntry kStripEntriesMain[];
extern const int kStripCountMain;
extern const StripEntry kStripEntriesLargeH[];
extern const int kStripCountLargeH;
extern const StripEntry kStripEntriesProtein[];
extern const int kStripCountProtein;
extern const StripEntry kStripEntriesTriplet[];
extern const int kStripCountTriplet;
#ifdef SBF_WITH_SWEEP
#define SBF_DECLARE_UNIT(M, S)                       \
    extern const StripEntry kStripEntriesM##M##S##_[]; \
    extern const int kStripCountM##M##S##_;
SBF_SWEEP_UNITS(SBF_DECLARE_UNIT)
#undef SBF_DECLARE_UNIT
#endif

bool find_alphabet_strip(int alphabet, int k, int m, int s, int H, const void **insert, const void **query,
                         int *threads) {
    const StripEntry *table = alphabet == SBF_ALPHABET_PROTEIN ? kStripEntriesProtein : kStripEntriesTriplet;
    const int count = alphabet == SBF_ALPHABET_PROTEIN ? kStripCountProtein
                      : alphabet == SBF_ALPHABET_DNA_TRIPLET ? kStripCountTriplet : 0;
    for (int i = 0; i < count; ++i) {
        const StripEntry &e = table[i];
        if (e.k == k && e.m == m && e.s == s && e.H == H) {
            *insert = e.insert;
            *query = e.query;
            *threads = e.threads;
            return true;
        }
    }
    return false;
}

bool find_specialized(int k, int m, int s, int H, const void **insert, const void **query,
                      int *threads) {
    struct Table {
        const StripEntry *e;
        const int *n;
    };
    static const Table tables[] = {
        {kStripEntriesMain, &kStripCountMain},
        {kStripEntriesLargeH, &kStripCountLargeH},
#ifdef SBF_WITH_SWEEP
#define SBF_TABLE_UNIT(M, S) {kStripEntriesM##M##S##_, &kStripCountM##M##S##_},
        SBF_SWEEP_UNITS(SBF_TABLE_UNIT)
#undef SBF_TABLE_UNIT
#endif
    };
    for (const Table &t : tables)
        for (int i = 0; i < *t.n; ++i) {
            const StripEntry &e = t.e[i];
            if (e.insert && e.k == k && e.m == m && e.s == s && e.H == H) {
                *insert = e.insert;
                *query = e.query;
                *threads = e.threads;
                return true;
            }
        }
    return false;
}
}  // namespace sbf

namespace {

thread_local std::string g_last_error;

int vfail(int code, const char *fmt, va_list ap) {
    char buf[512];
    vsnprintf(buf, sizeof buf, fmt, ap);
    g_last_error = buf;
    return code;
}

int fail(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vfail(code, fmt, ap);
    va_end(ap);
    return code;
}

int cuda_fail(cudaError_t e, const char *what) {
    return fail(SBF_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

inline cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

int launch(const void *fn, int grid, int threads, const sbf::LaunchArgs &la, cudaStream_t st) {
    sbf::LaunchArgs copy = la;
    void *args[] = {&copy};
    cudaError_t e = cudaLaunchKernel(fn, dim3(grid), dim3(threads), args, 0, st);
    if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
    return SBF_OK;
}

int launch_check(const sbf_filter *f, const int64_t *offsets, int64_t n, cudaStream_t st,
                 int *nonuniform = nullptr) {
    const int64_t blocks = std::min<int64_t>((n + 255) / 256, f->grid_check);
    if (nonuniform) {
        cudaError_t e = cudaMemsetAsync(nonuniform, 0, sizeof(int), st);
        if (e != cudaSuccess) return cuda_fail(e, "flag reset");
    }
    sbf::check_offsets_kernel<<<(int)std::max<int64_t>(blocks, 1), 256, 0, st>>>(offsets, n, f->status,
                                                                                 nonuniform);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "offsets check launch");
    return SBF_OK;
}

sbf::LaunchArgs make_args(const sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n,
                          uint32_t *out, bool device_seq = true) {
    sbf::LaunchArgs la;
    la.seq = reinterpret_cast<const uint8_t *>(seq);
    la.offsets = offsets;
    la.n = n;
    la.words = f->words;
    la.out = out;
    la.status = f->status;
    la.shard_mask = f->num_shards - 1;
    la.seed = f->seed;
    la.k = f->k;
    la.m = f->m;
    la.s = f->s;
    la.H = f->H;
    la.device_seq = device_seq ? 1 : 0;
    la.rec_len = 0;
    la.nonuniform = nullptr;
    la.out_words_end = INT64_MAX;
    la.sectors = f->sectors;
    la.wait_test = 0;
    return la;
}

int grid_for(const void *fn, int threads, int sms) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, threads, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    return per_sm * sms;
}

int check_device(const sbf_filter *f) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev != f->device)
        return fail(SBF_ERR_INVALID_ARG, "filter lives on device %d but device %d is current", f->device, dev);
    return SBF_OK;
}

}  // namespace

int sbf::set_error(int code, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vfail(code, fmt, ap);
    va_end(ap);
    return code;
}

int sbf::launch_insert(sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n, void *stream,
                       bool device_seq, bool run_check) {
    if (n == 0) return SBF_OK;
    cudaStream_t st = as_stream(stream);
    if (run_check)
        if (int rc = launch_check(f, offsets, n, st)) return rc;
    return launch(f->insert_kernel, f->grid_insert, f->threads,
                  make_args(f, seq, offsets, n, nullptr, device_seq), st);
}

int sbf::launch_offsets_check(const sbf_filter *f, const int64_t *offsets, int64_t n, void *stream,
                              int *nonuniform) {
    if (n == 0) return SBF_OK;
    return launch_check(f, offsets, n, as_stream(stream), nonuniform);
}

int sbf::launch_query(const sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n,
                      uint32_t *out_bits, void *stream, bool device_seq, int *flag_word,
                      int64_t out_words_end, bool run_check) {
    if (n == 0) return SBF_OK;
    cudaStream_t st = as_stream(stream);
    // Where the query kernel can run a uniform batch as a dense one, the
    // offsets check reports uniformity into a word of this call's own (a
    // stream-ordered allocation from the filter's pool, or the caller's), so
    // that concurrent queries of one filter never share it.  Without a word
    // the kernel keeps the CSR geometry, which is correct for every batch.
    int *flag = nullptr;
    bool owned = false;
    if (!run_check) {
        // offsets checked (and the flag set) by the caller beforehand
        flag = f->query_detects_dense ? flag_word : nullptr;
    } else if (f->query_detects_dense) {
        if (flag_word) {
            flag = flag_word;
        } else if (cudaMallocFromPoolAsync(reinterpret_cast<void **>(&flag), sizeof(int), f->flag_pool, st) ==
                   cudaSuccess) {
            owned = true;
        } else {
            cudaGetLastError();
            flag = nullptr;
        }
    }
    int rc = run_check ? launch_check(f, offsets, n, st, flag) : SBF_OK;
    if (rc == SBF_OK) {
        sbf::LaunchArgs la = make_args(f, seq, offsets, n, out_bits, device_seq);
        la.nonuniform = flag;
        la.out_words_end = out_words_end;
        rc = launch(f->query_kernel, f->grid_query, f->threads_query, la, st);
    }
    if (owned) cudaFreeAsync(flag, st);
    return rc;
}

extern "C" {

const char *sbf_last_error(void) { return g_last_error.c_str(); }

sbf_filter *sbf_create(uint64_t num_bits, int k, int m, int s, int H, uint64_t seed) {
    return sbf_create_alphabet(num_bits, k, m, s, H, seed, SBF_ALPHABET_DNA);
}

sbf_filter *sbf_create_alphabet(uint64_t num_bits, int k, int m, int s, int H, uint64_t seed, int alphabet) {
    return sbf_create_ex(num_bits, k, m, s, H, seed, alphabet, 0);
}

int sbf_get_flags(const sbf_filter *f) {
    if (!f) return -1;
    return (f->sectors ? SBF_FLAG_HASHED_SECTORS : 0) | (f->runtime_requested ? SBF_FLAG_RUNTIME_KERNELS : 0);
}

sbf_filter *sbf_create_ex(uint64_t num_bits, int k, int m, int s, int H, uint64_t seed, int alphabet, int flags) {
    g_last_error.clear();
    if (flags & ~(SBF_FLAG_HASHED_SECTORS | SBF_FLAG_RUNTIME_KERNELS)) {
        fail(SBF_ERR_INVALID_ARG, "unknown flags 0x%x", flags);
        return nullptr;
    }
    if (num_bits < 1) {
        fail(SBF_ERR_INVALID_ARG, "num_bits must be >= 1");
        return nullptr;
    }
    if (alphabet < SBF_ALPHABET_DNA || alphabet > SBF_ALPHABET_DNA_TRIPLET) {
        fail(SBF_ERR_INVALID_ARG, "unknown alphabet %d", alphabet);
        return nullptr;
    }
    // Sec. IV-C: a k-mer packs into one 64-bit word
    const int kmax = alphabet == SBF_ALPHABET_PROTEIN ? 12 : alphabet == SBF_ALPHABET_DNA_TRIPLET ? 10 : 32;
    if (k < 1 || k > kmax || m < 1 || m > k || s < 1 || s > k) {
        fail(SBF_ERR_INVALID_ARG, "need 1 <= m <= k <= %d and 1 <= s <= k (k=%d m=%d s=%d)", kmax, k, m, s);
        return nullptr;
    }
    if (H < 1 || H > sbf::kMaxH) {
        fail(SBF_ERR_INVALID_ARG, "H must be in 1..%d, got %d", sbf::kMaxH, H);
        return nullptr;
    }
    const uint64_t need = num_bits / 256 + (num_bits % 256 != 0);
    uint64_t shards = 1;
    while (shards < need) shards <<= 1;
    if (shards > (1ull << 40)) {
        fail(SBF_ERR_INVALID_ARG, "filter too large: %llu shards", (unsigned long long)shards);
        return nullptr;
    }
    auto *f = new sbf_filter;
    f->k = k;
    f->m = m;
    f->s = s;
    f->H = H;
    f->alphabet = alphabet;
    f->seed = seed;
    f->sectors = (flags & SBF_FLAG_HASHED_SECTORS) ? 1 : 0;
    // hash-chosen sectors (H < 4) run on the runtime-parameter kernels: the
    // compile-time specialisations keep the paper's layout only
    f->runtime_requested = (flags & SBF_FLAG_RUNTIME_KERNELS) != 0;
    f->runtime_only = f->runtime_requested || (f->sectors && H < 4);
    const bool may_specialise = !f->runtime_only;
    f->num_shards = shards;
    cudaError_t e = cudaGetDevice(&f->device);
    int sms = 0;
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, f->device);
    if (e != cudaSuccess) {
        cuda_fail(e, "no usable CUDA device");
        delete f;
        return nullptr;
    }
    e = cudaMalloc(reinterpret_cast<void **>(&f->words), shards * 32);
    if (e != cudaSuccess) {
        fail(SBF_ERR_OOM, "cudaMalloc of %llu bytes: %s", (unsigned long long)(shards * 32), cudaGetErrorString(e));
        cudaGetLastError();
        delete f;
        return nullptr;
    }
    e = cudaMalloc(reinterpret_cast<void **>(&f->status), sizeof(int));
    if (e == cudaSuccess) e = cudaMemset(f->words, 0, shards * 32);
    if (e == cudaSuccess) e = cudaMemset(f->status, 0, sizeof(int));
    if (e != cudaSuccess) {
        cuda_fail(e, "filter initialisation");
        cudaFree(f->words);
        cudaFree(f->status);
        delete f;
        return nullptr;
    }
    const void *ins = nullptr, *qry = nullptr;
    int threads = 0;
    // The strip kernels key runs by shard with bit 31 marking invalid k-mers.
    int threads_query = 0;
    if (alphabet != SBF_ALPHABET_DNA && may_specialise && shards <= (1ull << 31) &&
        sbf::find_alphabet_strip(alphabet, k, m, s, H, &ins, &qry, &threads)) {
        f->specialized = true;
        f->strip = true;
        threads_query = threads;
    } else if (alphabet != SBF_ALPHABET_DNA) {
        bool spec = false;
        sbf::find_alphabet_kernels(alphabet, k, m, s, H, &ins, &qry, &spec, may_specialise);
        f->specialized = spec;
        threads = 256;
    } else if (may_specialise && shards <= (1ull << 31) && sbf::find_specialized(k, m, s, H, &ins, &qry, &threads)) {
        f->specialized = true;
        f->strip = true;
    } else {
        ins = sbf::generic_insert_kernel();
        qry = sbf::generic_query_kernel();
        threads = 256;
    }
    if (threads_query == 0) threads_query = threads;
    // a DNA filter several times larger than L2: every run's shard update is a
    // DRAM read-modify-write, and the insert flushes runs through its warp's
    // run queue (one 32-byte request per run) where it has that form
    if (alphabet == SBF_ALPHABET_DNA && f->strip) {
        int l2 = 0;
        if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, f->device) == cudaSuccess && l2 > 0 &&
            shards * 32 > (uint64_t)sbf::kQueuedInsertL2Multiple * (uint64_t)l2)
            if (const void *q = sbf::queued_insert_kernel(k, m, s, H)) ins = q;
        cudaGetLastError();
    }
    f->insert_kernel = ins;
    f->query_kernel = qry;
    f->threads = threads;
    f->threads_query = threads_query;
    f->grid_insert = grid_for(ins, threads, sms);
    f->grid_query = grid_for(qry, threads_query, sms);
    if (alphabet == SBF_ALPHABET_DNA && may_specialise && shards <= (1ull << 31)) {
        f->dense_query_kernel = sbf::dense_query_kernel(k, m, s, H, &f->threads_dense);
        if (f->dense_query_kernel) {
            f->grid_dense = grid_for(f->dense_query_kernel, f->threads_dense, sms);
            if (f->dense_query_kernel == f->query_kernel) {
                // the per-call uniformity words come from a pool of the
                // filter's own that keeps its memory between calls
                cudaMemPoolProps props = {};
                props.allocType = cudaMemAllocationTypePinned;
                props.location.type = cudaMemLocationTypeDevice;
                props.location.id = f->device;
                if (cudaMemPoolCreate(&f->flag_pool, &props) == cudaSuccess) {
                    uint64_t keep = UINT64_MAX;
                    cudaMemPoolSetAttribute(f->flag_pool, cudaMemPoolAttrReleaseThreshold, &keep);
                    // map the pool's memory now, not under the first queries
                    void *warm = nullptr;
                    if (cudaMallocFromPoolAsync(&warm, size_t(1) << 20, f->flag_pool, 0) == cudaSuccess) {
                        cudaFreeAsync(warm, 0);
                        cudaStreamSynchronize(0);
                    }
                    cudaGetLastError();
                    f->query_detects_dense = true;
                } else {
                    cudaGetLastError();
                    f->flag_pool = nullptr;
                }
            }
        }
    }
    f->grid_check = 4 * sms;
    return f;
}

void sbf_destroy(sbf_filter *f) {
    if (!f) return;
    int prev = -1;
    cudaGetDevice(&prev);
    if (prev != f->device) cudaSetDevice(f->device);
    cudaDeviceSynchronize();
    sbf::destroy_stager(f->stager);
    cudaFree(f->words);
    cudaFree(f->status);
    if (f->flag_pool) cudaMemPoolDestroy(f->flag_pool);
    if (prev >= 0 && prev != f->device) cudaSetDevice(prev);
    delete f;
}

uint64_t sbf_num_shards(const sbf_filter *f) { return f ? f->num_shards : 0; }

int sbf_get_params(const sbf_filter *f, int *k, int *m, int *s, int *H, uint64_t *seed) {
    if (!f) return fail(SBF_ERR_INVALID_ARG, "NULL filter");
    if (k) *k = f->k;
    if (m) *m = f->m;
    if (s) *s = f->s;
    if (H) *H = f->H;
    if (seed) *seed = f->seed;
    return SBF_OK;
}

int sbf_is_specialized(const sbf_filter *f) { return f && f->specialized ? 1 : 0; }

int sbf_get_alphabet(const sbf_filter *f) { return f ? f->alphabet : -1; }

int sbf_insert(sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n, void *stream) {
    if (!f || !seq || !offsets || n < 0) return fail(SBF_ERR_INVALID_ARG, "sbf_insert: bad arguments");
    if (n == 0) return SBF_OK;
    if (int rc = check_device(f)) return rc;
    return sbf::launch_insert(f, seq, offsets, n, stream, true);
}

int sbf_query(const sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n,
              uint32_t *out_bits, void *stream) {
    if (!f || !seq || !offsets || !out_bits || n < 0)
        return fail(SBF_ERR_INVALID_ARG, "sbf_query: bad arguments");
    if (n == 0) return SBF_OK;
    if (int rc = check_device(f)) return rc;
    return sbf::launch_query(f, seq, offsets, n, out_bits, stream, true);
}

int sbf_query_dense(const sbf_filter *f, const char *seq, int64_t n_records, int64_t record_len,
                    uint32_t *out_bits, void *stream) {
    if (!f || !seq || !out_bits || n_records < 0 || record_len < 1)
        return fail(SBF_ERR_INVALID_ARG, "sbf_query_dense: bad arguments");
    if (f->alphabet != SBF_ALPHABET_DNA) return fail(SBF_ERR_INVALID_ARG, "sbf_query_dense: DNA filters only");
    if (n_records == 0) return SBF_OK;
    if (n_records > (int64_t(1) << 40) / record_len)
        return fail(SBF_ERR_INVALID_ARG, "sbf_query_dense: batch too large");
    if (int rc = check_device(f)) return rc;
    sbf::LaunchArgs la = make_args(f, seq, nullptr, n_records, out_bits, true);
    la.rec_len = record_len;
    // one record per strip when the filter has a dense strip kernel and the
    // records fit it; the runtime-parameter kernel otherwise
    if (f->dense_query_kernel && record_len <= sbf::kDenseMax)
        return launch(f->dense_query_kernel, f->grid_dense, f->threads_dense, la, as_stream(stream));
    return launch(sbf::generic_query_kernel(), f->grid_check * 2, 256, la, as_stream(stream));
}

int sbf_copy_bits(const sbf_filter *f, void *dst, uint64_t dst_bytes, void *stream) {
    if (!f || !dst) return fail(SBF_ERR_INVALID_ARG, "sbf_copy_bits: bad arguments");
    const uint64_t bytes = f->num_shards * 32;
    if (dst_bytes < bytes) return fail(SBF_ERR_INVALID_ARG, "sbf_copy_bits: need %llu bytes", (unsigned long long)bytes);
    cudaError_t e = cudaMemcpyAsync(dst, f->words, bytes, cudaMemcpyDefault, as_stream(stream));
    return e == cudaSuccess ? SBF_OK : cuda_fail(e, "sbf_copy_bits");
}

int sbf_load_bits(sbf_filter *f, const void *src, uint64_t src_bytes, void *stream) {
    if (!f || !src) return fail(SBF_ERR_INVALID_ARG, "sbf_load_bits: bad arguments");
    const uint64_t bytes = f->num_shards * 32;
    if (src_bytes != bytes) return fail(SBF_ERR_INVALID_ARG, "sbf_load_bits: need exactly %llu bytes", (unsigned long long)bytes);
    cudaError_t e = cudaMemcpyAsync(f->words, src, bytes, cudaMemcpyDefault, as_stream(stream));
    return e == cudaSuccess ? SBF_OK : cuda_fail(e, "sbf_load_bits");
}

int sbf_clear(sbf_filter *f, void *stream) {
    if (!f) return fail(SBF_ERR_INVALID_ARG, "NULL filter");
    cudaError_t e = cudaMemsetAsync(f->words, 0, f->num_shards * 32, as_stream(stream));
    return e == cudaSuccess ? SBF_OK : cuda_fail(e, "sbf_clear");
}

int sbf_test_wait_timeout(sbf_filter *f, int polls, void *stream) {
    if (!f || polls < 1) return fail(SBF_ERR_INVALID_ARG, "sbf_test_wait_timeout: bad arguments");
    if (!f->strip) return fail(SBF_ERR_INVALID_ARG, "sbf_test_wait_timeout: the filter's kernels have no bounded waits");
    if (int rc = check_device(f)) return rc;
    sbf::LaunchArgs la = make_args(f, nullptr, nullptr, 0, nullptr);
    la.wait_test = polls;
    return launch(f->insert_kernel, 1, f->threads, la, as_stream(stream));
}

int sbf_get_status(sbf_filter *f, void *stream) {
    if (!f) return fail(SBF_ERR_INVALID_ARG, "NULL filter");
    cudaStream_t st = as_stream(stream);
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "stream");
    int st_word = 0;
    e = cudaMemcpy(&st_word, f->status, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (st_word) {
        e = cudaMemset(f->status, 0, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "status clear");
        if (st_word & sbf::kStatusBadOffsets)
            return fail(SBF_ERR_BAD_OFFSETS, "malformed offsets (decreasing or negative); work was skipped");
        if (st_word & sbf::kStatusTimeout)
            return fail(SBF_ERR_CUDA, "a bounded device wait timed out; the call's work is incomplete");
    }
    return SBF_OK;
}

}  // extern "C"
