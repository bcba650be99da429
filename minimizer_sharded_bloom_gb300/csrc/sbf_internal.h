// sbf_internal.h -- the filter object and helpers shared by the C ABI units.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "sbf.h"

struct sbf_filter {
    int device = 0;
    int k = 0, m = 0, s = 0, H = 0;
    int alphabet = SBF_ALPHABET_DNA;
    uint64_t seed = 0;
    int sectors = 0;            // 1: hash-chosen sectors for H < 4 (SBF_FLAG_HASHED_SECTORS)
    uint64_t num_shards = 0;
    uint64_t *words = nullptr;  // num_shards * 4 words
    int *status = nullptr;      // sticky device status
    const void *insert_kernel = nullptr;
    const void *query_kernel = nullptr;
    int threads = 256;          // threads per block of the insert kernel
    int threads_query = 256;    // ... and of the query kernel
    const void *dense_query_kernel = nullptr;  // dense batches (strip kernel), if any
    bool query_detects_dense = false;          // query_kernel runs uniform CSR batches as dense
    cudaMemPool_t flag_pool = nullptr;         // ... with a per-call flag word from this pool
    int threads_dense = 0, grid_dense = 0;
    int grid_insert = 0, grid_query = 0;
    int grid_check = 0;
    bool specialized = false;
    bool runtime_only = false;  // never a compile-time specialisation (the flag, or hashed sectors)
    bool runtime_requested = false;  // SBF_FLAG_RUNTIME_KERNELS given at creation
    bool strip = false;         // insert/query kernels are strip kernels (bounded mbarrier waits)
    void *stager = nullptr;     // host-facing staging buffers, created on first use
    int64_t host_chunk = int64_t(1) << 25;  // host-facing chunk, in positions
    int host_mode = 0;          // 0: read host buffers in place when possible; 1: always stage
};

namespace sbf {
// Input bytes per symbol of an alphabet (3 for DNA triplets, else 1).
inline int symbol_bytes(int alphabet) { return alphabet == SBF_ALPHABET_DNA_TRIPLET ? 3 : 1; }
// Bytes one k-mer of f covers.
inline int64_t kmer_bytes(const sbf_filter *f) { return (int64_t)f->k * symbol_bytes(f->alphabet); }
// Records the calling thread's error message and returns `code`.
int set_error(int code, const char *fmt, ...);
void destroy_stager(void *stager);
// Launch the check + insert/query kernels; device_seq = false when seq is host
// memory read in place (the kernel then loads tile bytes without TMA).
// run_check = false: the caller has already checked these offsets on the
// device (and, for a query, set flag_word from that check or passed nullptr).
int launch_insert(sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n, void *stream,
                  bool device_seq, bool run_check = true);
// flag_word: a device int the call may use to detect a uniform batch (the
// no-alloc path passes one of its own); nullptr: allocated per call.
// out_words_end: answer words at or past this index are left unwritten.
int launch_query(const sbf_filter *f, const char *seq, const int64_t *offsets, int64_t n,
                 uint32_t *out_bits, void *stream, bool device_seq, int *flag_word = nullptr,
                 int64_t out_words_end = INT64_MAX, bool run_check = true);
// The device check of an offsets array (device-accessible) alone; a bad array
// sets the sticky status, which every later launch of the filter honours.
// nonuniform (zeroed here first): set when record lengths differ.
int launch_offsets_check(const sbf_filter *f, const int64_t *offsets, int64_t n, void *stream,
                         int *nonuniform = nullptr);
}  // namespace sbf
