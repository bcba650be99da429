// sbf_kernels.h -- internal interface between the C ABI and the kernels.
#pragma once

#include <cstdint>

#include "sbf_device.cuh"

namespace sbf {

// Runtime-parameter kernels (any valid k, m, s, H), sbf_generic.cu.
const void *generic_insert_kernel();
const void *generic_query_kernel();
__global__ void check_offsets_kernel(const int64_t *off, int64_t n, int *status, int *nonuniform);

// Dense batches (fixed-length records): the strip-kernel query for records of
// at most kDenseMax bytes at (k, m, s, H), or nullptr.  The same kernel is the
// filter's CSR query there: it runs a CSR batch whose records all have one
// length <= kDenseMax, starting at offset 0, as a dense batch.
constexpr int kDenseMax = 160;
const void *dense_query_kernel(int k, int m, int s, int H, int *threads);

// The insert strip kernel with the warp run-queue flush (FQ = 1) at (k, m,
// s, H), or nullptr; the same block size as the filter's insert kernel.
const void *queued_insert_kernel(int k, int m, int s, int H);
// Filters of more than this many L2 sizes take the queued insert.
constexpr int kQueuedInsertL2Multiple = 8;

// The protein and triplet alphabets' strip-kernel specialisations (shards
// <= 2^31): false when (alphabet, k, m, s, H) has none.
bool find_alphabet_strip(int alphabet, int k, int m, int s, int H, const void **insert, const void **query,
                         int *threads);

// Protein and DNA-triplet kernels, sbf_alphabet.cu: the compile-time
// specialisation for (k, m, s, H) when there is one (*specialized = true),
// else the runtime-parameter kernel.  False for any other alphabet.  256
// threads per block.
bool find_alphabet_kernels(int alphabet, int k, int m, int s, int H, const void **insert, const void **query,
                           bool *specialized, bool may_specialise = true);

// Compile-time specialised kernels.  Returns false when (k, m, s, H) has no
// specialisation; *insert / *query / *threads are set otherwise.
bool find_specialized(int k, int m, int s, int H, const void **insert, const void **query,
                      int *threads);

}  // namespace sbf
