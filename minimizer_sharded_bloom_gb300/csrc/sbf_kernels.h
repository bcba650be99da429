// sbf_kernels.h -- internal interface between the C ABI and the kernels.
#pragma once

#include <cstdint>

#include "sbf_device.cuh"

namespace sbf {

// Runtime-parameter kernels (any valid k, m, s, H), sbf_generic.cu.
const void *generic_insert_kernel();
const void *generic_query_kernel();
__global__ void check_offsets_kernel(const int64_t *off, int64_t n, int *status);

// Protein and DNA-triplet kernels (runtime k, m, s, H), sbf_alphabet.cu;
// nullptr for any other alphabet.  256 threads per block.
const void *alphabet_insert_kernel(int alphabet);
const void *alphabet_query_kernel(int alphabet);

// Compile-time specialised kernels.  Returns false when (k, m, s, H) has no
// specialisation; *insert / *query / *threads are set otherwise.
bool find_specialized(int k, int m, int s, int H, const void **insert, const void **query,
                      int *threads);

}  // namespace sbf
