// sbf_registry.h -- which (k, m, s, H) get a compile-time specialised kernel.
//
// The paper's operating point k=31, m=16, s=28, H=4 ("cuSBF", Sec. V-B) plus
// the benchmarked sweep grid at k = 31: s in {20, 24, 28, 31}, m in {12, 14, 16,
// 18, 21}, H in {1, 2, 4, 6, 8}.  Every other valid combination runs the
// runtime-parameter kernel, with identical results.  Each (m, s) pair is one
// translation unit (sbf_inst_m<m>_s<s>.cu) so that they compile in parallel.
#pragma once

#include "sbf_strip.cuh"

// (m, s) units of the sweep grid
#define SBF_SWEEP_UNITS(X)                                                  \
    X(12, 20) X(12, 24) X(12, 28) X(12, 31) X(14, 20) X(14, 24) X(14, 28)   \
    X(14, 31) X(16, 20) X(16, 24) X(16, 28) X(16, 31) X(18, 20) X(18, 24)   \
    X(18, 28) X(18, 31) X(21, 20) X(21, 24) X(21, 28) X(21, 31)

namespace sbf {

// The main operating point lives in its own unit; the grid unit that would
// repeat it registers an empty slot instead of a second copy of the kernels.
template <int K, int M, int S, int H>
inline StripEntry grid_entry() {
    if constexpr (K == 31 && M == 16 && S == 28 && H == 4) {
        return StripEntry{0, 0, 0, 0, nullptr, nullptr, 0};
    } else {
        return strip_entry<K, M, S, H>();
    }
}

}  // namespace sbf

#define SBF_GRID_ENTRY(K, M, S, H) grid_entry<K, M, S, H>(),

#define SBF_REGISTER_MS(M, S)                                                        \
    extern const StripEntry kStripEntriesM##M##S##_[];                               \
    extern const int kStripCountM##M##S##_;                                          \
    const StripEntry kStripEntriesM##M##S##_[] = {                                   \
        SBF_GRID_ENTRY(31, M, S, 1) SBF_GRID_ENTRY(31, M, S, 2) SBF_GRID_ENTRY(31, M, S, 4) \
        SBF_GRID_ENTRY(31, M, S, 6) SBF_GRID_ENTRY(31, M, S, 8)};                    \
    const int kStripCountM##M##S##_ = 5;

#define SBF_REGISTER_ONE(NAME, K, M, S, H)                                   \
    extern const StripEntry kStripEntries##NAME[];                           \
    extern const int kStripCount##NAME;                                      \
    const StripEntry kStripEntries##NAME[] = {strip_entry<K, M, S, H>()};    \
    const int kStripCount##NAME = 1;
