// The paper's Pareto-optimal operating point k=31, m=16, s=28, H=4
// ("cuSBF", Sec. V-B), in a unit of its own so that it compiles first.  Its
// query kernel is the dense-capable one (records of at most kDenseMax bytes,
// one per strip): sbf_query_dense calls it with a record length, and the CSR
// query calls it too, where it takes the dense geometry for a batch whose
// records the offsets check found to be all of one length.  Its insert also
// comes with the run-queue flush (FQ = 1) for filters much larger than L2.
#include "sbf_kernels.h"
#include "sbf_registry.h"

namespace sbf {
using MainDense = StripCfg<31, 16, 28, 4, 0, kDenseMax>;
static_assert(MainDense::NT == StripCfg<31, 16, 28, 4>::NT, "insert and query share a block size");

extern const StripEntry kStripEntriesMain[];
extern const int kStripCountMain;
const StripEntry kStripEntriesMain[] = {
    StripEntry{31, 16, 28, 4, reinterpret_cast<const void *>(&strip_kernel<31, 16, 28, 4, false, 0>),
               reinterpret_cast<const void *>(&strip_kernel<31, 16, 28, 4, true, 0, kDenseMax>),
               MainDense::NT}};
const int kStripCountMain = 1;

const void *queued_insert_kernel(int k, int m, int s, int H) {
    if (k == 31 && m == 16 && s == 28 && H == 4)
        return reinterpret_cast<const void *>(&strip_kernel<31, 16, 28, 4, false, 0, 0, 1>);
    return nullptr;
}

const void *dense_query_kernel(int k, int m, int s, int H, int *threads) {
    if (k == 31 && m == 16 && s == 28 && H == 4) {
        *threads = MainDense::NT;
        return reinterpret_cast<const void *>(&strip_kernel<31, 16, 28, 4, true, 0, kDenseMax>);
    }
    return nullptr;
}
}  // namespace sbf
