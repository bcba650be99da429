// The paper's Pareto-optimal operating point k=31, m=16, s=28, H=4
// ("cuSBF", Sec. V-B), in a unit of its own so that it compiles first; with
// the dense-batch query (records of at most kDenseMax bytes, one per strip).
#include "sbf_kernels.h"
#include "sbf_registry.h"

namespace sbf {
SBF_REGISTER_ONE(Main, 31, 16, 28, 4)

const void *dense_query_kernel(int k, int m, int s, int H, int *threads) {
    if (k == 31 && m == 16 && s == 28 && H == 4) {
        *threads = StripCfg<31, 16, 28, 4, 0, kDenseMax>::NT;
        return reinterpret_cast<const void *>(&strip_kernel<31, 16, 28, 4, true, 0, kDenseMax>);
    }
    return nullptr;
}
}  // namespace sbf
