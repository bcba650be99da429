// The paper's Pareto-optimal operating point k=31, m=16, s=28, H=4
// ("cuSBF", Sec. V-B), in a unit of its own so that it compiles first.
#include "sbf_registry.h"

namespace sbf {
SBF_REGISTER_ONE(Main, 31, 16, 28, 4)
}  // namespace sbf
