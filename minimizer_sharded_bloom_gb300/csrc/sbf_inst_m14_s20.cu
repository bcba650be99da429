// Sweep-grid specialisations for k = 31, m = 14, s = 20, H in {1, 2, 4, 6, 8}.
#include "sbf_registry.h"

namespace sbf {
SBF_REGISTER_MS(14, 20)
}  // namespace sbf
