// Sweep-grid specialisations for k = 31, m = 18, s = 24, H in {1, 2, 4, 6, 8}.
#include "sbf_registry.h"

namespace sbf {
SBF_REGISTER_MS(18, 24)
}  // namespace sbf
