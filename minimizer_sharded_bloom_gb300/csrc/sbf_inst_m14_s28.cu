// Sweep-grid specialisations for k = 31, m = 14, s = 28, H in {1, 2, 4, 6, 8}.
#include "sbf_registry.h"

namespace sbf {
SBF_REGISTER_MS(14, 28)
}  // namespace sbf
