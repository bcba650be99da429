// The protein alphabet's benchmarked point (k=12, m=8, s=10, H=4; Sec. IV-A's
// 5-bit symbols) on the strip kernel.
#include "sbf_registry.h"

namespace sbf {
extern const StripEntry kStripEntriesProtein[];
extern const int kStripCountProtein;
const StripEntry kStripEntriesProtein[] = {strip_entry<12, 8, 10, 4, kAlphabetProtein>()};
const int kStripCountProtein = 1;
}  // namespace sbf
