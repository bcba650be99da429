// The paper's larger hash counts at the operating point k=31, m=16, s=28:
// H = 12 and 16 (Fig. 4 sweeps H in {4, 8, 12, 16}), which use the salted
// multiply of Sec. IV-G instead of bit-slicing.
#include "sbf_registry.h"

namespace sbf {
extern const StripEntry kStripEntriesLargeH[];
extern const int kStripCountLargeH;
const StripEntry kStripEntriesLargeH[] = {strip_entry<31, 16, 28, 12>(), strip_entry<31, 16, 28, 16>()};
const int kStripCountLargeH = 2;
}  // namespace sbf
