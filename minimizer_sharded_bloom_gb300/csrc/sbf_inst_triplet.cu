// The DNA-triplet alphabet's benchmarked point (k=10, m=5, s=8, H=4; Sec.
// IV-A's 6-bit codons) on the strip kernel, three frame passes per tile.
#include "sbf_registry.h"

namespace sbf {
extern const StripEntry kStripEntriesTriplet[];
extern const int kStripCountTriplet;
const StripEntry kStripEntriesTriplet[] = {strip_entry<10, 5, 8, 4, kAlphabetTriplet>()};
const int kStripCountTriplet = 1;
}  // namespace sbf
