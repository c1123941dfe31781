// Paged prefill for head dimension 256: the tcgen05 kernel.
#include "pgqa_prefill_tc.cuh"

namespace pgqa {
cudaError_t launch_prefill_hd256(const PrefillLaunchArgs &a, bool set_attr) { return launch_prefill_tc<256>(a, set_attr); }
}  // namespace pgqa
