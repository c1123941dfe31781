// Paged prefill kernel instantiated for head dimension 256.
#include "pgqa_prefill.cuh"

namespace pgqa {
cudaError_t launch_prefill_hd256(const PrefillLaunchArgs &a, bool set_attr) { return launch_prefill<256>(a, set_attr); }
}  // namespace pgqa
