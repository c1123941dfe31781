// Paged prefill kernel instantiated for head dimension 512.
#include "pgqa_prefill.cuh"

namespace pgqa {
cudaError_t launch_prefill_hd512(const PrefillLaunchArgs &a, bool set_attr) { return launch_prefill<512>(a, set_attr); }
}  // namespace pgqa
