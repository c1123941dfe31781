// Paged prefill kernel instantiated for head dimension 64.
#include "pgqa_prefill.cuh"

namespace pgqa {
cudaError_t launch_prefill_hd64(const PrefillLaunchArgs &a, bool set_attr) { return launch_prefill<64>(a, set_attr); }
}  // namespace pgqa
