// Paged prefill for head dimension 64: the tcgen05 kernel.
#include "pgqa_prefill_tc.cuh"

namespace pgqa {
cudaError_t launch_prefill_hd64(const PrefillLaunchArgs &a, bool set_attr) { return launch_prefill_tc<64>(a, set_attr); }
}  // namespace pgqa
