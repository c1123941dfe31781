// Paged prefill for head dimension 128: the tcgen05 kernel.
#include "pgqa_prefill_tc.cuh"

namespace pgqa {
cudaError_t launch_prefill_hd128(const PrefillLaunchArgs &a, bool set_attr) { return launch_prefill_tc<128>(a, set_attr); }
}  // namespace pgqa
