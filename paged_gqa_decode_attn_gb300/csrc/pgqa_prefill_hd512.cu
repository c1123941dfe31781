// Paged prefill for head dimension 512: the mma.sync kernel (O of 128 rows x 512 dims would fill
// all of tensor memory).
#include "pgqa_prefill.cuh"

namespace pgqa {
cudaError_t launch_prefill_hd512(const PrefillLaunchArgs &a, bool set_attr) { return launch_prefill<512>(a, set_attr); }
}  // namespace pgqa
