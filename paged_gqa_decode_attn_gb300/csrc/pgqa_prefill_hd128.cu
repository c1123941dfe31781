// Paged prefill kernel instantiated for head dimension 128.
#include "pgqa_prefill.cuh"

namespace pgqa {
cudaError_t launch_prefill_hd128(const PrefillLaunchArgs &a, bool set_attr) { return launch_prefill<128>(a, set_attr); }
}  // namespace pgqa
