// Paged prefill for head dimension 512: the tcgen05 kernel as CTA pairs, each
// CTA over half of the head dims (O of 128 rows x 512 dims would fill all of
// one SM's tensor memory).
#include "pgqa_prefill_tc.cuh"

namespace pgqa {
cudaError_t launch_prefill_hd512(const PrefillLaunchArgs &a, bool set_attr) { return launch_prefill_tc<512>(a, set_attr); }
}  // namespace pgqa
