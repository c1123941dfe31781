// Paged prefill for head dimension 512: the tcgen05 kernel as CTA pairs, each
// CTA over half of the head dims (O of 128 rows x 512 dims would fill all of
// one SM's tensor memory).
#include "pgqa_prefill_tc.cuh"

namespace pgqa {
cudaError_t launch_prefill_hd512(const PrefillLaunchArgs &a, bool set_attr) { return launch_prefill_tc<512>(a, set_attr); }
int prefill_pair_capacity_hd512()
{
    if (cudaFuncSetAttribute(prefill_tc_kernel<512, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TcGeo<512>::kAlloc) != cudaSuccess)
        return 0;
    return prefill_tc_pair_capacity<512>();
}
}  // namespace pgqa
