// Split-KV decode kernels instantiated for head dimension 512.
#include "pgqa_launch.cuh"

namespace pgqa {
cudaError_t launch_decode_hd512(const LaunchArgs &a, bool set_attr) { return launch_decode<512>(a, set_attr); }
cudaError_t launch_combine_hd512(const DecodeParams &p, cudaStream_t stream) { return launch_combine<512>(p, stream); }
int cluster_capacity_hd512(int cluster) { return cluster_capacity<512>(cluster); }
int ctas_per_sm_hd512() { return ctas_per_sm<512>(); }
}  // namespace pgqa
