// Split-KV decode kernels instantiated for head dimension 256.
#include "pgqa_launch.cuh"

namespace pgqa {
cudaError_t launch_decode_hd256(const LaunchArgs &a, bool set_attr) { return launch_decode<256>(a, set_attr); }
int cluster_capacity_hd256(int cluster) { return cluster_capacity<256>(cluster); }
int ctas_per_sm_hd256() { return ctas_per_sm<256>(); }
cudaError_t launch_combine_hd256(const DecodeParams &p, cudaStream_t stream) { return launch_combine<256>(p, stream); }
}  // namespace pgqa
