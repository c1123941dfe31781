// Split-KV decode kernels instantiated for head dimension 64.
#include "pgqa_launch.cuh"

namespace pgqa {
cudaError_t launch_decode_hd64(const LaunchArgs &a, bool set_attr) { return launch_decode<64>(a, set_attr); }
int cluster_capacity_hd64(int cluster) { return cluster_capacity<64>(cluster); }
int ctas_per_sm_hd64() { return ctas_per_sm<64>(); }
cudaError_t launch_combine_hd64(const DecodeParams &p, cudaStream_t stream) { return launch_combine<64>(p, stream); }
}  // namespace pgqa
