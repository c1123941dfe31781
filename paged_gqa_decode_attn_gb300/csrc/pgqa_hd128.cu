// Split-KV decode kernels instantiated for head dimension 128.
#include "pgqa_launch.cuh"

namespace pgqa {
cudaError_t launch_decode_hd128(const LaunchArgs &a, bool set_attr) { return launch_decode<128>(a, set_attr); }
int cluster_capacity_hd128(int cluster) { return cluster_capacity<128>(cluster); }
int ctas_per_sm_hd128() { return ctas_per_sm<128>(); }
cudaError_t launch_combine_hd128(const DecodeParams &p, cudaStream_t stream) { return launch_combine<128>(p, stream); }
}  // namespace pgqa
