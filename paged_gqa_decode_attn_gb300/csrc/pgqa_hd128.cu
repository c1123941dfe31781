// Split-KV decode kernels instantiated for head dimension 128.
#include "pgqa_launch.cuh"

namespace pgqa {
cudaError_t launch_decode_hd128(const LaunchArgs &a, bool set_attr) { return launch_decode<128>(a, set_attr); }
int cluster_capacity_hd128(int cluster) { return cluster_capacity<128>(cluster); }
}  // namespace pgqa
