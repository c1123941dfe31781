// Host-side launch of the split kernel (and, without merge counters, the
// combine kernel) for one head dimension.  Each pgqa_hd*.cu instantiates one
// head dimension so the four compile in parallel.
#pragma once

#include "pgqa_device.cuh"

namespace pgqa {

struct LaunchArgs {
    DecodeParams p;
    const CUtensorMap *tm_k;
    const CUtensorMap *tm_v;
    cudaStream_t stream;
};

// Dynamic shared memory the split kernel of head dimension `hd` asks for.
int split_kernel_smem_bytes(int hd);

template <int HD>
cudaError_t launch_decode(const LaunchArgs &a, bool set_attr)
{
    if (set_attr) {
        cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<HD>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Smem<HD>::kAlloc);
        if (e != cudaSuccess)
            return e;
    }
    const DecodeParams &p = a.p;
    dim3 grid(p.splits, p.nkv * p.hsg, p.rows);
    decode_split_kernel<HD><<<grid, Geo<HD>::kThreads, Smem<HD>::kAlloc, a.stream>>>(*a.tm_k, *a.tm_v, p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return e;
    if (p.splits > 1 && p.counters == nullptr) {
        decode_combine_kernel<HD><<<p.rows * p.nh, combine_threads<HD>(), 0, a.stream>>>(p);
        e = cudaGetLastError();
    }
    return e;
}

cudaError_t launch_decode_hd64(const LaunchArgs &a, bool set_attr);
cudaError_t launch_decode_hd128(const LaunchArgs &a, bool set_attr);
cudaError_t launch_decode_hd256(const LaunchArgs &a, bool set_attr);
cudaError_t launch_decode_hd512(const LaunchArgs &a, bool set_attr);

}  // namespace pgqa
