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
    cudaError_t e;
    if (p.cluster > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(Geo<HD>::kThreads);
        cfg.dynamicSmemBytes = Smem<HD>::kAlloc;
        cfg.stream = a.stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = p.cluster;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, decode_split_kernel<HD>, *a.tm_k, *a.tm_v, p);
    } else {
        decode_split_kernel<HD><<<grid, Geo<HD>::kThreads, Smem<HD>::kAlloc, a.stream>>>(*a.tm_k, *a.tm_v, p);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess)
        return e;
    if (p.splits > 1 && p.counters == nullptr) {
        decode_combine_kernel<HD><<<p.rows * p.nh, combine_threads<HD>(), 0, a.stream>>>(p);
        e = cudaGetLastError();
    }
    return e;
}

// How many clusters of `cluster` split CTAs can be resident at once (0: the
// on-chip merge cannot be used).  Also sets the kernel's attributes.
template <int HD>
int cluster_capacity(int cluster)
{
    if (cudaFuncSetAttribute(decode_split_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<HD>::kAlloc) != cudaSuccess)
        return 0;
    if (cluster > kMaxCluster)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster, 1, 1);
    cfg.blockDim = dim3(Geo<HD>::kThreads);
    cfg.dynamicSmemBytes = Smem<HD>::kAlloc;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, decode_split_kernel<HD>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

int cluster_capacity_hd64(int cluster);
int cluster_capacity_hd128(int cluster);
int cluster_capacity_hd256(int cluster);
int cluster_capacity_hd512(int cluster);

cudaError_t launch_decode_hd64(const LaunchArgs &a, bool set_attr);
cudaError_t launch_decode_hd128(const LaunchArgs &a, bool set_attr);
cudaError_t launch_decode_hd256(const LaunchArgs &a, bool set_attr);
cudaError_t launch_decode_hd512(const LaunchArgs &a, bool set_attr);

}  // namespace pgqa
