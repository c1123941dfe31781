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

// The combine kernel alone, over rows * nh (row, head) pairs of p.splits
// partials in p.part_o / p.part_ml, into p.o.  It may overlap the tail of the
// kernel before it (programmatic dependent launch) and waits for it before
// reading the partials.
template <int HD>
cudaError_t launch_combine(const DecodeParams &p, cudaStream_t stream)
{
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t c2 = {};
    c2.gridDim = dim3(static_cast<unsigned>(p.rows) * p.nh, combine_slices<HD>());
    c2.blockDim = dim3(32 * combine_warps(p.splits));
    c2.dynamicSmemBytes = combine_smem_bytes(p.splits);
    c2.stream = stream;
    c2.attrs = attr;
    c2.numAttrs = 1;
    return cudaLaunchKernelEx(&c2, decode_combine_kernel<HD>, p);
}

template <int HD>
cudaError_t launch_decode(const LaunchArgs &a, bool set_attr)
{
    if (set_attr) {
        cudaError_t e = cudaFuncSetAttribute(decode_split_kernel<HD>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             Smem<HD>::kAllocCluster);
        if (e != cudaSuccess)
            return e;
    }
    const DecodeParams &p = a.p;
    dim3 grid(p.splits, p.nkv * p.hsg, p.rows);
    // Every launch may overlap the tail of the previous kernel in the stream
    // (programmatic dependent launch); the kernels wait for it before any
    // memory access.
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (p.cluster > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = p.cluster;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(Geo<HD>::kThreads);
    cfg.dynamicSmemBytes = p.cluster > 1 ? Smem<HD>::kAllocCluster : Smem<HD>::kAlloc;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    cudaError_t e = cudaLaunchKernelEx(&cfg, decode_split_kernel<HD>, *a.tm_k, *a.tm_v, p);
    if (e != cudaSuccess)
        return e;
    if (p.splits > 1 && p.counters == nullptr)
        e = launch_combine<HD>(p, a.stream);
    return e;
}

// How many clusters of `cluster` split CTAs can be resident at once (0: the
// on-chip merge cannot be used).  Also sets the kernel's attributes.
template <int HD>
int cluster_capacity(int cluster)
{
    if (cudaFuncSetAttribute(decode_split_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<HD>::kAllocCluster) != cudaSuccess)
        return 0;
    if (cluster > kMaxCluster)
        return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster, 1, 1);
    cfg.blockDim = dim3(Geo<HD>::kThreads);
    cfg.dynamicSmemBytes = Smem<HD>::kAllocCluster;
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

// Split CTAs (of the cluster-launch shape, the larger shared memory) that can
// be resident on one SM at once.  Also sets the kernel's attributes.
template <int HD>
int ctas_per_sm()
{
    if (cudaFuncSetAttribute(decode_split_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Smem<HD>::kAllocCluster) != cudaSuccess)
        return 0;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_split_kernel<HD>, Geo<HD>::kThreads,
                                                      Smem<HD>::kAllocCluster) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_combine_hd64(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_combine_hd128(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_combine_hd256(const DecodeParams &p, cudaStream_t stream);
cudaError_t launch_combine_hd512(const DecodeParams &p, cudaStream_t stream);
int cluster_capacity_hd64(int cluster);
int cluster_capacity_hd128(int cluster);
int cluster_capacity_hd256(int cluster);
int cluster_capacity_hd512(int cluster);
int ctas_per_sm_hd64();
int ctas_per_sm_hd128();
int ctas_per_sm_hd256();
int ctas_per_sm_hd512();

cudaError_t launch_decode_hd64(const LaunchArgs &a, bool set_attr);
cudaError_t launch_decode_hd128(const LaunchArgs &a, bool set_attr);
cudaError_t launch_decode_hd256(const LaunchArgs &a, bool set_attr);
cudaError_t launch_decode_hd512(const LaunchArgs &a, bool set_attr);

}  // namespace pgqa
