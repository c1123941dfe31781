// Device code of the split-KV paged GQA decode attention for sm_103a.
//
// What is computed is the decode attention of span-02
// `engine/crates/kernels/tests/gpu.rs` (`attn::attn_decode`, checked there
// against its f64 `reference`): query rows at positions qpos attend with GQA,
// scale 1.0, causally and (sliding layers) within `window`, over a bf16 pool
// [page][nkv][16][hd] reached through block_table[off[r] + p/16] and an
// optional page map.  Each of `splits` CTAs per (row, kv head) tile covers a
// page-aligned slice of the visible range and leaves a partial (running max,
// sum, unnormalised O); the last CTA of the tile (merge counters) or a
// separate combine kernel merges them.
//
// GB300 design:
//  * one producer warp streams whole (page, kv head) tiles of K and V into a
//    ring of shared-memory stages with TMA (cp.async.bulk.tensor, one 4-D box
//    per tile where the driver takes it) and the 128-byte swizzle, completion
//    counted on mbarriers;
//  * the consumer warps form Cfg<HD>::kGroups page groups of Cfg<HD>::kWpg
//    warps each (four groups of one warp at hd 64/128, four of two at hd 256,
//    two of four at hd 512).  Pages go round-robin to the groups, and a group
//    owns the ring stages s with s % kGroups == its index.  The warps of a
//    group split the head dimension: each computes S^T = K Q^T over its dims
//    on the tensor cores (mma.sync m16n8k16 bf16 -> f32, the page's 16 tokens
//    as MMA rows and up to 8 query rows -- all query heads of the kv head, or
//    packed rows -- as columns, so each KV byte leaves HBM once), the group
//    sums the partial scores through a small double-buffered shared array
//    (one named barrier per page), and every warp of the group runs the same
//    online softmax and O^T += V^T P^T for its dims, with P moved from the S
//    accumulators to the PV operand by movmatrix, never through shared
//    memory.  When every page is consumed the groups' (m, l, O) merge in
//    shared memory;
//  * online softmax in the log2 domain with quad shuffles; the O rescale is
//    skipped when no running max moved;
//  * the splits of a tile then merge in one of three ways, all with the same
//    arithmetic in the same order, so they agree bit for bit: inside a
//    thread-block cluster (2, 4 or 8 splits with merge counters), each CTA
//    pushing its (M, L) and a slice of its O into the slice owner's shared
//    memory with st.async; in the tile's last CTA, found through the merge
//    counters (other counts up to 8); or in the sliced combine kernel (no
//    counters, or more than 8 splits);
//  * every wait is bounded (about one second) and reports through a device
//    error word instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>

namespace pgqa {

constexpr int kPage = 16;                 // tokens per KV page
constexpr int kQRows = 8;                 // query rows (heads) per CTA: one MMA n-tile
constexpr int kBoxElems = 64;             // 128-byte swizzle atom: 64 bf16 per row
constexpr int kBoxBytes = kPage * kBoxElems * 2;   // one TMA box: 16 rows x 128 B
constexpr int kMaxSplits = 256;
constexpr int kMaxCluster = 8;            // largest thread-block cluster for the on-chip merge
constexpr int kGroupSplits = 8;           // the combine kernel merges more splits than this in two levels
constexpr int kMaxGroups = (kMaxSplits + kGroupSplits - 1) / kGroupSplits;
constexpr long long kWaitLimitCycles = 2000000000ll;   // bounded waits: ~1 s at 2 GHz
constexpr unsigned int kErrTimeoutFull = 1u;
constexpr unsigned int kErrTimeoutEmpty = 2u;
constexpr unsigned int kErrTimeoutCluster = 4u;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTraceEvents = 32;          // per-CTA slots of a trace build: 16 events x (ns, SM cycles)
constexpr int kAllConsumersBarrier = 15;  // named barrier of every consumer warp

// Per head dimension: the stage ring (about 128 KB of K/V in flight per SM
// keeps HBM streaming at full rate), and how the consumer warps share the
// pages.  Pages go round-robin to kGroups page groups; a group owns the ring
// stages s with s % kGroups == its index, so it waits for their mbarrier
// phases strictly in order.  The kWpg warps of a group split the head
// dimension and exchange partial scores once per page.
template <int HD>
struct Cfg;
template <>
struct Cfg<64> { static constexpr int kStages = 16, kGroups = 4, kWpg = 1, kMinBlocks = 3; };
template <>
struct Cfg<128> { static constexpr int kStages = 8, kGroups = 4, kWpg = 1, kMinBlocks = 3; };
template <>
struct Cfg<256> { static constexpr int kStages = 8, kGroups = 4, kWpg = 2, kMinBlocks = 1; };
template <>
struct Cfg<512> { static constexpr int kStages = 6, kGroups = 2, kWpg = 4, kMinBlocks = 1; };

template <int HD>
constexpr int kLgHd = HD == 64 ? 6 : HD == 128 ? 7 : HD == 256 ? 8 : 9;

template <int HD>
struct Geo {
    static constexpr int kStages = Cfg<HD>::kStages;
    static constexpr int kGroups = Cfg<HD>::kGroups;
    static constexpr int kWpg = Cfg<HD>::kWpg;
    static constexpr int kConsumerWarps = kGroups * kWpg;
    static constexpr int kConsumerThreads = kConsumerWarps * 32;
    static constexpr int kThreads = kConsumerThreads + 32;      // + one producer warp
    static constexpr int kDims = HD / kWpg;                     // head dims per consumer warp
    static constexpr int kBlocks = kDims / 16;                  // 16-dim MMA blocks per consumer warp
    static_assert(kStages % kGroups == 0, "each stage must belong to one page group");
    static_assert(kBlocks >= 1, "at least one 16-dim block per warp");
    static_assert((kQRows * HD / 4) % kConsumerThreads == 0, "merge: whole float4 outputs per thread");
};

template <int HD>
struct Smem {
    using G = Geo<HD>;
    static constexpr int kTile = kPage * HD * 2;                   // one (page, kv head) tile
    static constexpr int kStage = 2 * kTile;                       // K + V
    static constexpr int kStagesBytes = G::kStages * kStage;
    static constexpr int kXOff = kStagesBytes;                     // S exchange: float4 [groups][2][wpg][32]
    static constexpr int kXBytes = G::kGroups * 2 * G::kWpg * 32 * 16;
    static constexpr int kBarOff = kXOff + kXBytes;
    static constexpr int kBarBytes = (2 * G::kStages + 2) * 8;      // full, empty; cluster receive O, (M, L)
    static constexpr int kMiscOff = kBarOff + kBarBytes;
    static constexpr int kTotal = kMiscOff + 16;
    static constexpr int kAlloc = kTotal + 1024;                   // slack for 1024-B alignment
    // cluster launches only: the slices of the peers' partials that this CTA
    // merges, O [cluster][8][hd / cluster] f32 (32 hd bytes for any cluster
    // size), then (M, L) [cluster][8]
    static constexpr int kRecvOff = (kTotal + 15) / 16 * 16;
    static constexpr int kRecvMlOff = kRecvOff + kQRows * HD * 4;
    static constexpr int kRecvBytes = kQRows * HD * 4 + kMaxCluster * kQRows * 8;
    static constexpr int kAllocCluster = kRecvOff + kRecvBytes + 1024;
    // merge of the page groups' results, in the stage ring once every page is
    // consumed: O [groups][8][hd + 4] f32, (m, l) [groups][8], weights [8][groups + 2]
    static constexpr int kObufStride = HD + 4;
    static constexpr int kObufBytes = G::kGroups * kQRows * kObufStride * 4;
    static constexpr int kMlOff = kObufBytes;
    static constexpr int kStatOff = kMlOff + G::kGroups * kQRows * 8;
    static_assert(kStatOff + kQRows * (G::kGroups + 2) * 4 <= kStagesBytes, "group merge scratch");
    static_assert(kAllocCluster <= 227 * 1024, "shared memory");
};

struct DecodeParams {
    __nv_bfloat16 *o;        // [rows][nh][hd]
    float *part_o;           // [rows*nh][splits][hd]
    float2 *part_ml;         // [rows*nh][splits]: (max in log2 units, sum)
    const __nv_bfloat16 *q;  // [rows][nh][hd]
    const int32_t *block_table;
    const int32_t *off;
    const int32_t *qpos;
    const int32_t *kvpos;    // may be null
    const int32_t *page_map; // may be null
    uint32_t *counters;      // may be null: separate combine kernel
    unsigned int *err;       // device error word
    int rows, nh, nkv, window, splits, g;
    int hsg;                 // head subgroups of up to 8 heads per kv head
    int pack;                // rows per packing group (1 = no packing)
    int cluster;             // > 1: the splits of a tile are one cluster of this size, merged on chip
    int whole_tile_box;      // 1: one 4-D TMA box per (page, kv head) tile; 0: hd/64 3-D boxes
    unsigned long long *trace;   // per-CTA timestamps (trace builds only), or null
    // Speculative L2 prefetch before the dependency wait (0: none).  The
    // extents of the caller's allocations, from each pointer to its
    // allocation's end: block-table and page-map entries, and (page, kv head)
    // tiles of both pools.
    long long spec_tiles;
    long long spec_bt_len;
    long long spec_pm_len;
    const __nv_bfloat16 *k_pool;
    const __nv_bfloat16 *v_pool;
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity; gives up after about one second
// (kWaitLimitCycles of the SM clock), records `code` in the error word and
// returns false.  The bound uses the SM cycle counter, which is cheap to read
// between polls; the nanosecond global timer is not.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, unsigned int *err,
                                                  unsigned int code)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > kWaitLimitCycles) {
            atomicOr(err, code);
            return false;
        }
    }
    return true;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x,
                                            int y, int z)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z)
        : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y,
                                            int z, int w)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(x), "r"(y), "r"(z), "r"(w)
        : "memory");
}

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// Ticket: atomic add with release (this CTA's partials, ordered before by a
// CTA barrier, become visible with it) and acquire (the other CTAs'
// partials are visible to whoever observes the final count, and through a
// following CTA barrier to the rest of the CTA).
__device__ __forceinline__ unsigned int atomic_add_acq_rel(unsigned int *addr, unsigned int v)
{
    unsigned int old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], %2;" : "=r"(old) : "l"(addr), "r"(v) : "memory");
    return old;
}

// Thread-block cluster helpers (distributed shared memory).  Every thread
// of the cluster arrives once, right after the receive barrier is set up
// (the mbarrier-init fence orders that set-up), and waits before its first
// access to a peer.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// Address of this CTA's shared location `addr` in the shared memory of cluster CTA `rank`.
__device__ __forceinline__ uint32_t map_to_cta(uint32_t addr, int rank)
{
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(addr), "r"(rank));
    return out;
}

// Asynchronous store into a peer's shared memory; its bytes count down the
// transaction count of the peer's mbarrier `bar` (both cluster addresses).
__device__ __forceinline__ void st_async_f32x4(uint32_t addr, float4 v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                     addr),
                 "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void st_async_f32x2(uint32_t addr, float2 v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];" ::"r"(addr),
                 "f"(v.x), "f"(v.y), "r"(bar)
                 : "memory");
}

// Programmatic dependent launch: wait until the grids this one depends on
// have completed with their memory visible; then allow the next grid in the
// stream to start launching (it runs the same wait before touching memory).
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// 16-byte asynchronous global -> shared copy through L2 (generic proxy).
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(reinterpret_cast<uint64_t>(src))
                 : "memory");
}

__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Named barrier `id` over `threads` threads (a multiple of 32).
template <int id, int threads>
__device__ __forceinline__ void named_bar_sync()
{
    asm volatile("bar.sync %0, %1;" ::"n"(id), "n"(threads) : "memory");
}

__device__ __forceinline__ void group_bar_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                              uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

// D = A(16x16, row) * B(16x8, col) + D, bf16 inputs, f32 accumulate.
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose of an 8x8 b16 matrix held in the warp's fragment layout (lane t
// holds row t/4, columns 2(t%4) and 2(t%4)+1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x)
{
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ float bf16_round(float x)
{
    return __bfloat162float(__float2bfloat16_rn(x));
}

// Byte offset of 16-byte unit `u` (0..7) of row `row` inside one 128-byte
// swizzled TMA box: the unit index is XORed with the row index mod 8.
__device__ __forceinline__ uint32_t swz(int row, int u)
{
    return static_cast<uint32_t>(row * 128 + ((u ^ (row & 7)) << 4));
}

// ---------------------------------------------------------------- merge
//
// The S split partials (m_s, l_s, O_s) of one (row, head) merge as
//   M = max_s m_s,  w_s = (m_s == -inf) ? 0 : 2^(m_s - M),  L = sum_s w_s l_s,
//   o[d] = bf16_rn( (sum_s w_s O_s[d]) / L ), or 0 when L == 0.
// With more than kGroupSplits splits (combine kernel only) the merge runs in
// two levels: splits [8g, 8g+8) merge into an unnormalised group partial
// (M_g, L_g, O_g), and the group partials merge into o -- the same formula at
// both levels.  The last-CTA merge and the combine kernel run exactly these
// operations in exactly this order, so they agree bit for bit:
//  * merge_stats_warp (one warp): lane l takes splits l, l+32, ... in order,
//    then a fixed xor-butterfly combines the lanes; every lane ends with the
//    same bits because float max and addition are commutative;
//  * O: one fused multiply-add per split, splits in increasing order.

// Writes w[s] for s < S and returns L (in every lane).  1 <= S <= kMaxSplits.
// All loads are issued up front (clamped to valid splits, then masked).
// The statistics of merge_stats_warp from values already in registers: lane
// l holds splits l, l+32, ... in v[] ((-inf, 0) beyond S).
//
// With kLanes < 32 (S <= kLanes, kPer = 1) the butterflies start at
// kLanes / 2: the skipped steps would only combine lanes < S with lanes
// holding (-inf, 0) -- an exact max with -inf and an exact sum with +0 --
// so the result is the same bit for bit, with fewer shuffles.
template <int kPer, int kLanes = 32>
__device__ __forceinline__ float merge_stats_values(float2 (&v)[kPer], int S, float *w, int lane,
                                                    float *m_out = nullptr)
{
    static_assert(kLanes == 32 || kPer == 1, "narrow butterflies hold one value per lane");
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        if (lane + 32 * j >= S)
            v[j] = make_float2(-INFINITY, 0.f);
        mx = fmaxf(mx, v[j].x);
    }
#pragma unroll
    for (int k = kLanes / 2; k; k >>= 1)
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, k));
    if (m_out)
        *m_out = mx;
    float L = 0.f;
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int s = lane + 32 * j;
        if (s < S) {
            const float ws = (v[j].x == -INFINITY) ? 0.f : exp2f(v[j].x - mx);
            w[s] = ws;
            L = __fmaf_rn(ws, v[j].y, L);
        }
    }
#pragma unroll
    for (int k = kLanes / 2; k; k >>= 1)
        L = __fadd_rn(L, __shfl_xor_sync(0xffffffffu, L, k));
    return L;
}

// The statistics of merge_stats_values<1, kMaxCluster> for C <= kMaxCluster
// splits, computed by one thread: pair j at ml[j * stride], weights into w[],
// returns L.  The sum follows the butterfly as lane 0 sees it -- pairs 0 and
// 4, 2 and 6, 1 and 5, 3 and 7 first, then those sums over 2, then over 1 --
// with +0 for pairs past C, so the bits are those of the warp version (and of
// merge_stats_warp, whose wider butterfly only adds exact zeros first).
__device__ __forceinline__ float cluster_merge_weights(const float2 *ml, int stride, int C, float (&w)[kMaxCluster])
{
    static_assert(kMaxCluster == 8, "the butterfly below is written for 8 lanes");
    float2 v[kMaxCluster];
    float mx = -INFINITY;
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j) {
        v[j] = j < C ? ml[j * stride] : make_float2(-INFINITY, 0.f);
        mx = fmaxf(mx, v[j].x);
    }
    float l[kMaxCluster];
#pragma unroll
    for (int j = 0; j < kMaxCluster; ++j) {
        w[j] = (j >= C || v[j].x == -INFINITY) ? 0.f : exp2f(v[j].x - mx);
        l[j] = j < C ? __fmaf_rn(w[j], v[j].y, 0.f) : 0.f;
    }
    const float a0 = __fadd_rn(l[0], l[4]), a1 = __fadd_rn(l[1], l[5]);
    const float a2 = __fadd_rn(l[2], l[6]), a3 = __fadd_rn(l[3], l[7]);
    return __fadd_rn(__fadd_rn(a0, a2), __fadd_rn(a1, a3));
}

__device__ __forceinline__ float merge_stats_warp(const float2 *ml, int S, float *w, int lane,
                                                  float *m_out = nullptr)
{
    constexpr int kPer = kMaxSplits / 32;
    float2 v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j)
        v[j] = __ldcg(&ml[min(lane + 32 * j, S - 1)]);
    return merge_stats_values(v, S, w, lane, m_out);
}

__device__ __forceinline__ void fma4(float4 &acc, float w, const float4 &v)
{
    acc.x = __fmaf_rn(w, v.x, acc.x);
    acc.y = __fmaf_rn(w, v.y, acc.y);
    acc.z = __fmaf_rn(w, v.z, acc.z);
    acc.w = __fmaf_rn(w, v.w, acc.w);
}

__device__ __forceinline__ __nv_bfloat16 merge_finish(float acc, float L)
{
    return L > 0.f ? __float2bfloat16_rn(__fdiv_rn(acc, L)) : __float2bfloat16_rn(0.f);
}

// Four merged outputs -> o (8-byte store).
__device__ __forceinline__ void store_out4(__nv_bfloat16 *dst, const float4 &acc, float L)
{
    __nv_bfloat162 a, b;
    a.x = merge_finish(acc.x, L);
    a.y = merge_finish(acc.y, L);
    b.x = merge_finish(acc.z, L);
    b.y = merge_finish(acc.w, L);
    uint2 u;
    u.x = *reinterpret_cast<uint32_t *>(&a);
    u.y = *reinterpret_cast<uint32_t *>(&b);
    *reinterpret_cast<uint2 *>(dst) = u;
}

// Visible KV range [lo, hi] of row r (hi < lo: nothing visible).
__device__ __forceinline__ void row_window(const DecodeParams &p, int r, int &lo, int &hi)
{
    const int qp = __ldg(p.qpos + r);
    hi = p.kvpos ? min(qp, __ldg(p.kvpos + r)) : qp;    // causal: never past the query's own position
    lo = p.window > 0 ? max(0, qp + 1 - p.window) : 0;
}

// ---------------------------------------------------------------- speculative prefetch
//
// A split CTA may be resident well before the kernel ahead of it in the stream
// completes: when the combine kernel of the previous call runs, this call's
// CTAs take the SMs its split CTAs leave.  Until its dependency wait returns,
// such a CTA may read nothing that the previous kernel could still be writing
// and rely on it.  It may, though, guess: it reads off, qpos, kvpos, the block
// table and the page map as they stand and prefetches the first pages of its
// range into L2, which the wait leaves idle.  The guess is only a hint:
//  * every read goes through L2 alone (ld.global.cg), so no line it brings in
//    can be read stale from the L1 after the wait;
//  * every index is checked against the extent of the allocation it points
//    into (measured on the host), so a stale or never-written entry cannot
//    make an access outside the caller's memory;
//  * a wrong guess costs bandwidth, not correctness: the loads after the wait
//    read the inputs as they then are.
// Budget: up to 512 KB of K and V per CTA, at most 32 pages.
template <int HD>
__device__ __forceinline__ void speculative_prefetch(const DecodeParams &p, int lane, int kh)
{
    constexpr int kPages = 8192 / HD < 32 ? 8192 / HD : 32;
    const int rz = blockIdx.z;
    const int g0 = p.pack > 1 ? rz - rz % p.pack : rz;
    const int gn = p.pack > 1 ? min(p.pack, p.rows - g0) : 1;
    int off_i = 0, lo_i = 1, hi_i = 0;
    if (lane < gn) {
        off_i = __ldcg(p.off + g0 + lane);
        const int qp = __ldcg(p.qpos + g0 + lane);
        hi_i = p.kvpos ? min(qp, __ldcg(p.kvpos + g0 + lane)) : qp;
        lo_i = p.window > 0 ? max(0, qp + 1 - p.window) : 0;
    }
    // the packing verdict and the union range, as after the wait
    const int off0 = __shfl_sync(0xffffffffu, off_i, 0);
    const bool live = lane < gn && hi_i >= lo_i;
    const bool same = __all_sync(0xffffffffu, lane >= gn || off_i == off0);
    int max_lo = live ? lo_i : INT_MIN, min_hi = live ? hi_i : INT_MAX;
    int lo_u = live ? lo_i : INT_MAX, hi_u = live ? hi_i : INT_MIN;
#pragma unroll
    for (int k = 16; k; k >>= 1) {
        max_lo = max(max_lo, __shfl_xor_sync(0xffffffffu, max_lo, k));
        min_hi = min(min_hi, __shfl_xor_sync(0xffffffffu, min_hi, k));
        lo_u = min(lo_u, __shfl_xor_sync(0xffffffffu, lo_u, k));
        hi_u = max(hi_u, __shfl_xor_sync(0xffffffffu, hi_u, k));
    }
    const bool packed = gn > 1 && same &&
                        (max_lo == INT_MIN || static_cast<long long>(max_lo) <= static_cast<long long>(min_hi) + 1);
    int off_r = off0;
    if (packed) {
        if (rz != g0)
            return;                  // the group's first CTA prefetches for it
    } else {
        const int l = rz - g0;       // this CTA's own row
        off_r = __shfl_sync(0xffffffffu, off_i, l & 31);
        lo_u = __shfl_sync(0xffffffffu, lo_i, l & 31);
        hi_u = __shfl_sync(0xffffffffu, hi_i, l & 31);
    }
    if (hi_u < lo_u)
        return;
    const long long p0 = lo_u >> 4, np = (hi_u >> 4) - p0 + 1;
    const long long pb = p0 + (static_cast<long long>(blockIdx.x) * np) / p.splits;
    const long long pn = p0 + (static_cast<long long>(blockIdx.x + 1) * np) / p.splits - pb;
    if (lane >= pn || lane >= kPages)
        return;
    const long long idx = static_cast<long long>(off_r) + pb + lane;
    if (idx < 0 || idx >= p.spec_bt_len)
        return;
    long long ph = __ldcg(p.block_table + idx);
    if (p.page_map) {
        if (ph < 0 || ph >= p.spec_pm_len)
            return;
        ph = __ldcg(p.page_map + ph);
    }
    const long long tile = ph * p.nkv + kh;
    if (ph < 0 || tile >= p.spec_tiles)
        return;
    const size_t e = static_cast<size_t>(tile) * (kPage * HD);
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.k_pool + e), "r"(kPage * HD * 2) : "memory");
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.v_pool + e), "r"(kPage * HD * 2) : "memory");
}

// ---------------------------------------------------------------- tracing
//
// A library built with PGQA_TRACE records, per CTA, the global timer (ns) at a
// few phase boundaries into DecodeParams::trace; other builds compile the
// hooks away.
enum TraceEvent {
    kTrStart = 0,        // CTA starts its work (after any packing exit)
    kTrReady = 1,        // barriers initialised
    kTrFirstTma = 2,     // producer issued its first copy
    kTrFirstPage = 3,    // consumers hold the first page
    kTrLoopDone = 4,     // every page consumed
    kTrPartial = 5,      // output or partial written
    kTrTicket = 6,       // merge ticket taken
    kTrStats = 7,        // last CTA: merge weights ready
    kTrMerged = 8,       // last CTA: output written
    kTrFence = 9,        // last CTA: after the acquire fence
    kTrGroupO = 10,      // group results in shared memory
    kTrGroupStats = 11,  // group weights ready
    kTrPushed = 12,      // cluster merge: slices pushed to their owners
};

// Slots of a CTA's trace record: 0-15 the SM cycle counter at each event;
// 16 the global timer (ns) at kTrStart, 17 at the CTA's last event, 18 the
// cycles one global-timer read took, 19 whether whole-tile TMA boxes were used,
// 20 the SM the CTA ran on, 21 its page count.
__device__ __forceinline__ void trace_event(const DecodeParams &p, int ev, bool last = false)
{
#ifdef PGQA_TRACE
    if (p.trace) {
        const size_t cta = (static_cast<size_t>(blockIdx.z) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        unsigned long long *rec = p.trace + cta * kTraceEvents;
        const long long c0 = clock64();
        rec[ev] = static_cast<unsigned long long>(c0);
        if (ev == kTrStart || last) {
            unsigned long long t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            const long long c1 = clock64();
            rec[ev == kTrStart ? 16 : 17] = t;
            if (ev == kTrStart) {
                rec[18] = static_cast<unsigned long long>(c1 - c0);
                rec[19] = static_cast<unsigned long long>(p.whole_tile_box);
            }
        }
    }
#else
    (void)p;
    (void)ev;
    (void)last;
#endif
}

__device__ __forceinline__ void trace_placement(const DecodeParams &p, int npages)
{
#ifdef PGQA_TRACE
    if (p.trace) {
        const size_t cta = (static_cast<size_t>(blockIdx.z) * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;
        unsigned int sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        p.trace[cta * kTraceEvents + 20] = sm;
        p.trace[cta * kTraceEvents + 21] = static_cast<unsigned long long>(npages);
    }
#else
    (void)p;
    (void)npages;
#endif
}

// ---------------------------------------------------------------- merges of more than 8 splits
//
// The combine kernel runs one CTA per (row, head) and slice of up to 32 float4 of the head dimension
// (hd / 128 slices, at least one), one lane per float4.  Warp w merges split
// groups w, w + kCombineWarps, ...: a group's (m, l) and O loads are all in
// flight at once, so the merge costs about one L2 round trip per level
// instead of one per split.  Warp 0 then merges the groups.  The statistics
// routine and the per-element fused multiply-add order are the in-kernel
// merges', so up to kGroupSplits splits the two agree bit for bit.  Reads
// rows*nh*S*(hd+2)*4 bytes (the (m, l) pairs once per slice), writes
// rows*nh*hd*2.
constexpr int kCombineWarps = 8;

// float4 of the head dimension per CTA, and CTAs per (row, head)
template <int HD>
__host__ __device__ constexpr int combine_slice()
{
    return HD / 4 < 32 ? HD / 4 : 32;
}

template <int HD>
__host__ __device__ constexpr int combine_slices()
{
    return HD / 4 / combine_slice<HD>();
}

// Warps of a combine CTA and its dynamic shared memory (the group outputs of
// two-level merges), for S splits.
__host__ __device__ constexpr int combine_warps(int S)
{
    return S <= kGroupSplits ? 1 : ((S + kGroupSplits - 1) / kGroupSplits < kCombineWarps
                                         ? (S + kGroupSplits - 1) / kGroupSplits : kCombineWarps);
}
__host__ __device__ constexpr int combine_smem_bytes(int S)
{
    return S <= kGroupSplits ? 0 : (S + kGroupSplits - 1) / kGroupSplits * 32 * 16;
}

// The n <= kGroupSplits partial rows at src, src + HD/4, ... (zero beyond n
// or off this lane's slice), every load issued before any is used.
template <int HD>
__device__ __forceinline__ void combine_load_group(float4 (&v)[kGroupSplits], const float4 *src, int n, bool mine)
{
#pragma unroll
    for (int j = 0; j < kGroupSplits; ++j)
        v[j] = (mine && j < n) ? __ldcg(src + static_cast<size_t>(j) * (HD / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
}

// The merge of the S > kGroupSplits partials of one (row, head) over float4
// slice c of its head dimension (lanes past the slice idle), by warps
// warp0 .. warp0 + nw - 1 of the calling CTA: warp w merges split groups
// w, w + nw, ... (up to kGroupSplits splits each) into og, then the first of
// them merges the groups and writes o.  `sync` is a barrier over those warps.
// The combine kernel runs this for every (row, head) and slice.
template <int HD, typename Sync>
__device__ __forceinline__ void merge_two_level(const DecodeParams &p, size_t rh, int c, int w, int nw, int lane,
                                                float (*gw)[kGroupSplits], float2 *gml, float *wts, float4 *og,
                                                Sync sync)
{
    const int S = p.splits;
    const int d4 = c * combine_slice<HD>() + lane;
    const bool mine = lane < combine_slice<HD>();
    const float4 *po = reinterpret_cast<const float4 *>(p.part_o + rh * S * HD) + d4;
    const float2 *pml = p.part_ml + rh * S;
    const int ng = (S + kGroupSplits - 1) / kGroupSplits;
    float4 v[kGroupSplits];
    for (int g = w; g < ng; g += nw) {
        const int n = min(kGroupSplits, S - g * kGroupSplits);
        combine_load_group<HD>(v, po + static_cast<size_t>(g) * kGroupSplits * (HD / 4), n, mine);
        float m = 0.f;
        const float L = merge_stats_warp(pml + g * kGroupSplits, n, gw[g], lane, &m);
        if (lane == 0)
            gml[g] = make_float2(m, L);
        __syncwarp();
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kGroupSplits; ++j)
            if (j < n)
                fma4(a, gw[g][j], v[j]);
        og[g * 32 + lane] = a;
    }
    sync();
    if (w != 0)
        return;
    constexpr int kPer = (kMaxGroups + 31) / 32;
    float2 sv[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j)
        sv[j] = gml[min(lane + 32 * j, ng - 1)];
    const float L = merge_stats_values(sv, ng, wts, lane);
    __syncwarp();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int g = 0; g < ng; ++g)
        fma4(acc, wts[g], og[g * 32 + lane]);
    if (mine)
        store_out4(p.o + rh * HD + d4 * 4, acc, L);
}

// ---------------------------------------------------------------- main kernel
//
// Grid (splits, nkv * hsg, rows); block = the consumer warps of Cfg<HD> + one
// producer warp.  A CTA serves up to 8 query rows of the MMA: the heads of one
// kv head (a subgroup of 8 when nh/nkv > 8) of one row, or, when `pack` > 1
// and a group of `pack` consecutive rows shares its block-table span (equal
// off) and has pairwise-overlapping windows, of all rows of the group: the
// group's first CTA then serves them all and the others exit at once, so KV
// shared by the rows leaves HBM and enters shared memory once.
// HBM-bound: per (page, kv head) it moves 2 * 16 * hd * 2 bytes and runs
// 3 * hd / 16 MMAs, below the legacy tensor pipe's rate.
template <int HD>
__global__ void __launch_bounds__(Geo<HD>::kThreads, Cfg<HD>::kMinBlocks)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const DecodeParams p)
{
    using SM = Smem<HD>;
    using GE = Geo<HD>;
    constexpr int NS = GE::kStages;
    constexpr int NG = GE::kGroups;
    constexpr int WPG = GE::kWpg;
    constexpr int NW = GE::kConsumerWarps;
    constexpr int NT = GE::kConsumerThreads;
    constexpr int KB = GE::kBlocks;           // 16-dim blocks per consumer warp
    constexpr int kChunks = HD / kBoxElems;   // TMA boxes per tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_full = s_base + SM::kBarOff;
    const uint32_t s_empty = s_full + NS * 8;
    int *s_misc = reinterpret_cast<int *>(smem + SM::kMiscOff);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int split = blockIdx.x;
    const int kh = blockIdx.y / p.hsg;
    const int hs = blockIdx.y - kh * p.hsg;
    const int rz = blockIdx.z;
    const int head0 = kh * p.g + hs * kQRows;
    const int nh_sub = min(kQRows, p.g - hs * kQRows);
    const int S = p.splits;

    const uint32_t s_recv = s_full + 2 * NS * 8;    // cluster launches: peers' O slices arrived
    const uint32_t s_recv_ml = s_recv + 8;          // cluster launches: peers' (M, L) arrived
    // Barriers first: the init fence then has no earlier load to wait for.
    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(s_full + 8 * s, 1);
            mbar_init(s_empty + 8 * s, WPG);
        }
        if (p.cluster > 1) {
            // complete once every peer (this CTA included) has pushed its O
            // slice, and its (M, L), of all 8 query rows
            mbar_init(s_recv, 1);
            mbar_arrive_expect_tx(s_recv, kQRows * HD * 4);
            mbar_init(s_recv_ml, 1);
            mbar_arrive_expect_tx(s_recv_ml, p.cluster * kQRows * 8);
        }
        mbar_init_fence();
    }
    if (p.cluster > 1)
        cluster_arrive_relaxed();
    // The tensor maps are kernel parameters, which no earlier kernel writes:
    // fetching them now hides the descriptor latency of the first copies.
    if (warp == NW && lane == 0) {
        tma_prefetch_map(&tm_k);
        tma_prefetch_map(&tm_v);
    }
    if (p.spec_tiles > 0 && warp == NW)
        speculative_prefetch<HD>(p, lane, kh);
    // Nothing above relies on a value read from global memory: wait here for
    // the previous kernel in the stream (inputs may be its outputs), then let
    // the next one launch.
    grid_dependency_wait();
    grid_launch_dependents();

    // ---- rows served: this CTA's own, or a packing group led by its first row.
    // One round of metadata loads: lane i of every warp loads row g0 + i of
    // the packing group (just row rz without packing).  Everything else --
    // the packing verdict, the union range, off of the first served row and
    // each query row's window -- comes from shuffles, identical in every warp,
    // so the CTA decides uniformly.
    const int g0 = p.pack > 1 ? rz - rz % p.pack : rz;
    const int gn = p.pack > 1 ? min(p.pack, p.rows - g0) : 1;
    int off_i = 0, lo_i = 1, hi_i = 0;
    if (lane < gn) {
        off_i = __ldg(p.off + g0 + lane);
        row_window(p, g0 + lane, lo_i, hi_i);
    }
    int r0 = rz, nr = 1;
    if (gn > 1) {
        const bool live = lane < gn && hi_i >= lo_i;
        const int off0 = __shfl_sync(0xffffffffu, off_i, 0);
        const bool same = __all_sync(0xffffffffu, lane >= gn || off_i == off0);
        int max_lo = live ? lo_i : INT_MIN, min_hi = live ? hi_i : INT_MAX;
#pragma unroll
        for (int k = 16; k; k >>= 1) {
            max_lo = max(max_lo, __shfl_xor_sync(0xffffffffu, max_lo, k));
            min_hi = min(min_hi, __shfl_xor_sync(0xffffffffu, min_hi, k));
        }
        const bool overlap = max_lo == INT_MIN ||
                             static_cast<long long>(max_lo) <= static_cast<long long>(min_hi) + 1;
        if (same && overlap) {
            if (rz != g0) {           // served by the group's first CTA
                if (p.cluster > 1)
                    cluster_wait();
                return;
            }
            r0 = g0;
            nr = gn;
        }
    }
    const int nq = nr * nh_sub;        // query rows in use (<= 8)
    const int lb = r0 - g0;            // metadata lane of the first served row
    const int off_r0 = __shfl_sync(0xffffffffu, off_i, lb);
    if (tid == 0)
        trace_event(p, kTrStart);

    // ---- union of the served rows' visible ranges; this split's page share
    int lo_u = 0, hi_u = -1;
    {
        const bool served = lane >= lb && lane < lb + nr && hi_i >= lo_i;
        int lo_m = served ? lo_i : INT_MAX, hi_m = served ? hi_i : INT_MIN;
#pragma unroll
        for (int k = 16; k; k >>= 1) {
            lo_m = min(lo_m, __shfl_xor_sync(0xffffffffu, lo_m, k));
            hi_m = max(hi_m, __shfl_xor_sync(0xffffffffu, hi_m, k));
        }
        if (hi_m != INT_MIN) {
            lo_u = lo_m;
            hi_u = hi_m;
        }
    }
    int page_begin = 0, npages_mine = 0;
    if (hi_u >= lo_u) {
        const int p0 = lo_u >> 4;
        const int np = (hi_u >> 4) - p0 + 1;
        if (np <= (1 << 22)) {       // (S + 1) * np < 2^31: 32-bit arithmetic
            page_begin = p0 + (split * np) / S;
            npages_mine = p0 + ((split + 1) * np) / S - page_begin;
        } else {
            page_begin = p0 + static_cast<int>((static_cast<long long>(split) * np) / S);
            npages_mine = p0 + static_cast<int>((static_cast<long long>(split + 1) * np) / S) - page_begin;
        }
    }

    if (tid == 0)
        trace_placement(p, npages_mine);

    // ---- loads that need no barrier go out before the barrier set-up
    const int32_t *tbl = nullptr;
    int phys_first = 0;              // producer: physical page of lane's first-chunk page
    const int gid = lane >> 2;       // MMA group: query row of S, d row of O^T
    const int tig = lane & 3;        // thread in group
    const int grp = warp / WPG;      // consumer: page group
    const int wig = warp - grp * WPG;    // consumer: warp within the group
    const int dq0 = wig * GE::kDims; // consumer: first head dim of this warp
    uint32_t qa[KB][2];
    int lo_a = 1, hi_a = 0;          // visible ranges of query rows 2tig and 2tig+1 (empty if unused)
    int lo_b = 1, hi_b = 0;
    // windows of query rows 2tig and 2tig+1 (each thread's O^T columns)
    {
        const int la = lb + (2 * tig) / nh_sub, lbb = lb + (2 * tig + 1) / nh_sub;
        const int wla = __shfl_sync(0xffffffffu, lo_i, la & 31), wha = __shfl_sync(0xffffffffu, hi_i, la & 31);
        const int wlb = __shfl_sync(0xffffffffu, lo_i, lbb & 31), whb = __shfl_sync(0xffffffffu, hi_i, lbb & 31);
        if (2 * tig < nq) {
            lo_a = wla;
            hi_a = wha;
        }
        if (2 * tig + 1 < nq) {
            lo_b = wlb;
            hi_b = whb;
        }
    }
    if (warp == NW) {
        tbl = p.block_table + off_r0 + page_begin;
        if (lane < npages_mine) {
            phys_first = __ldg(tbl + lane);
            if (p.page_map)
                phys_first = __ldg(p.page_map + phys_first);
        }
    } else {
        // Query row r of the MMA is (row r0 + r / nh_sub, head head0 + r % nh_sub);
        // rows >= nq are zero.  A-fragments of this warp's dims come straight
        // from global memory into registers.
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
            qa[kb][0] = qa[kb][1] = 0u;
        if (gid < nq) {
            const size_t rh = static_cast<size_t>(r0 + gid / nh_sub) * p.nh + head0 + gid % nh_sub;
            const uint32_t *qg = reinterpret_cast<const uint32_t *>(p.q + rh * HD + dq0);
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                qa[kb][0] = __ldg(qg + kb * 8 + tig);          // dims 16kb + 2tig, +1
                qa[kb][1] = __ldg(qg + kb * 8 + 4 + tig);      // dims 16kb + 8 + 2tig, +1
            }
        }
    }

    __syncthreads();
    if (tid == 0)
        trace_event(p, kTrReady);
    if (p.cluster > 1 && warp < NW)
        cluster_wait();              // consumers: every peer's receive barrier is set up

    if (warp == NW) {
        // ------------------------------------------------ producer warp
        bool ok = true;
        for (int c0 = 0; c0 < npages_mine && ok; c0 += 32) {
            int phys = phys_first;
            if (c0 > 0) {
                phys = 0;
                if (c0 + lane < npages_mine) {
                    phys = __ldg(tbl + c0 + lane);
                    if (p.page_map)
                        phys = __ldg(p.page_map + phys);
                }
            }
            const int n = min(32, npages_mine - c0);
            for (int j = 0; j < n; ++j) {
                const int ph = __shfl_sync(0xffffffffu, phys, j);
                if (lane == 0 && ok) {
                    const int i = c0 + j;
                    const int st = i % NS;
                    if (i >= NS)
                        ok = mbar_wait_bounded(s_empty + 8 * st, ((i / NS) - 1) & 1, p.err, kErrTimeoutEmpty);
                    if (ok) {
                        const uint32_t bar = s_full + 8 * st;
                        const uint32_t dk = s_base + st * SM::kStage;
                        const uint32_t dv = dk + SM::kTile;
                        const int tile = ph * p.nkv + kh;
                        mbar_arrive_expect_tx(bar, SM::kStage);
                        if (p.whole_tile_box) {
                            tma_load_4d(dk, &tm_k, bar, 0, 0, 0, tile);
                            tma_load_4d(dv, &tm_v, bar, 0, 0, 0, tile);
                        } else {
#pragma unroll
                            for (int c = 0; c < kChunks; ++c) {
                                tma_load_3d(dk + c * kBoxBytes, &tm_k, bar, c * kBoxElems, 0, tile);
                                tma_load_3d(dv + c * kBoxBytes, &tm_v, bar, c * kBoxElems, 0, tile);
                            }
                        }
                        if (i == 0)
                            trace_event(p, kTrFirstTma);
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        __syncwarp();
        if (p.cluster > 1)           // each thread that arrived also waits
            cluster_wait();
        return;
    }

    // ---------------------------------------------------- consumer warps
    // Scores are computed transposed, S^T = K Q^T: the page's 16 tokens are the
    // MMA rows and the 8 query rows its columns, so no MMA row is padding.
    // Lane (gid, tig) holds S^T for tokens gid and gid+8 of query rows 2tig and
    // 2tig+1 -- the same query rows as its O^T columns, so the softmax state
    // of those two rows lives in the lane that rescales them.
    float acc[KB][4];              // O^T: dims dq0 + 16mt + {gid, gid+8}, query rows {2tig, 2tig+1}
#pragma unroll
    for (int mt = 0; mt < KB; ++mt)
        acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY;   // running max of query rows 2tig, 2tig+1 (log2 units)
    float l_a = 0.f, l_b = 0.f;               // this lane's share of their running sums

    // per-lane ldmatrix row/unit selectors
    const int lm_i = lane >> 3, lm_r = lane & 7;
    const int k_tok = (lm_i & 1) * 8 + lm_r;       // K as A operand: matrices (tok lo/hi) x (dims lo/hi)
    const int k_half = lm_i >> 1;
    const int v_tok = (lm_i >> 1) * 8 + lm_r;      // V^T as A operand via .trans: (tok lo/hi) x (dims lo/hi)
    const int v_half = lm_i & 1;
    float4 *sx = reinterpret_cast<float4 *>(smem + SM::kXOff) + grp * (2 * WPG * 32);

    bool ok = true;
    int jj = 0;                    // this group's page count
    for (int i = grp; i < npages_mine; i += NG, ++jj) {
        const int st = i % NS;
        if (ok)
            ok = mbar_wait_bounded(s_full + 8 * st, (i / NS) & 1, p.err, kErrTimeoutFull);
        if (i == 0 && wig == 0 && lane == 0)
            trace_event(p, kTrFirstPage);
        const uint32_t sk = s_base + st * SM::kStage;
        const uint32_t sv = sk + SM::kTile;
        const int pos0 = (page_begin + i) * kPage;

        // (partial) S^T over this warp's dims, even and odd 16-dim blocks in
        // separate accumulators
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if (ok) {
#pragma unroll
            for (int kb = 0; kb < KB; ++kb) {
                const int k16 = dq0 / 16 + kb;
                uint32_t a0, a1, a2, a3;
                ldsm_x4(sk + (k16 >> 2) * kBoxBytes + swz(k_tok, (k16 & 3) * 2 + k_half), a0, a1, a2, a3);
                mma_bf16_16816(sc[kb & 1], a0, a1, a2, a3, qa[kb][0], qa[kb][1]);
            }
        }
        float4 sfull = make_float4(sc[0][0] + sc[1][0], sc[0][1] + sc[1][1], sc[0][2] + sc[1][2],
                                   sc[0][3] + sc[1][3]);
        if (WPG > 1) {
            // full S^T = sum of the group's partials, in warp order
            float4 *xb = sx + (jj & 1) * (WPG * 32);
            xb[wig * 32 + lane] = sfull;
            group_bar_sync(1 + grp, WPG * 32);
            sfull = xb[lane];
#pragma unroll
            for (int w = 1; w < WPG; ++w) {
                const float4 v = xb[w * 32 + lane];
                sfull.x += v.x;
                sfull.y += v.y;
                sfull.z += v.z;
                sfull.w += v.w;
            }
        }

        // mask to each query row's [lo, hi], scale to log2 units:
        // x0/x1 token gid, x2/x3 token gid+8; x0/x2 query row 2tig, x1/x3 row 2tig+1
        const int ta = pos0 + gid, tb = ta + 8;
        float x[4];
        x[0] = (ta >= lo_a && ta <= hi_a) ? sfull.x * kLog2e : -INFINITY;
        x[1] = (ta >= lo_b && ta <= hi_b) ? sfull.y * kLog2e : -INFINITY;
        x[2] = (tb >= lo_a && tb <= hi_a) ? sfull.z * kLog2e : -INFINITY;
        x[3] = (tb >= lo_b && tb <= hi_b) ? sfull.w * kLog2e : -INFINITY;

        // online softmax: the 8 lanes of a tig column hold a query row's 16 scores
        float mxa = fmaxf(x[0], x[2]), mxb = fmaxf(x[1], x[3]);
#pragma unroll
        for (int k = 4; k < 32; k <<= 1) {
            mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, k));
            mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, k));
        }
        const float mna = fmaxf(m_a, mxa), mnb = fmaxf(m_b, mxb);
        float al_a = 1.f, al_b = 1.f;
        float pr[4] = {0.f, 0.f, 0.f, 0.f};
        if (mna != -INFINITY) {
            al_a = exp2f(m_a - mna);
            pr[0] = bf16_round(exp2f(x[0] - mna));
            pr[2] = bf16_round(exp2f(x[2] - mna));
        }
        if (mnb != -INFINITY) {
            al_b = exp2f(m_b - mnb);
            pr[1] = bf16_round(exp2f(x[1] - mnb));
            pr[3] = bf16_round(exp2f(x[3] - mnb));
        }
        m_a = mna;
        m_b = mnb;
        l_a = __fmaf_rn(l_a, al_a, pr[0] + pr[2]);
        l_b = __fmaf_rn(l_b, al_b, pr[1] + pr[3]);
        // P^T as the PV B fragment: transpose the (token x query) 8x8 tiles
        const uint32_t pb0 = movmatrix_trans(pack_bf16x2(pr[0], pr[1]));   // tokens 0-7
        const uint32_t pb1 = movmatrix_trans(pack_bf16x2(pr[2], pr[3]));   // tokens 8-15

        if (__any_sync(0xffffffffu, al_a != 1.f || al_b != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < KB; ++mt) {
                acc[mt][0] *= al_a;
                acc[mt][1] *= al_b;
                acc[mt][2] *= al_a;
                acc[mt][3] *= al_b;
            }
        }

        // positions of this page outside every served row's range may hold any
        // bits: zero this warp's dims of their V rows, so 0 * NaN cannot reach
        // the accumulators
        const bool edge = pos0 < lo_u || pos0 + kPage - 1 > hi_u;
        if (edge && ok) {
            constexpr int kUnits = GE::kDims / 8;     // 16-byte units of one token row this warp owns
            for (int e = lane; e < kPage * kUnits; e += 32) {
                const int t = e / kUnits;
                if (pos0 + t < lo_u || pos0 + t > hi_u) {
                    const int col = dq0 / 8 + (e - t * kUnits);   // 16-byte unit of the row
                    *reinterpret_cast<uint4 *>(smem + (sv - s_base) + (col >> 3) * kBoxBytes + swz(t, col & 7)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
            }
            __syncwarp();
        }

        // O^T += V^T P^T over this warp's dims
        if (ok) {
#pragma unroll
            for (int mt = 0; mt < KB; ++mt) {
                const int m16 = dq0 / 16 + mt;
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(sv + (m16 >> 2) * kBoxBytes + swz(v_tok, (m16 & 3) * 2 + v_half), a0, a1, a2, a3);
                mma_bf16_16816(acc[mt], a0, a1, a2, a3, pb0, pb1);
            }
        }

        if (edge)
            fence_proxy_async_smem();      // generic writes above vs the next TMA into this stage
        __syncwarp();
        if (lane == 0)
            mbar_arrive(s_empty + 8 * st);
    }
#pragma unroll
    for (int k = 4; k < 32; k <<= 1) {
        l_a += __shfl_xor_sync(0xffffffffu, l_a, k);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, k);
    }
    named_bar_sync<kAllConsumersBarrier, NT>();      // every page consumed: the stage ring is free
    if (tid == 0)
        trace_event(p, kTrLoopDone);

    // ---------------------------------------------------- merge of the page groups
    float *obuf = reinterpret_cast<float *>(smem);
    float2 *mlbuf = reinterpret_cast<float2 *>(smem + SM::kMlOff);
    float *stat = reinterpret_cast<float *>(smem + SM::kStatOff);
    {
        float *ob = obuf + grp * kQRows * SM::kObufStride;
#pragma unroll
        for (int mt = 0; mt < KB; ++mt) {
            const int d = dq0 + mt * 16 + gid;
            ob[(2 * tig) * SM::kObufStride + d] = acc[mt][0];
            ob[(2 * tig + 1) * SM::kObufStride + d] = acc[mt][1];
            ob[(2 * tig) * SM::kObufStride + d + 8] = acc[mt][2];
            ob[(2 * tig + 1) * SM::kObufStride + d + 8] = acc[mt][3];
        }
        if (wig == 0 && gid == 0) {
            mlbuf[grp * kQRows + 2 * tig] = make_float2(m_a, l_a);
            mlbuf[grp * kQRows + 2 * tig + 1] = make_float2(m_b, l_b);
        }
    }
    named_bar_sync<kAllConsumersBarrier, NT>();
    if (tid == 0)
        trace_event(p, kTrGroupO);
    // weights of the page groups for query row q, w_g = 2^(m_g - max_g m_g)
    // (0 for a group that saw nothing); every thread that needs them computes
    // them the same way, so all copies agree bit for bit
    auto group_weights = [&](int q, float (&w)[NG]) {
        float mx = -INFINITY;
#pragma unroll
        for (int g = 0; g < NG; ++g)
            mx = fmaxf(mx, mlbuf[g * kQRows + q].x);
#pragma unroll
        for (int g = 0; g < NG; ++g) {
            const float m = mlbuf[g * kQRows + q].x;
            w[g] = (m == -INFINITY) ? 0.f : exp2f(m - mx);
        }
        return mx;
    };
    // this split's (M, L) of query row q (an empty partial past the served rows)
    auto split_stats = [&](int q) {
        float mx = -INFINITY, L = 0.f;
        if (q < nq) {
            float w[NG];
            mx = group_weights(q, w);
#pragma unroll
            for (int g = 0; g < NG; ++g)
                L = __fmaf_rn(w[g], mlbuf[g * kQRows + q].y, L);
        }
        return make_float2(mx, L);
    };

    if (p.cluster > 1) {
        // ------------------------------------------------ on-chip merge of the cluster
        // The S = cluster splits of this tile are the CTAs of one cluster.
        // CTA r merges dims [r*hd/S, (r+1)*hd/S) of every query row: each CTA
        // pushes that slice of its partial O, and its (M, L), into CTA r's
        // receive buffer with asynchronous stores that complete on CTA r's
        // receive barrier.  The merge then runs on local shared memory, with
        // the same operations in the same order as the combine kernel, and
        // no CTA reads a peer, so none waits for its peers before exiting.
        // Every thread derives the weights it needs itself: no barrier
        // between the group merge, the pushes and the final merge.
        const int C = p.cluster;                         // 2, 4 or 8
        const int lg_slice = kLgHd<HD> - (31 - __clz(C));
        const int slice = 1 << lg_slice;                 // hd / C
        float *recv_o = reinterpret_cast<float *>(smem + SM::kRecvOff);
        float2 *recv_ml = reinterpret_cast<float2 *>(smem + SM::kRecvMlOff);
        if (tid < kQRows) {
            // this split's (M, L) to every slice owner, ahead of the O slices,
            // so the owners' merge weights overlap the O transfer
            const float2 ml = split_stats(tid);
            const uint32_t a = smem_u32(recv_ml + split * kQRows + tid);
            for (int j = 0; j < C; ++j)
                st_async_f32x2(map_to_cta(a, j), ml, map_to_cta(s_recv_ml, j));
        }
        constexpr int kVec = HD / 4;
#pragma unroll
        for (int k = 0; k < kQRows * kVec / NT; ++k) {
            const int e = tid + k * NT;
            const int q = e / kVec, d = (e - q * kVec) * 4;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            if (q < nq) {
                float w[NG];
                group_weights(q, w);
                const float *ob = obuf + q * SM::kObufStride + d;
#pragma unroll
                for (int g = 0; g < NG; ++g) {
                    const float4 v = *reinterpret_cast<const float4 *>(ob + g * kQRows * SM::kObufStride);
                    o.x = __fmaf_rn(w[g], v.x, o.x);
                    o.y = __fmaf_rn(w[g], v.y, o.y);
                    o.z = __fmaf_rn(w[g], v.z, o.z);
                    o.w = __fmaf_rn(w[g], v.w, o.w);
                }
            }
            const int j = d >> lg_slice;
            st_async_f32x4(map_to_cta(smem_u32(recv_o + ((split * kQRows + q) << lg_slice) + (d & (slice - 1))), j),
                           o, map_to_cta(s_recv, j));
        }
        if (tid == 0)
            trace_event(p, kTrPushed);
        if (!mbar_wait_bounded(s_recv_ml, 0, p.err, kErrTimeoutCluster))
            return;
        if (tid == 0)
            trace_event(p, kTrTicket);
        const int d0 = split * slice;
        bool have = false;
        for (int e = tid; e < (nq << lg_slice); e += NT) {
            const int q = e >> lg_slice, dd = e & (slice - 1);
            float w[kMaxCluster];
            const float L = cluster_merge_weights(recv_ml + q, kQRows, C, w);
            if (!have) {
                if (tid == 0)
                    trace_event(p, kTrStats);
                if (!mbar_wait_bounded(s_recv, 0, p.err, kErrTimeoutCluster))
                    return;
                have = true;
            }
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < kMaxCluster; ++j)
                if (j < C)
                    acc = __fmaf_rn(w[j], recv_o[((j * kQRows + q) << lg_slice) + dd], acc);
            const size_t rh = static_cast<size_t>(r0 + q / nh_sub) * p.nh + head0 + q % nh_sub;
            p.o[rh * HD + d0 + dd] = merge_finish(acc, L);
        }
        if (tid == 0)
            trace_event(p, kTrMerged, true);
        return;
    }

    if (tid < kQRows) {
        const float2 ml = split_stats(tid);
        float w[NG];
        if (tid < nq)
            group_weights(tid, w);
#pragma unroll
        for (int g = 0; g < NG; ++g)
            stat[tid * (NG + 2) + g] = tid < nq ? w[g] : 0.f;
        stat[tid * (NG + 2) + NG] = ml.y;
        stat[tid * (NG + 2) + NG + 1] = ml.x;
        if (S > 1 && tid < nq) {
            const size_t rh = static_cast<size_t>(r0 + tid / nh_sub) * p.nh + head0 + tid % nh_sub;
            p.part_ml[rh * S + split] = ml;
        }
    }
    named_bar_sync<kAllConsumersBarrier, NT>();
    if (tid == 0)
        trace_event(p, kTrGroupStats);
    // this split's O (or, with one split, the output): four consecutive dims
    // per thread and step, so loads and stores go out 16 (8) bytes wide
    {
        constexpr int kVec4 = HD / 4;
#pragma unroll
        for (int k = 0; k < kQRows * kVec4 / NT; ++k) {
            const int e = tid + k * NT;
            const int q = e / kVec4, d = (e - q * kVec4) * 4;
            if (q < nq) {
                const float *st = stat + q * (NG + 2);
                const size_t rh = static_cast<size_t>(r0 + q / nh_sub) * p.nh + head0 + q % nh_sub;
                float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int g = 0; g < NG; ++g)
                    fma4(o, st[g], *reinterpret_cast<const float4 *>(obuf + (g * kQRows + q) * SM::kObufStride + d));
                if (S == 1)
                    store_out4(p.o + rh * HD + d, o, st[NG]);
                else
                    *reinterpret_cast<float4 *>(p.part_o + (rh * S + split) * HD + d) = o;
            }
        }
    }
    if (tid == 0)
        trace_event(p, kTrPartial, S == 1 || p.counters == nullptr);
    if (S == 1 || p.counters == nullptr)
        return;

    // ---------------------------------------------------- last-CTA merge
    // Only with counters, which the host passes for S <= kGroupSplits alone
    // (more splits merge in the combine kernel).  The S partial rows of every
    // served query row come into the (now free) stage ring by cp.async while
    // the weights are computed; each thread then accumulates its kOwn float4
    // outputs (query row q, dims 4*d4..+3) in split order.
    constexpr int kVec = HD / 4;                               // float4 per query row
    constexpr int kOwn = kQRows * kVec / NT;                   // float4 outputs per thread
    constexpr int kWStride = kGroupSplits + 1;                 // weights and L of one query row
    constexpr int kStageOff = (kQRows * kWStride * 4 + 15) / 16 * 16;
    static_assert(kStageOff + kGroupSplits * kQRows * HD * 4 <= SM::kStagesBytes, "merge staging");
    float *wts = reinterpret_cast<float *>(smem);
    float *stg = reinterpret_cast<float *>(smem + kStageOff);
    auto rowhead = [&](int q) {
        return static_cast<size_t>(r0 + q / nh_sub) * p.nh + head0 + q % nh_sub;
    };

    // Tickets: the barrier orders every thread's stores before thread 0's
    // acquire-release atomic; the winner's threads see all partials after the
    // second barrier.
    const int tile_id = (r0 * p.nkv + kh) * p.hsg + hs;
    unsigned int *cnt = p.counters + tile_id;
    named_bar_sync<kAllConsumersBarrier, NT>();
    if (tid == 0)
        s_misc[0] = static_cast<int>(atomic_add_acq_rel(cnt, 1u));
    named_bar_sync<kAllConsumersBarrier, NT>();
    const int t = s_misc[0];
    if (tid == 0)
        trace_event(p, kTrTicket, t != S - 1);
    if (t != S - 1)
        return;

    // rows s of every query row -> stg[(s * nq + q) * HD]
    for (int e = tid; e < S * nq * kVec; e += NT) {
        const int sq = e / kVec, d4 = e - sq * kVec;
        const int sp = sq / nq, q = sq - sp * nq;
        cp_async16(smem_u32(stg + static_cast<size_t>(sq) * HD + d4 * 4),
                   p.part_o + (rowhead(q) * S + sp) * HD + d4 * 4);
    }
    for (int q = warp; q < nq; q += NW) {
        const float L = merge_stats_warp(p.part_ml + rowhead(q) * S, S, wts + q * kWStride, lane);
        if (lane == 0)
            wts[q * kWStride + kGroupSplits] = L;
    }
    cp_async_wait_all();
    named_bar_sync<kAllConsumersBarrier, NT>();  // staged rows and weights visible to every thread
    float4 oacc[kOwn];
#pragma unroll
    for (int k = 0; k < kOwn; ++k)
        oacc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < S; ++sp) {
#pragma unroll
        for (int k = 0; k < kOwn; ++k) {
            const int e = tid + k * NT;
            const int q = e / kVec, d4 = e - q * kVec;
            if (q < nq)
                fma4(oacc[k], wts[q * kWStride + sp],
                     *reinterpret_cast<const float4 *>(stg + static_cast<size_t>(sp * nq + q) * HD + d4 * 4));
        }
    }
#pragma unroll
    for (int k = 0; k < kOwn; ++k) {
        const int e = tid + k * NT;
        const int q = e / kVec, d4 = e - q * kVec;
        if (q < nq)
            store_out4(p.o + rowhead(q) * HD + d4 * 4, oacc[k], wts[q * kWStride + kGroupSplits]);
    }
    if (tid == 0) {
        cnt[0] = 0u;                   // ready for the next call, which is ordered after this kernel
        trace_event(p, kTrMerged, true);
    }
}

// ---------------------------------------------------------------- combine kernel
//
// The merge of the split partials as a kernel of its own (see above).
template <int HD>
__global__ void __launch_bounds__(kCombineWarps * 32) decode_combine_kernel(const DecodeParams p)
{
    __shared__ float gw[kMaxGroups][kGroupSplits];   // weights inside each group (one level: gw[0])
    __shared__ float2 gml[kMaxGroups];               // two levels: (M_g, L_g)
    __shared__ float wts[kMaxGroups];                // two levels: weights of the groups
    extern __shared__ float4 og[];                   // two levels: [group][32] unnormalised group outputs
    const size_t rh = blockIdx.x;
    const int S = p.splits;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // The next kernel may launch at once: its own dependency wait still waits
    // for this grid to complete, and this grid completes only after the split
    // kernel it waits for here.  Its CTAs then take the SMs the split CTAs
    // leave, ready (and prefetching) by the time this merge ends.
    grid_launch_dependents();
    grid_dependency_wait();          // the split kernel's partials
    if (S <= kGroupSplits) {         // one level, one warp
        const int d4 = blockIdx.y * combine_slice<HD>() + lane;
        const bool mine = lane < combine_slice<HD>();
        const float4 *po = reinterpret_cast<const float4 *>(p.part_o + rh * S * HD) + d4;
        float4 v[kGroupSplits];
        combine_load_group<HD>(v, po, S, mine);
        const float L = merge_stats_warp(p.part_ml + rh * S, S, gw[0], lane);
        __syncwarp();
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < kGroupSplits; ++j)
            if (j < S)
                fma4(acc, gw[0][j], v[j]);
        if (mine)
            store_out4(p.o + rh * HD + d4 * 4, acc, L);
        return;
    }
    // two levels: groups of 8 splits, each merged as above into (M_g, L_g, O_g), then the groups
    merge_two_level<HD>(p, rh, blockIdx.y, warp, blockDim.x >> 5, lane, gw, gml, wts, og, [] { __syncthreads(); });
}

}  // namespace pgqa
