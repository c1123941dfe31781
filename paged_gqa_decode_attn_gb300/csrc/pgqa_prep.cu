// The step before paged attention: per-head RMSNorm of the projected Q and K
// (weights; V weightless, optional), rotary position embedding of Q and K over
// the first rotary_dim dims (rotate-half pairs (i, i + rotary_dim/2), angle
// pos * theta^(-2i/rotary_dim), the remaining dims passed through), Q written
// to its buffer and K, V written into the [page][nkv][16][hd] pools at the
// token's slot: page block_table[off[r] + pos[r]/16] (then page_map), slot
// pos[r] % 16.  It is the QK-RMSNorm/RoPE pool write whose device gates
// pegainfer PR #1002 describes ("anchor -> flat kernel -> paged prefill ->
// paged decode"); the pages give no formula, so the plainest reading is taken
// (include/pgqa.h states it).
//
// Memory-bound: every head vector is read once and written once.  Persistent
// CTAs, two per SM, each a producer warp and eight consumer warps around a
// ring of shared-memory stages.  A work item is a run of up to vpi head
// vectors of one row (all of a row when they fit).  The producer fetches an
// item's vectors -- contiguous runs of q_in, k_in, v_in -- with bulk copies
// that complete on the stage's full barrier, after writing the row's slot
// (pos, page) and its norm-and-rotation table into the stage.  Consumers work
// the vectors out of shared memory, each warp a contiguous run of them, up to
// four of one kind side by side (so that their shuffle chains overlap) with
// lane l holding dims [E l, E l + E), E = hd / 32, store them and release the
// stage.
//
// Norm and rotation fold into the table: with rs = 1/sqrt(mean x^2 + eps)
// common to the vector, dim d becomes rs (x_d A_d + x_p B_d), p the partner
// d +- half, A_d = w_d cos a, B_d = -w_p sin a (low half) or +w_p sin a (high
// half), and A_d = w_d, B_d = 0 past rotary_dim.  A lane shuffles its
// partner's raw bf16 words and does two packed f32x2 ops and a scale.  The
// angle is carried in turns from an f64 frequency split into a float pair, so
// dropping whole turns is exact and positions up to 2^24 keep ~1e-7 turns.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "pgqa.h"
#include "pgqa_device.cuh"

namespace pgqa {

int device_info(int *num_sms, unsigned int **err);   // pgqa_api.cu
int current_context_id(unsigned long long *id);      // pgqa_api.cu

namespace {

constexpr int kPrepConsumerWarps = 8;
constexpr int kPrepThreads = 32 * (kPrepConsumerWarps + 1);
constexpr int kPrepCtasPerSm = 2;
constexpr int kPrepSmemBudget = 110 * 1024;   // per CTA, two beside each other on an SM
constexpr int kPrepMaxStages = 8;
constexpr int kPrepItemDataBytes = 16 * 1024;  // head-vector bytes of one item at most
constexpr int kPrepMetaBytes = 16;

struct PrepParams {
    __nv_bfloat16 *q_out;
    __nv_bfloat16 *k_pool;
    __nv_bfloat16 *v_pool;
    const __nv_bfloat16 *q_in;
    const __nv_bfloat16 *k_in;
    const __nv_bfloat16 *v_in;
    const __nv_bfloat16 *q_weight;
    const __nv_bfloat16 *k_weight;
    const int32_t *pos;
    const int32_t *block_table;
    const int32_t *off;
    const int32_t *page_map;
    unsigned int *err;
    int nh, nkv, rotary_dim, norm_v;
    int vpi;            // head vectors per item
    int items_per_row;  // ceil((nh + 2 nkv) / vpi)
    int nitems;         // rows * items_per_row
    int stages;
    int stage_bytes;    // table (16 hd) + meta (16) + vpi * hd * 2
    float eps;
    float2 turns[256];  // theta^(-2i/rotary_dim) / (2 pi) = x + y, i < rotary_dim / 2
};

// E bf16 of one lane, packed two to a word as loaded and stored.
template <int E>
struct Packed {
    uint32_t w[E / 2];
};

template <int E>
__device__ __forceinline__ void load_packed(const __nv_bfloat16 *src, Packed<E> &r)
{
    if constexpr (E == 2) {
        r.w[0] = *reinterpret_cast<const unsigned int *>(src);
    } else if constexpr (E == 4) {
        const uint2 t = *reinterpret_cast<const uint2 *>(src);
        r.w[0] = t.x;
        r.w[1] = t.y;
    } else {
#pragma unroll
        for (int c = 0; c < E / 8; ++c) {
            const uint4 t = reinterpret_cast<const uint4 *>(src)[c];
            r.w[4 * c] = t.x;
            r.w[4 * c + 1] = t.y;
            r.w[4 * c + 2] = t.z;
            r.w[4 * c + 3] = t.w;
        }
    }
}

template <int E>
__device__ __forceinline__ void store_packed(__nv_bfloat16 *dst, const Packed<E> &r)
{
    if constexpr (E == 2) {
        *reinterpret_cast<unsigned int *>(dst) = r.w[0];
    } else if constexpr (E == 4) {
        *reinterpret_cast<uint2 *>(dst) = make_uint2(r.w[0], r.w[1]);
    } else {
#pragma unroll
        for (int c = 0; c < E / 8; ++c)
            reinterpret_cast<uint4 *>(dst)[c] = make_uint4(r.w[4 * c], r.w[4 * c + 1], r.w[4 * c + 2], r.w[4 * c + 3]);
    }
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// The angle of rotation pair i at position fpos, as (cos, sin): carried in
// turns, pos * (g.x + g.y) with the product's rounding error recovered
// exactly, so dropping whole turns loses nothing.
__device__ __forceinline__ void pair_angle(float fpos, float2 g, float &c, float &s)
{
    const float t = fpos * g.x;
    const float t_err = fmaf(fpos, g.x, -t);
    const float frac = (t - rintf(t)) + fmaf(fpos, g.y, t_err);
    sincospif(2.0f * frac, &s, &c);
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}

// Producer warp: item n of this CTA is global item blockIdx.x + n gridDim.x
// (row it / items_per_row, run it % items_per_row) in stage n % stages.
template <int HD>
__device__ void prep_producer(const PrepParams &p, unsigned char *smem, uint32_t bar_full, uint32_t bar_empty,
                              int my_items)
{
    constexpr int E = HD / 32;
    constexpr int kPairs = E / 2;
    const int lane = threadIdx.x & 31;
    const int d0 = E * lane;
    const int half = p.rotary_dim >> 1;
    const bool low = d0 < half, high = !low && d0 < p.rotary_dim;
    const int pd0 = low ? d0 + half : (high ? d0 - half : d0);
    // this lane's weights and its rotation partners' (the table of lane l
    // serves consumer lane l); at hd 512 they are read again for every item
    // (from L1), since holding them beside the frequencies would not fit the
    // registers of two CTAs per SM
    constexpr bool kHoldWeights = HD <= 256;
    Packed<E> wq, wk, pq, pk;
    auto load_weights = [&]() {
        load_packed<E>(p.q_weight + d0, wq);
        load_packed<E>(p.k_weight + d0, wk);
        load_packed<E>(p.q_weight + pd0, pq);
        load_packed<E>(p.k_weight + pd0, pk);
    };
    if constexpr (kHoldWeights)
        load_weights();
    // this lane's frequencies, read once: a parameter read with a per-lane
    // index is serialised across the warp
    float2 g[E];
#pragma unroll
    for (int e = 0; e < E; ++e)
        g[e] = (low || high) ? p.turns[(low ? d0 : pd0) + e] : make_float2(0.f, 0.f);
    const int nvec = p.nh + 2 * p.nkv;

    for (int b = 0; b < my_items; b += 32) {
        // the slots of 32 items, one per lane
        int pos_j = 0, page_j = 0;
        if (b + lane < my_items) {
            const int r = (blockIdx.x + (b + lane) * gridDim.x) / p.items_per_row;
            pos_j = __ldg(p.pos + r);
            page_j = __ldg(p.block_table + __ldg(p.off + r) + pos_j / 16);
            if (p.page_map)
                page_j = __ldg(p.page_map + page_j);
        }
        const int nb = min(32, my_items - b);
        for (int k = 0; k < nb; ++k) {
            const int n = b + k;
            const int stage = n % p.stages;
            const int pos = __shfl_sync(0xffffffffu, pos_j, k);
            const int page = __shfl_sync(0xffffffffu, page_j, k);
            if (n >= p.stages) {
                bool ok = true;
                if (lane == 0)
                    ok = mbar_wait_bounded(bar_empty + 8 * stage, ((n / p.stages) - 1) & 1, p.err, kErrTimeoutEmpty);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0))
                    return;
                mbar_try_wait(bar_empty + 8 * stage, ((n / p.stages) - 1) & 1);   // every lane acquires
            }
            unsigned char *st = smem + static_cast<size_t>(stage) * p.stage_bytes;
            // table: {A_d, A_d+1, B_d, B_d+1} of lane l's word w (d = E l + 2w)
            // at [32 w + l], Q then K
            float4 *tq = reinterpret_cast<float4 *>(st) + lane;
            float4 *tk = tq + 32 * kPairs;
            const float fpos = static_cast<float>(pos);
            if constexpr (!kHoldWeights)
                load_weights();
#pragma unroll
            for (int w = 0; w < kPairs; ++w) {
                const float wq0 = bf16_lo(wq.w[w]), wq1 = bf16_hi(wq.w[w]);
                const float wk0 = bf16_lo(wk.w[w]), wk1 = bf16_hi(wk.w[w]);
                if (low || high) {
                    float c0, s0, c1, s1;
                    pair_angle(fpos, g[2 * w], c0, s0);
                    pair_angle(fpos, g[2 * w + 1], c1, s1);
                    if (low) {
                        s0 = -s0;
                        s1 = -s1;
                    }
                    tq[32 * w] = make_float4(wq0 * c0, wq1 * c1, bf16_lo(pq.w[w]) * s0, bf16_hi(pq.w[w]) * s1);
                    tk[32 * w] = make_float4(wk0 * c0, wk1 * c1, bf16_lo(pk.w[w]) * s0, bf16_hi(pk.w[w]) * s1);
                } else {
                    tq[32 * w] = make_float4(wq0, wq1, 0.f, 0.f);
                    tk[32 * w] = make_float4(wk0, wk1, 0.f, 0.f);
                }
            }
            const int it = blockIdx.x + n * gridDim.x;
            const int r = it / p.items_per_row;
            const int va = (it % p.items_per_row) * p.vpi;
            const int vb = min(nvec, va + p.vpi);
            const uint32_t bar = bar_full + 8 * stage;
            if (lane == 0) {
                *reinterpret_cast<int2 *>(st + 16 * HD) = make_int2(pos, page);
                mbar_arrive_expect_tx(bar, static_cast<uint32_t>((vb - va) * HD * 2));
                const uint32_t dst = smem_u32(st) + 16 * HD + kPrepMetaBytes;
                int a = va, e = min(vb, p.nh);
                if (a < e)
                    bulk_g2s(dst + (a - va) * HD * 2, p.q_in + (static_cast<size_t>(r) * p.nh + a) * HD,
                             (e - a) * HD * 2, bar);
                a = max(va, p.nh);
                e = min(vb, p.nh + p.nkv);
                if (a < e)
                    bulk_g2s(dst + (a - va) * HD * 2, p.k_in + (static_cast<size_t>(r) * p.nkv + a - p.nh) * HD,
                             (e - a) * HD * 2, bar);
                a = max(va, p.nh + p.nkv);
                if (a < vb)
                    bulk_g2s(dst + (a - va) * HD * 2,
                             p.v_in + (static_cast<size_t>(r) * p.nkv + a - p.nh - p.nkv) * HD, (vb - a) * HD * 2,
                             bar);
            } else {
                mbar_arrive(bar);
            }
        }
    }
}

// NV head vectors of one kind, consecutive in the stage, worked side by side
// so that their dependent chains (the sum-of-squares shuffles, rsqrt, the
// partner shuffles) overlap.  Vector j goes to dst + j * dst_stride.  Each
// vector's arithmetic and its order are those of a vector worked alone.
template <int HD, int NV>
__device__ __forceinline__ void norm_rotate(const __nv_bfloat16 *src, __nv_bfloat16 *dst, size_t dst_stride,
                                            const float4 (&tab)[HD / 64], bool scale, float eps, int src_lane)
{
    constexpr int E = HD / 32;
    constexpr int kPairs = E / 2;
    Packed<E> in[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j)
        load_packed<E>(src + j * HD, in[j]);
    // the f32 values are re-derived from the packed words where they are
    // used (a shift or a mask): keeping them would double the registers
    float ss[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kPairs; ++w) {
            const float2 x = make_float2(bf16_lo(in[j].w[w]), bf16_hi(in[j].w[w]));
            acc = __ffma2_rn(x, x, acc);
        }
        ss[j] = acc.x + acc.y;
    }
    uint32_t yw[NV][kPairs];
#pragma unroll
    for (int j = 0; j < NV; ++j)
#pragma unroll
        for (int w = 0; w < kPairs; ++w)
            yw[j][w] = __shfl_sync(0xffffffffu, in[j].w[w], src_lane);
#pragma unroll
    for (int m = 16; m; m >>= 1)
#pragma unroll
        for (int j = 0; j < NV; ++j)
            ss[j] += __shfl_xor_sync(0xffffffffu, ss[j], m);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
        const float rs = scale ? rsqrtf(ss[j] * (1.0f / HD) + eps) : 1.0f;
        const float2 rs2 = make_float2(rs, rs);
        Packed<E> out;
#pragma unroll
        for (int w = 0; w < kPairs; ++w) {
            const float2 x = make_float2(bf16_lo(in[j].w[w]), bf16_hi(in[j].w[w]));
            float2 u = __fmul2_rn(x, make_float2(tab[w].x, tab[w].y));
            u = __ffma2_rn(make_float2(bf16_lo(yw[j][w]), bf16_hi(yw[j][w])), make_float2(tab[w].z, tab[w].w), u);
            u = __fmul2_rn(u, rs2);
            const __nv_bfloat162 t = __floats2bfloat162_rn(u.x, u.y);
            out.w[w] = *reinterpret_cast<const uint32_t *>(&t);
        }
        store_packed<E>(dst + j * dst_stride, out);
    }
}

template <int HD>
__device__ void prep_consumer(const PrepParams &p, const unsigned char *smem, uint32_t bar_full,
                              uint32_t bar_empty, int my_items)
{
    constexpr int E = HD / 32;
    constexpr int kPairs = E / 2;
    // vectors worked side by side at most (hd 512 keeps one: more would not
    // fit the registers of two CTAs per SM)
    constexpr int kNv = HD <= 256 ? 4 : 1;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int d0 = E * lane;
    const int half = p.rotary_dim >> 1;
    const int nl = half / E;
    // this lane's dims are all low, all high or all beyond rotary_dim
    // (rotary_dim is a multiple of 2E); past it the partner is the lane itself
    const int src_lane = d0 < half ? lane + nl : (d0 < p.rotary_dim ? lane - nl : lane);
    const int nvec = p.nh + 2 * p.nkv;

    for (int n = 0; n < my_items; ++n) {
        const int stage = n % p.stages;
        const bool ok = mbar_wait_bounded(bar_full + 8 * stage, (n / p.stages) & 1, p.err, kErrTimeoutFull);
        if (!__all_sync(0xffffffffu, ok))
            return;
        const unsigned char *st = smem + static_cast<size_t>(stage) * p.stage_bytes;
        const int2 meta = *reinterpret_cast<const int2 *>(st + 16 * HD);
        const int it = blockIdx.x + n * gridDim.x;
        const int r = it / p.items_per_row;
        const int va = (it % p.items_per_row) * p.vpi;
        const int vb = min(nvec, va + p.vpi);
        const size_t slot = (static_cast<size_t>(meta.y) * p.nkv * 16 + meta.x % 16) * HD + d0;
        const unsigned char *data = st + 16 * HD + kPrepMetaBytes;

        // warp w takes a contiguous run of the item's vectors, so Q, K and V
        // come in long runs and the table of the current kind stays in
        // registers; V takes A = 1, B = 0 and, without norm_v, rs = 1
        const int cnt = (vb - va + kPrepConsumerWarps - 1) / kPrepConsumerWarps;
        const int wa = va + warp * cnt;
        const int wb = min(vb, wa + cnt);
        int tab_kind = -1;
        float4 tab[kPairs];
        for (int v = wa; v < wb;) {
            const int kind = v < p.nh ? 0 : (v < p.nh + p.nkv ? 1 : 2);
            if (kind != tab_kind) {
                const float4 *t = reinterpret_cast<const float4 *>(st) + (kind == 0 ? 0 : 32 * kPairs) + lane;
#pragma unroll
                for (int w = 0; w < kPairs; ++w)
                    tab[w] = kind == 2 ? make_float4(1.f, 1.f, 0.f, 0.f) : t[32 * w];
                tab_kind = kind;
            }
            // the run of this kind left to the warp
            const int kind_end = min(wb, kind == 0 ? p.nh : (kind == 1 ? p.nh + p.nkv : nvec));
            const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(data) + (v - va) * HD + d0;
            const bool scale = !(kind == 2 && !p.norm_v);
            __nv_bfloat16 *dst;
            size_t stride = static_cast<size_t>(16) * HD;
            if (kind == 0) {
                dst = p.q_out + (static_cast<size_t>(r) * p.nh + v) * HD + d0;
                stride = HD;
            } else if (kind == 2) {
                dst = p.v_pool + slot + static_cast<size_t>(v - p.nh - p.nkv) * 16 * HD;
            } else {
                dst = p.k_pool + slot + static_cast<size_t>(v - p.nh) * 16 * HD;
            }
            if (kNv >= 4 && v + 4 <= kind_end) {
                norm_rotate<HD, (kNv >= 4 ? 4 : 1)>(src, dst, stride, tab, scale, p.eps, src_lane);
                v += 4;
            } else if (kNv >= 2 && v + 2 <= kind_end) {
                norm_rotate<HD, (kNv >= 2 ? 2 : 1)>(src, dst, stride, tab, scale, p.eps, src_lane);
                v += 2;
            } else {
                norm_rotate<HD, 1>(src, dst, stride, tab, scale, p.eps, src_lane);
                v += 1;
            }
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(bar_empty + 8 * stage);
    }
}

template <int HD>
__global__ void __launch_bounds__(kPrepThreads, kPrepCtasPerSm) qk_norm_rope_kernel(const __grid_constant__ PrepParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const uint32_t bar_full = smem_u32(smem) + p.stages * p.stage_bytes;
    const uint32_t bar_empty = bar_full + 8 * p.stages;
    if (threadIdx.x == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(bar_full + 8 * s, 32);
            mbar_init(bar_empty + 8 * s, kPrepConsumerWarps);
        }
        mbar_init_fence();
    }
    __syncthreads();
    const int my_items =
        p.nitems > static_cast<int>(blockIdx.x) ? (p.nitems - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
    if ((threadIdx.x >> 5) == kPrepConsumerWarps)
        prep_producer<HD>(p, smem, bar_full, bar_empty, my_items);
    else
        prep_consumer<HD>(p, smem, bar_full, bar_empty, my_items);
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

template <int HD>
cudaError_t launch_prep(const PrepParams &p, int grid, cudaStream_t s)
{
    const int bytes = p.stages * p.stage_bytes + 16 * p.stages;
    // the smem attribute belongs to a CUDA context: set once per context
    // (a device reset makes a new one) on each device
    static std::mutex mu;
    static unsigned long long set_for_ctx[64];   // 0: not set in any context yet
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    unsigned long long ctx = 0;
    if (current_context_id(&ctx) != PGQA_OK)
        ctx = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64 || ctx == 0 || set_for_ctx[dev] != ctx) {
            e = cudaFuncSetAttribute(qk_norm_rope_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     kPrepSmemBudget);
            if (e != cudaSuccess)
                return e;
            if (dev >= 0 && dev < 64)
                set_for_ctx[dev] = ctx;
        }
    }
    qk_norm_rope_kernel<HD><<<grid, kPrepThreads, bytes, s>>>(p);
    return cudaGetLastError();
}

}  // namespace
}  // namespace pgqa

extern "C" int pgqa_qk_norm_rope_write(void *q_out, void *k_pool, void *v_pool, const void *q_in, const void *k_in,
                                       const void *v_in, const void *q_weight, const void *k_weight,
                                       const int32_t *pos, const int32_t *block_table, const int32_t *off,
                                       const int32_t *page_map, int rows, int nh, int nkv, int hd, int rotary_dim,
                                       float theta, float eps, int norm_v, void *stream)
{
    if (rows < 0 || nh < 1 || nkv < 1 || nh % nkv != 0 || !(theta > 0.f) || !std::isfinite(theta) || !(eps >= 0.f))
        return PGQA_ERR_INVALID_ARGUMENT;
    if (hd != 64 && hd != 128 && hd != 256 && hd != 512)
        return PGQA_ERR_UNSUPPORTED_HD;
    if (rotary_dim < 0 || rotary_dim > hd || rotary_dim % (hd / 16) != 0)
        return PGQA_ERR_INVALID_ARGUMENT;
    if (rows == 0)
        return PGQA_OK;
    if (!q_out || !k_pool || !v_pool || !q_in || !k_in || !v_in || !q_weight || !k_weight || !pos || !block_table ||
        !off)
        return PGQA_ERR_INVALID_ARGUMENT;
    const void *bufs[] = {q_out, k_pool, v_pool, q_in, k_in, v_in, q_weight, k_weight};
    for (const void *b : bufs)
        if (!pgqa::aligned16(b))
            return PGQA_ERR_MISALIGNED;
    const long long nvec = static_cast<long long>(nh) + 2ll * nkv;
    if (nvec * rows > (1ll << 31) - 1)
        return PGQA_ERR_INVALID_ARGUMENT;
    int num_sms = 0;
    unsigned int *err = nullptr;
    const int st = pgqa::device_info(&num_sms, &err);
    if (st != PGQA_OK)
        return st;

    pgqa::PrepParams p;
    p.q_out = static_cast<__nv_bfloat16 *>(q_out);
    p.k_pool = static_cast<__nv_bfloat16 *>(k_pool);
    p.v_pool = static_cast<__nv_bfloat16 *>(v_pool);
    p.q_in = static_cast<const __nv_bfloat16 *>(q_in);
    p.k_in = static_cast<const __nv_bfloat16 *>(k_in);
    p.v_in = static_cast<const __nv_bfloat16 *>(v_in);
    p.q_weight = static_cast<const __nv_bfloat16 *>(q_weight);
    p.k_weight = static_cast<const __nv_bfloat16 *>(k_weight);
    p.pos = pos;
    p.block_table = block_table;
    p.off = off;
    p.page_map = page_map;
    p.err = err;
    p.nh = nh;
    p.nkv = nkv;
    p.rotary_dim = rotary_dim;
    p.norm_v = norm_v ? 1 : 0;
    p.eps = eps;
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    for (int i = 0; i < rotary_dim / 2; ++i) {
        const double g = std::pow(static_cast<double>(theta), -2.0 * i / rotary_dim) / kTwoPi;
        const float hi = static_cast<float>(g);
        p.turns[i] = make_float2(hi, static_cast<float>(g - static_cast<double>(hi)));
    }
    // Items: a whole row when its vectors fit kPrepItemDataBytes, and finer
    // runs (down to 8 vectors, one per consumer warp) while there are fewer
    // items than two per CTA slot.
    int vpi = static_cast<int>(std::min<long long>(nvec, pgqa::kPrepItemDataBytes / (2 * hd)));
    const long long slots = static_cast<long long>(num_sms) * pgqa::kPrepCtasPerSm;
    while (vpi > pgqa::kPrepConsumerWarps && static_cast<long long>(rows) * ((nvec + vpi - 1) / vpi) < 2 * slots)
        vpi = std::max(pgqa::kPrepConsumerWarps, (vpi + 1) / 2);
    p.vpi = vpi;
    p.items_per_row = static_cast<int>((nvec + vpi - 1) / vpi);
    if (static_cast<long long>(rows) * p.items_per_row > (1ll << 31) - 1)
        return PGQA_ERR_INVALID_ARGUMENT;
    p.nitems = rows * p.items_per_row;
    p.stage_bytes = 16 * hd + pgqa::kPrepMetaBytes + vpi * hd * 2;
    p.stages = std::min(pgqa::kPrepMaxStages, (pgqa::kPrepSmemBudget - 16 * pgqa::kPrepMaxStages) / p.stage_bytes);
    if (p.stages < 2)
        return PGQA_ERR_INVALID_ARGUMENT;
    const int grid = static_cast<int>(std::min<long long>(p.nitems, slots));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    switch (hd) {
    case 64: e = pgqa::launch_prep<64>(p, grid, s); break;
    case 128: e = pgqa::launch_prep<128>(p, grid, s); break;
    case 256: e = pgqa::launch_prep<256>(p, grid, s); break;
    default: e = pgqa::launch_prep<512>(p, grid, s); break;
    }
    return e == cudaSuccess ? PGQA_OK : PGQA_ERR_CUDA;
}
