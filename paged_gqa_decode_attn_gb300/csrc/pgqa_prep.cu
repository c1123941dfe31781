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
// A block takes one row (or a share of its head vectors when rows are few).
// It first builds the row's rotation table: for each i < rotary_dim / 2 the
// angle pos * theta^(-2i/rotary_dim) is carried in turns, the frequency over
// 2 pi given by the host from an f64 pow as a float pair (hi + lo), so the
// product's whole turns drop out exactly and the remainder keeps ~1e-7 turns
// at any position below 2^24 -- a plain f32 angle loses ~0.01 rad by
// position 10^5.  Then one warp per head vector: lane l holds dims
// [E l, E l + E), E = hd / 32, loaded and stored as one vector; the sum of
// squares is a warp reduction and each rotation pair meets across lanes
// half / E apart by one shuffle per element.  Memory-bound: each vector is
// read once and written once; the next vector's load is issued before the
// current one is worked.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>

#include "pgqa.h"

namespace pgqa {
namespace {

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
    int nh, nkv, rotary_dim, norm_v, vec_per_block;
    float eps;
    float2 turns[256];  // theta^(-2i/rotary_dim) / (2 pi) = x + y, i < rotary_dim / 2
};

template <int E>
struct Vec;
template <>
struct Vec<2> { using T = uint32_t; };
template <>
struct Vec<4> { using T = uint2; };
template <>
struct Vec<8> { using T = uint4; };

template <int E>
__device__ __forceinline__ void load_bf16(const __nv_bfloat16 *src, float (&x)[E])
{
    if constexpr (E <= 8) {
        typename Vec<E>::T raw = *reinterpret_cast<const typename Vec<E>::T *>(src);
        const __nv_bfloat16 *b = reinterpret_cast<const __nv_bfloat16 *>(&raw);
#pragma unroll
        for (int e = 0; e < E; ++e)
            x[e] = __bfloat162float(b[e]);
    } else {
        float (&lo)[8] = *reinterpret_cast<float(*)[8]>(&x[0]);
        float (&hi)[8] = *reinterpret_cast<float(*)[8]>(&x[8]);
        load_bf16<8>(src, lo);
        load_bf16<8>(src + 8, hi);
    }
}

template <int E>
__device__ __forceinline__ void store_bf16(__nv_bfloat16 *dst, const float (&y)[E])
{
    if constexpr (E <= 8) {
        typename Vec<E>::T raw;
        __nv_bfloat16 *b = reinterpret_cast<__nv_bfloat16 *>(&raw);
#pragma unroll
        for (int e = 0; e < E; ++e)
            b[e] = __float2bfloat16_rn(y[e]);
        *reinterpret_cast<typename Vec<E>::T *>(dst) = raw;
    } else {
        const float (&lo)[8] = *reinterpret_cast<const float(*)[8]>(&y[0]);
        const float (&hi)[8] = *reinterpret_cast<const float(*)[8]>(&y[8]);
        store_bf16<8>(dst, lo);
        store_bf16<8>(dst + 8, hi);
    }
}

template <int HD>
__device__ __forceinline__ const __nv_bfloat16 *vec_src(const PrepParams &p, int r, int v)
{
    if (v < p.nh)
        return p.q_in + (static_cast<size_t>(r) * p.nh + v) * HD;
    v -= p.nh;
    const __nv_bfloat16 *base = v < p.nkv ? p.k_in : p.v_in;
    return base + (static_cast<size_t>(r) * p.nkv + (v < p.nkv ? v : v - p.nkv)) * HD;
}

// grid (rows, ny); block y takes head vectors [vec_per_block y, ..) of row
// blockIdx.x -- Q heads, then K heads, then V heads -- warp w every 8th from w.
template <int HD>
__global__ void __launch_bounds__(256) qk_norm_rope_kernel(const __grid_constant__ PrepParams p)
{
    constexpr int E = HD / 32;
    __shared__ float s_cos[HD / 2], s_sin[HD / 2];
    const int r = blockIdx.x;
    const int pos = __ldg(p.pos + r);
    const int half = p.rotary_dim >> 1;
    const float fpos = static_cast<float>(pos);
    for (int i = threadIdx.x; i < half; i += blockDim.x) {
        const float2 g = p.turns[i];
        const float t = fpos * g.x;
        const float t_err = fmaf(fpos, g.x, -t);   // exact rounding error of the product
        const float frac = (t - rintf(t)) + fmaf(fpos, g.y, t_err);
        float sn, cs;
        sincospif(2.0f * frac, &sn, &cs);
        s_cos[i] = cs;
        s_sin[i] = sn;
    }
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int d0 = E * lane;
    const int nvec = p.nh + 2 * p.nkv;
    const int vend = min(nvec, (blockIdx.y + 1) * p.vec_per_block);
    int v = blockIdx.y * p.vec_per_block + (threadIdx.x >> 5);
    if (v >= vend)
        return;
    int page = 0;
    if (p.nkv > 0) {
        page = __ldg(p.block_table + __ldg(p.off + r) + pos / 16);
        if (p.page_map)
            page = __ldg(p.page_map + page);
    }
    float x[E];
    load_bf16<E>(vec_src<HD>(p, r, v) + d0, x);
    for (; v < vend; v += 8) {
        float xn[E];
        if (v + 8 < vend)
            load_bf16<E>(vec_src<HD>(p, r, v + 8) + d0, xn);
        const bool is_q = v < p.nh;
        const bool is_v = v >= p.nh + p.nkv;
        if (!is_v || p.norm_v) {
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < E; ++e)
                ss = fmaf(x[e], x[e], ss);
#pragma unroll
            for (int k = 16; k; k >>= 1)
                ss += __shfl_xor_sync(0xffffffffu, ss, k);
            const float rs = 1.0f / sqrtf(ss / HD + p.eps);
            if (is_v) {
#pragma unroll
                for (int e = 0; e < E; ++e)
                    x[e] *= rs;
            } else {
                float w[E];
                load_bf16<E>((is_q ? p.q_weight : p.k_weight) + d0, w);
#pragma unroll
                for (int e = 0; e < E; ++e)
                    x[e] = x[e] * rs * w[e];
            }
        }
        if (!is_v && half > 0) {
            // pairs (i, i + half): this lane's dims are all low, all high or all
            // beyond rotary_dim (rotary_dim is a multiple of 2E)
            const bool low = d0 < half, high = !low && d0 < p.rotary_dim;
            const int src_lane = low ? lane + half / E : (high ? lane - half / E : lane);
            float y[E];
#pragma unroll
            for (int e = 0; e < E; ++e)
                y[e] = __shfl_sync(0xffffffffu, x[e], src_lane);
            if (low || high) {
                const int i0 = d0 - (high ? half : 0);
#pragma unroll
                for (int e = 0; e < E; ++e) {
                    const float c = s_cos[i0 + e], sn = s_sin[i0 + e];
                    x[e] = low ? fmaf(x[e], c, -y[e] * sn) : fmaf(x[e], c, y[e] * sn);
                }
            }
        }
        __nv_bfloat16 *dst;
        if (is_q) {
            dst = p.q_out + (static_cast<size_t>(r) * p.nh + v) * HD;
        } else {
            const int kh = is_v ? v - p.nh - p.nkv : v - p.nh;
            dst = (is_v ? p.v_pool : p.k_pool) + ((static_cast<size_t>(page) * p.nkv + kh) * 16 + pos % 16) * HD;
        }
        store_bf16<E>(dst + d0, x);
#pragma unroll
        for (int e = 0; e < E; ++e)
            x[e] = xn[e];
    }
}

bool aligned16(const void *ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

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
    // one vector per warp while rows are few (about 2048 blocks), else the whole row per block
    const int nvec = nh + 2 * nkv;
    const int groups = (nvec + 7) / 8;
    const int ny = std::min(groups, std::max(1, (2048 + rows - 1) / rows));
    p.vec_per_block = 8 * ((groups + ny - 1) / ny);
    const dim3 grid(rows, (nvec + p.vec_per_block - 1) / p.vec_per_block);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (hd) {
    case 64: pgqa::qk_norm_rope_kernel<64><<<grid, 256, 0, s>>>(p); break;
    case 128: pgqa::qk_norm_rope_kernel<128><<<grid, 256, 0, s>>>(p); break;
    case 256: pgqa::qk_norm_rope_kernel<256><<<grid, 256, 0, s>>>(p); break;
    default: pgqa::qk_norm_rope_kernel<512><<<grid, 256, 0, s>>>(p); break;
    }
    return cudaGetLastError() == cudaSuccess ? PGQA_OK : PGQA_ERR_CUDA;
}
