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
// GB300 design (see the header comment of each kernel for its roofline):
//  * one producer warp streams whole (page, kv head) tiles of K and V into a
//    ring of shared-memory stages with 3-D TMA (cp.async.bulk.tensor) and the
//    128-byte swizzle, completion counted on mbarriers;
//  * four consumer warps each take whole pages: S = Q K^T and O^T += V^T P^T
//    on the tensor cores (mma.sync m16n8k16 bf16 -> f32), all g = nh/nkv query
//    heads of the kv head packed into the MMA rows so each KV byte leaves HBM
//    once; the S accumulator fragment is, register for register, the B
//    fragment of the PV product, so P never touches shared memory;
//  * online softmax in the log2 domain with quad shuffles; the O rescale is
//    skipped when no running max moved;
//  * every wait is bounded (about one second) and reports through a device
//    error word instead of hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pgqa {

constexpr int kPage = 16;                 // tokens per KV page
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kQRows = 8;                 // query rows (heads) per CTA: one MMA n-tile
constexpr int kBoxElems = 64;             // 128-byte swizzle atom: 64 bf16 per row
constexpr int kBoxBytes = kPage * kBoxElems * 2;   // one TMA box: 16 rows x 128 B
constexpr int kMaxSplits = 256;
constexpr unsigned long long kWaitLimitNs = 1000000000ull;   // bounded waits: 1 s
constexpr unsigned int kErrTimeoutFull = 1u;
constexpr unsigned int kErrTimeoutEmpty = 2u;
constexpr float kLog2e = 1.4426950408889634f;

// Stage-ring depth and CTAs per SM by head dimension.  The ring depth is a
// multiple of the consumer-warp count: page i goes to warp i % 4 and stage
// i % kStages, so every stage is only ever consumed by one warp, which waits
// for its mbarrier phases strictly in order.  (A parity wait names the
// current or the previous phase; a warp that waited on phase k of a stage
// whose phase k-1 had not completed would pass at once.)
template <int HD>
struct Cfg;
template <>
struct Cfg<64> { static constexpr int kStages = 8, kMinBlocks = 4; };
template <>
struct Cfg<128> { static constexpr int kStages = 8, kMinBlocks = 3; };
template <>
struct Cfg<256> { static constexpr int kStages = 4, kMinBlocks = 2; };
template <>
struct Cfg<512> { static constexpr int kStages = 4, kMinBlocks = 1; };

template <int HD>
struct Smem {
    static constexpr int kTile = kPage * HD * 2;                   // one (page, kv head) tile
    static constexpr int kStage = 2 * kTile;                       // K + V
    static constexpr int kStagesBytes = Cfg<HD>::kStages * kStage;
    static constexpr int kQOff = kStagesBytes;
    static constexpr int kQBytes = kQRows * HD * 2;
    static constexpr int kBarOff = kQOff + kQBytes;
    static constexpr int kBarBytes = 2 * Cfg<HD>::kStages * 8;
    static constexpr int kMiscOff = kBarOff + kBarBytes;
    static constexpr int kTotal = kMiscOff + 16;
    static constexpr int kAlloc = kTotal + 1024;                   // slack for 1024-B alignment
    // merge scratch, reusing the stage ring once every page is consumed
    static constexpr int kObufStride = HD + 4;                     // floats; padded against bank conflicts
    static constexpr int kObufBytes = kConsumerWarps * kQRows * kObufStride * 4;
    static constexpr int kMlOff = kObufBytes;                      // float2 [warps][8]
    static constexpr int kStatOff = kMlOff + kConsumerWarps * kQRows * 8;   // per-q weights, L
    static_assert(kStatOff + kQRows * (kMaxSplits + 2) * 4 <= kStagesBytes, "merge scratch");
    static_assert(kAlloc <= 227 * 1024, "shared memory");
    static_assert(Cfg<HD>::kStages % kConsumerWarps == 0, "each stage must belong to one consumer warp");
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
    int rows, nh, nkv, window, splits, g, hsg;   // hsg = head subgroups of 8 per kv head
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
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

// Waits for the phase with the given parity; gives up after kWaitLimitNs,
// records `code` in the error word and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, unsigned int *err,
                                                  unsigned int code)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > kWaitLimitNs) {
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

__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void consumer_bar_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerThreads) : "memory");
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
// One (row, head)'s S partials (m_s, l_s, O_s) -> o.  Shared verbatim by the
// last-CTA merge and the combine kernel, so the two give the same bits:
//   M = max_s m_s,  w_s = (m_s == -inf) ? 0 : 2^(m_s - M),  L = sum_s w_s l_s,
//   o[d] = bf16_rn( (sum_s w_s O_s[d]) / L ), or 0 when L == 0,
// accumulated in split order with explicit fused multiply-adds.

__device__ __forceinline__ float merge_stats(const float2 *ml, int splits, float *w)
{
    float mx = -INFINITY;
    for (int s = 0; s < splits; ++s)
        mx = fmaxf(mx, __ldcg(&ml[s].x));
    float L = 0.f;
    for (int s = 0; s < splits; ++s) {
        const float2 v = __ldcg(&ml[s]);
        const float ws = (v.x == -INFINITY) ? 0.f : exp2f(v.x - mx);
        w[s] = ws;
        L = __fmaf_rn(ws, v.y, L);
    }
    return L;
}

__device__ __forceinline__ __nv_bfloat16 merge_value(const float *po, int hd, const float *w, int splits,
                                                     float L)
{
    float acc = 0.f;
    for (int s = 0; s < splits; ++s)
        acc = __fmaf_rn(w[s], __ldcg(po + static_cast<size_t>(s) * hd), acc);
    return L > 0.f ? __float2bfloat16_rn(__fdiv_rn(acc, L)) : __float2bfloat16_rn(0.f);
}

// ---------------------------------------------------------------- main kernel
//
// Grid (splits, nkv * hsg, rows); block = 4 consumer warps + 1 producer warp.
// HBM-bound: per (page, kv head) it moves 2 * 16 * hd * 2 bytes and runs
// 3 * hd / 16 MMAs, far below the tensor pipe's rate.
template <int HD>
__global__ void __launch_bounds__(kThreads, Cfg<HD>::kMinBlocks)
    decode_split_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                        const DecodeParams p)
{
    using SM = Smem<HD>;
    constexpr int NS = Cfg<HD>::kStages;
    constexpr int kChunks = HD / kBoxElems;   // TMA boxes per tile
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_q = s_base + SM::kQOff;
    const uint32_t s_full = s_base + SM::kBarOff;
    const uint32_t s_empty = s_full + NS * 8;
    int *s_misc = reinterpret_cast<int *>(smem + SM::kMiscOff);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int split = blockIdx.x;
    const int kh = blockIdx.y / p.hsg;
    const int hsg = blockIdx.y - kh * p.hsg;
    const int row = blockIdx.z;
    const int head0 = kh * p.g + hsg * kQRows;
    const int nq = min(kQRows, p.g - hsg * kQRows);
    const int S = p.splits;

    // visible range of this row and this split's page-aligned share of it
    const int qp = __ldg(p.qpos + row);
    const int hi = p.kvpos ? __ldg(p.kvpos + row) : qp;
    const int lo = p.window > 0 ? max(0, qp + 1 - p.window) : 0;
    int page_begin = 0, npages_mine = 0;
    if (hi >= lo) {
        const int p0 = lo >> 4;
        const int np = (hi >> 4) - p0 + 1;
        page_begin = p0 + static_cast<int>((static_cast<long long>(split) * np) / S);
        npages_mine = p0 + static_cast<int>((static_cast<long long>(split + 1) * np) / S) - page_begin;
    }

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(s_full + 8 * s, 1);
            mbar_init(s_empty + 8 * s, 1);
        }
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ------------------------------------------------ producer warp
        if (lane == 0) {
            tma_prefetch_map(&tm_k);
            tma_prefetch_map(&tm_v);
        }
        const int32_t *tbl = p.block_table + __ldg(p.off + row) + page_begin;
        bool ok = true;
        for (int c0 = 0; c0 < npages_mine && ok; c0 += 32) {
            int phys = 0;
            if (c0 + lane < npages_mine) {
                phys = __ldg(tbl + c0 + lane);
                if (p.page_map)
                    phys = __ldg(p.page_map + phys);
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
#pragma unroll
                        for (int c = 0; c < kChunks; ++c) {
                            tma_load_3d(dk + c * kBoxBytes, &tm_k, bar, c * kBoxElems, 0, tile);
                            tma_load_3d(dv + c * kBoxBytes, &tm_v, bar, c * kBoxElems, 0, tile);
                        }
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    // Q rows head0 .. head0+nq-1 of this row -> shared memory, swizzled by
    // 16-byte unit (unit u of q-row r sits at u ^ r); rows >= nq are zero.
    {
        constexpr int kUnits = HD / 8;
        const uint4 *qg = reinterpret_cast<const uint4 *>(p.q + (static_cast<size_t>(row) * p.nh + head0) * HD);
        for (int idx = tid; idx < kQRows * kUnits; idx += kConsumerThreads) {
            const int r = idx / kUnits, u = idx - r * kUnits;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (r < nq)
                v = __ldg(qg + r * kUnits + u);
            *reinterpret_cast<uint4 *>(smem + SM::kQOff + r * HD * 2 + ((u ^ r) << 4)) = v;
        }
    }
    consumer_bar_sync();

    const int gid = lane >> 2;     // MMA group: query row of S, d row of O^T
    const int tig = lane & 3;      // thread in group
    const bool row_live = gid < nq;

    float acc[HD / 16][4];
#pragma unroll
    for (int mt = 0; mt < HD / 16; ++mt)
        acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
    float m_run = -INFINITY;       // running max of q-row gid, log2 units
    float l_run = 0.f;             // this thread's share of the running sum

    // per-lane ldmatrix row/unit selectors
    const int lm_i = lane >> 3, lm_r = lane & 7;
    const int tok_sel = (lm_i >> 1) * 8 + lm_r;    // K/V token row addressed by this lane
    const int half_sel = lm_i & 1;                 // low / high 8 columns

    bool ok = true;
    for (int i = warp; i < npages_mine; i += kConsumerWarps) {
        const int st = i % NS;
        if (ok)
            ok = mbar_wait_bounded(s_full + 8 * st, (i / NS) & 1, p.err, kErrTimeoutFull);
        if (!ok)
            break;
        const uint32_t sk = s_base + st * SM::kStage;
        const uint32_t sv = sk + SM::kTile;
        const int pos0 = (page_begin + i) * kPage;

        // S = Q K^T over the page's 16 tokens: two n-tiles of 8 tokens
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kc = 0; kc < HD / 16; kc += 2) {
            uint32_t qa0, qa2, qb0, qb2;
            {
                const int u = kc * 2 + lm_i;    // 16-byte unit of the Q row
                ldsm_x4(s_q + lm_r * HD * 2 + ((u ^ lm_r) << 4), qa0, qa2, qb0, qb2);
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int k16 = kc + h;
                const int chunk = k16 >> 2;
                const int u = (k16 & 3) * 2 + half_sel;
                uint32_t b0n0, b1n0, b0n1, b1n1;
                ldsm_x4(sk + chunk * kBoxBytes + swz(tok_sel, u), b0n0, b1n0, b0n1, b1n1);
                const uint32_t a0 = h ? qb0 : qa0, a2 = h ? qb2 : qa2;
                mma_bf16_16816(s0, a0, 0u, a2, 0u, b0n0, b1n0);
                mma_bf16_16816(s1, a0, 0u, a2, 0u, b0n1, b1n1);
            }
        }

        // mask to [lo, hi], scale to log2 units
        const int t0 = pos0 + 2 * tig;
        float x[4];
        x[0] = (row_live && t0 >= lo && t0 <= hi) ? s0[0] * kLog2e : -INFINITY;
        x[1] = (row_live && t0 + 1 >= lo && t0 + 1 <= hi) ? s0[1] * kLog2e : -INFINITY;
        x[2] = (row_live && t0 + 8 >= lo && t0 + 8 <= hi) ? s1[0] * kLog2e : -INFINITY;
        x[3] = (row_live && t0 + 9 >= lo && t0 + 9 <= hi) ? s1[1] * kLog2e : -INFINITY;

        // online softmax for q-row gid (the 4 lanes of a group hold its 16 scores)
        float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float m_new = fmaxf(m_run, mx);
        float alpha = 1.f;
        float pr[4] = {0.f, 0.f, 0.f, 0.f};
        if (m_new != -INFINITY) {
            alpha = exp2f(m_run - m_new);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pr[e] = bf16_round(exp2f(x[e] - m_new));
        }
        m_run = m_new;
        l_run = __fmaf_rn(l_run, alpha, (pr[0] + pr[1]) + (pr[2] + pr[3]));
        const uint32_t pb0 = pack_bf16x2(pr[0], pr[1]);   // P^T rows 2tig, 2tig+1 -> B frag
        const uint32_t pb1 = pack_bf16x2(pr[2], pr[3]);   // P^T rows 8+2tig, 9+2tig

        // O^T columns are q-rows 2tig and 2tig+1: fetch their alphas
        const float al_a = __shfl_sync(0xffffffffu, alpha, (2 * tig) * 4);
        const float al_b = __shfl_sync(0xffffffffu, alpha, (2 * tig + 1) * 4);
        if (__any_sync(0xffffffffu, al_a != 1.f || al_b != 1.f)) {
#pragma unroll
            for (int mt = 0; mt < HD / 16; ++mt) {
                acc[mt][0] *= al_a;
                acc[mt][1] *= al_b;
                acc[mt][2] *= al_a;
                acc[mt][3] *= al_b;
            }
        }

        // positions of this page outside [lo, hi] may hold any bits: zero their V rows
        if (pos0 < lo || pos0 + kPage - 1 > hi) {
            const int t = lane & 15;
            if (pos0 + t < lo || pos0 + t > hi) {
                uint8_t *vrow = smem + (sv - s_base) + t * 128;
                for (int c = (lane >> 4); c < kChunks; c += 2) {
                    uint4 *dst = reinterpret_cast<uint4 *>(vrow + c * kBoxBytes);
#pragma unroll
                    for (int u = 0; u < 8; ++u)
                        dst[u] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            __syncwarp();
        }

        // O^T += V^T P^T: hd/16 m-tiles of 16 dims
#pragma unroll
        for (int mt = 0; mt < HD / 16; ++mt) {
            const int chunk = mt >> 2;
            const int u = (mt & 3) * 2 + half_sel;
            uint32_t a0, a1, a2, a3;
            ldsm_x4_trans(sv + chunk * kBoxBytes + swz(tok_sel, u), a0, a1, a2, a3);
            mma_bf16_16816(acc[mt], a0, a1, a2, a3, pb0, pb1);
        }

        if (pos0 < lo || pos0 + kPage - 1 > hi)
            fence_proxy_async_smem();      // generic writes above vs the next TMA into this stage
        __syncwarp();
        if (lane == 0)
            mbar_arrive(s_empty + 8 * st);
    }

    // ---------------------------------------------------- CTA-level merge
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    consumer_bar_sync();      // every page consumed: the stage ring is free

    float *obuf = reinterpret_cast<float *>(smem);
    float2 *mlbuf = reinterpret_cast<float2 *>(smem + SM::kMlOff);
    float *stat = reinterpret_cast<float *>(smem + SM::kStatOff);
    {
        float *ob = obuf + warp * kQRows * SM::kObufStride;
#pragma unroll
        for (int mt = 0; mt < HD / 16; ++mt) {
            const int d = mt * 16 + gid;
            ob[(2 * tig) * SM::kObufStride + d] = acc[mt][0];
            ob[(2 * tig + 1) * SM::kObufStride + d] = acc[mt][1];
            ob[(2 * tig) * SM::kObufStride + d + 8] = acc[mt][2];
            ob[(2 * tig + 1) * SM::kObufStride + d + 8] = acc[mt][3];
        }
        if (tig == 0)
            mlbuf[warp * kQRows + gid] = make_float2(m_run, l_run);
    }
    consumer_bar_sync();

    // per q-row: weights of the 4 warps' partials, the CTA's (M, L)
    if (tid < nq) {
        float mx = -INFINITY;
        for (int w = 0; w < kConsumerWarps; ++w)
            mx = fmaxf(mx, mlbuf[w * kQRows + tid].x);
        float L = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) {
            const float2 v = mlbuf[w * kQRows + tid];
            const float ws = (v.x == -INFINITY) ? 0.f : exp2f(v.x - mx);
            stat[tid * (kConsumerWarps + 2) + w] = ws;
            L = __fmaf_rn(ws, v.y, L);
        }
        stat[tid * (kConsumerWarps + 2) + kConsumerWarps] = L;
        stat[tid * (kConsumerWarps + 2) + kConsumerWarps + 1] = mx;
        if (S > 1)
            p.part_ml[(static_cast<size_t>(row) * p.nh + head0 + tid) * S + split] = make_float2(mx, L);
    }
    consumer_bar_sync();

    for (int idx = tid; idx < nq * HD; idx += kConsumerThreads) {
        const int q = idx / HD, d = idx - q * HD;
        const float *st = stat + q * (kConsumerWarps + 2);
        float o = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
            o = __fmaf_rn(st[w], obuf[(w * kQRows + q) * SM::kObufStride + d], o);
        const size_t rh = static_cast<size_t>(row) * p.nh + head0 + q;
        if (S == 1) {
            const float L = st[kConsumerWarps];
            p.o[rh * HD + d] = L > 0.f ? __float2bfloat16_rn(__fdiv_rn(o, L)) : __float2bfloat16_rn(0.f);
        } else {
            p.part_o[(rh * S + split) * HD + d] = o;
        }
    }
    if (S == 1 || p.counters == nullptr)
        return;

    // ---------------------------------------------------- last-CTA merge
    __threadfence();
    consumer_bar_sync();
    const int tile_id = (row * p.nkv + kh) * p.hsg + hsg;
    if (tid == 0)
        s_misc[0] = static_cast<int>(atomicAdd(p.counters + tile_id, 1u));
    consumer_bar_sync();
    if (s_misc[0] != S - 1)
        return;
    __threadfence();
    float *wts = stat;      // [nq][S + 1]
    if (tid < nq) {
        const size_t rh = static_cast<size_t>(row) * p.nh + head0 + tid;
        wts[tid * (S + 1) + S] = merge_stats(p.part_ml + rh * S, S, wts + tid * (S + 1));
    }
    consumer_bar_sync();
    for (int idx = tid; idx < nq * HD; idx += kConsumerThreads) {
        const int q = idx / HD, d = idx - q * HD;
        const size_t rh = static_cast<size_t>(row) * p.nh + head0 + q;
        p.o[rh * HD + d] = merge_value(p.part_o + rh * S * HD + d, HD, wts + q * (S + 1), S, wts[q * (S + 1) + S]);
    }
    if (tid == 0)
        p.counters[tile_id] = 0u;      // ready for the next call, which is ordered after this kernel
}

// ---------------------------------------------------------------- combine kernel
//
// One CTA per (row, head): merges the S partials with the same routine as the
// last-CTA path.  Reads rows*nh*S*(hd+2)*4 bytes, writes rows*nh*hd*2.
template <int HD>
__global__ void __launch_bounds__(128) decode_combine_kernel(const DecodeParams p)
{
    __shared__ float wts[kMaxSplits + 1];
    const size_t rh = blockIdx.x;
    const int S = p.splits;
    if (threadIdx.x == 0)
        wts[S] = merge_stats(p.part_ml + rh * S, S, wts);
    __syncthreads();
    for (int d = threadIdx.x; d < HD; d += blockDim.x)
        p.o[rh * HD + d] = merge_value(p.part_o + rh * S * HD + d, HD, wts, S, wts[S]);
}

}  // namespace pgqa
