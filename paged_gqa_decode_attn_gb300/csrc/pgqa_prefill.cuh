// Paged causal prefill on GB300 (sm_103a): every row of a tile of consecutive
// rows of one sequence attends, per head, to the positions [lo(r), hi(r)] of
// its sequence's KV pages (scale 1.0, GQA: head h reads kv head h / (nh/nkv)).
//
// It is the page's `attn::attn_prefill` -- span-02
// engine/crates/kernels/tests/gpu.rs, `run`, "prefill: all ctx rows causal":
// the same per-row attention as the decode test's reference, over every row,
// grouped by `make_tiles` / `prefill_rows_per_tile`, and bit-identical through
// the permuted pool behind a page map.
//
// One CTA serves one tile's chunk of up to 16*kBlocks query rows (row, head),
// heads fastest, for one kv head.  The KV pages of the chunk's union window
// stream through a TMA/mbarrier ring (the decode kernel's tensor maps); every
// consumer warp takes every page.  Warps form 16-query-row blocks; the kWpg
// warps of a block split the head dimension: each computes its partial
// S = Q K^T (mma.sync m16n8k16), the block exchanges and sums the partials in
// warp order, then each warp runs the online softmax and O += P V for its own
// dims.  P goes from the score accumulators to the PV A operand in registers.
#pragma once

#include "pgqa_device.cuh"

namespace pgqa {

constexpr unsigned int kErrTileRows = 8u;    // a tile longer than rows_per_tile

// Rows per tile: 128 where the tcgen05 kernel (pgqa_prefill_tc.cuh, M = 128
// query rows) serves the head dim, 32 at hd 512 where this file's mma.sync
// kernel does.

template <int HD>
struct PfCfg;
template <>
struct PfCfg<64> { static constexpr int kWpg = 1, kBlocks = 4, kStages = 8, kRowsPerTile = 128; };
template <>
struct PfCfg<128> { static constexpr int kWpg = 1, kBlocks = 4, kStages = 8, kRowsPerTile = 128; };
template <>
struct PfCfg<256> { static constexpr int kWpg = 2, kBlocks = 4, kStages = 8, kRowsPerTile = 128; };
template <>
struct PfCfg<512> { static constexpr int kWpg = 4, kBlocks = 2, kStages = 4, kRowsPerTile = 32; };

template <int HD>
struct PfGeo {
    using C = PfCfg<HD>;
    static constexpr int kWpg = C::kWpg;
    static constexpr int kBlocks = C::kBlocks;
    static constexpr int kStages = C::kStages;
    static constexpr int kConsumerWarps = kBlocks * kWpg;
    static constexpr int kConsumerThreads = kConsumerWarps * 32;
    static constexpr int kThreads = kConsumerThreads + 32;        // + one producer warp
    static constexpr int kQueryRows = kBlocks * 16;               // (row, head) pairs per CTA
    static constexpr int kDims = HD / kWpg;                       // head dims per consumer warp
    static constexpr int kKSteps = kDims / 16;                    // QK MMAs per 8 tokens
    static constexpr int kNTiles = kDims / 8;                     // PV MMAs per 16 tokens
    static constexpr int kTile = kPage * HD * 2;
    static constexpr int kStage = 2 * kTile;                      // K + V
    static constexpr int kStagesBytes = kStages * kStage;
    static constexpr int kXOff = kStagesBytes;                    // S exchange: [blocks][2][wpg][32][8] f32
    static constexpr int kXBytes = kWpg > 1 ? kBlocks * 2 * kWpg * 32 * 32 : 0;
    static constexpr int kBarOff = kXOff + kXBytes;
    static constexpr int kTotal = kBarOff + 2 * kStages * 8;
    static constexpr int kAlloc = kTotal + 1024;                  // slack for 1024-B alignment
    static_assert(kDims % 16 == 0 && kNTiles % 2 == 0, "16-dim MMA steps");
    static_assert(kAlloc <= 227 * 1024, "shared memory");
};

struct PrefillParams {
    __nv_bfloat16 *o;          // [rows][nh][hd]
    const __nv_bfloat16 *q;    // [rows][nh][hd]
    const int32_t *block_table;
    const int32_t *off;
    const int32_t *qpos;
    const int32_t *kvpos;      // may be null
    const int32_t *page_map;   // may be null
    const int32_t *tile_t0;    // [ntiles] first row of each tile
    const int32_t *tile_tn;    // [ntiles] rows of each tile
    unsigned int *err;
    int nh, nkv, g, window, rows_per_tile, whole_tile_box;
    int k_halves;              // tcgen05 kernel: K by one 5-D box per tile ([half][chunk][8][64]), else hd/64 boxes
    // split-KV (tcgen05 kernel only): with splits > 1 each (row, head) writes
    // one unnormalised partial per split -- (m, L) in log2 units into
    // part_ml[rh * splits + s] and O into part_o[(rh * splits + s) * hd] --
    // for the decode combine kernel, instead of o
    int splits;
    float *part_o;
    float2 *part_ml;
};

// Visible KV range [lo, hi] of row r (hi < lo: nothing visible).
__device__ __forceinline__ void prefill_window(const PrefillParams &p, int r, int &lo, int &hi)
{
    const int qp = __ldg(p.qpos + r);
    hi = p.kvpos ? min(qp, __ldg(p.kvpos + r)) : qp;    // causal: never past the query's own position
    lo = p.window > 0 ? max(0, qp + 1 - p.window) : 0;
}

template <int HD>
__global__ void __launch_bounds__(PfGeo<HD>::kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const PrefillParams p)
{
    using G = PfGeo<HD>;
    constexpr int NS = G::kStages;
    constexpr int WPG = G::kWpg;
    constexpr int NW = G::kConsumerWarps;
    constexpr int QR = G::kQueryRows;
    constexpr int KS = G::kKSteps;
    constexpr int NTL = G::kNTiles;
    constexpr int kChunks = HD / kBoxElems;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_full = s_base + G::kBarOff;
    const uint32_t s_empty = s_full + NS * 8;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int tile = blockIdx.x;
    const int kh = blockIdx.y;
    const int chunk = blockIdx.z;

    if (tid == 0) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(s_full + 8 * s, 1);
            mbar_init(s_empty + 8 * s, NW);
        }
        mbar_init_fence();
    }
    grid_dependency_wait();
    grid_launch_dependents();

    const int t0 = __ldg(p.tile_t0 + tile);
    const int tn = __ldg(p.tile_tn + tile);
    if (tn > p.rows_per_tile) {
        if (tid == 0)
            atomicOr(p.err, kErrTileRows);
        return;
    }
    const int g = p.g;
    const int nqr = tn * g;              // query rows of the tile
    const int qbase = chunk * QR;        // this CTA's first query row
    if (tn <= 0 || qbase >= nqr)
        return;

    // ---- union of the windows of the rows this CTA serves (positions
    // pr_first..pr_last of the tile, at most QR of them)
    const int pr_first = qbase / g;
    const int pr_last = min(tn - 1, (qbase + QR - 1) / g);
    int lo_m = INT_MAX, hi_m = INT_MIN;
    for (int pr = pr_first + lane; pr <= pr_last; pr += 32) {
        int lo, hi;
        prefill_window(p, t0 + pr, lo, hi);
        if (hi >= lo) {
            lo_m = min(lo_m, lo);
            hi_m = max(hi_m, hi);
        }
    }
#pragma unroll
    for (int k = 16; k; k >>= 1) {
        lo_m = min(lo_m, __shfl_xor_sync(0xffffffffu, lo_m, k));
        hi_m = max(hi_m, __shfl_xor_sync(0xffffffffu, hi_m, k));
    }
    int lo_u = 0, hi_u = -1;
    if (hi_m != INT_MIN) {
        lo_u = lo_m;
        hi_u = hi_m;
    }
    const int p_first = lo_u >> 4;
    const int npages = hi_u >= lo_u ? (hi_u >> 4) - p_first + 1 : 0;
    const int off0 = __ldg(p.off + t0);

    // ---- consumer set-up: the lane's two query rows (block rows gid and
    // gid + 8), their windows, and the block's union for skipping pages
    const int blk = warp / WPG;
    const int wib = warp - blk * WPG;
    const int dq0 = wib * G::kDims;
    const int gid = lane >> 2;
    const int tig = lane & 3;
    bool va = false, vb = false;
    int lo_a = 1, hi_a = 0, lo_b = 1, hi_b = 0;
    size_t rh_a = 0, rh_b = 0;
    uint32_t qa[KS][4];
    int blk_lo = INT_MAX, blk_hi = INT_MIN;
    if (warp < NW) {
        const int qra = qbase + blk * 16 + gid, qrb = qra + 8;
        if (qra < nqr) {
            const int pr = qra / g, h = qra - pr * g;
            prefill_window(p, t0 + pr, lo_a, hi_a);
            rh_a = static_cast<size_t>(t0 + pr) * p.nh + kh * g + h;
            va = true;
        }
        if (qrb < nqr) {
            const int pr = qrb / g, h = qrb - pr * g;
            prefill_window(p, t0 + pr, lo_b, hi_b);
            rh_b = static_cast<size_t>(t0 + pr) * p.nh + kh * g + h;
            vb = true;
        }
        if (va && hi_a >= lo_a) {
            blk_lo = lo_a;
            blk_hi = hi_a;
        }
        if (vb && hi_b >= lo_b) {
            blk_lo = min(blk_lo, lo_b);
            blk_hi = max(blk_hi, hi_b);
        }
#pragma unroll
        for (int k = 16; k; k >>= 1) {
            blk_lo = min(blk_lo, __shfl_xor_sync(0xffffffffu, blk_lo, k));
            blk_hi = max(blk_hi, __shfl_xor_sync(0xffffffffu, blk_hi, k));
        }
        // A fragments of Q (rows gid / gid+8, this warp's dims) straight from global memory
        const uint32_t *qga = reinterpret_cast<const uint32_t *>(p.q + rh_a * HD + dq0);
        const uint32_t *qgb = reinterpret_cast<const uint32_t *>(p.q + rh_b * HD + dq0);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qa[ks][0] = va ? __ldg(qga + ks * 8 + tig) : 0u;       // row gid, dims 16ks + 2tig, +1
            qa[ks][1] = vb ? __ldg(qgb + ks * 8 + tig) : 0u;       // row gid+8
            qa[ks][2] = va ? __ldg(qga + ks * 8 + 4 + tig) : 0u;   // row gid, dims 16ks + 8 + 2tig, +1
            qa[ks][3] = vb ? __ldg(qgb + ks * 8 + 4 + tig) : 0u;
        }
    }
    __syncthreads();                 // barriers initialised for every role

    if (warp == NW) {
        // ------------------------------------------------ producer warp
        if (lane == 0) {
            tma_prefetch_map(&tm_k);
            tma_prefetch_map(&tm_v);
        }
        const int32_t *tbl = p.block_table + off0 + p_first;
        bool ok = true;
        for (int c0 = 0; c0 < npages && ok; c0 += 32) {
            int phys = 0;
            if (c0 + lane < npages) {
                phys = __ldg(tbl + c0 + lane);
                if (p.page_map)
                    phys = __ldg(p.page_map + phys);
            }
            const int n = min(32, npages - c0);
            for (int j = 0; j < n; ++j) {
                const int ph = __shfl_sync(0xffffffffu, phys, j);
                if (lane == 0 && ok) {
                    const int i = c0 + j;
                    const int st = i % NS;
                    if (i >= NS)
                        ok = mbar_wait_bounded(s_empty + 8 * st, ((i / NS) - 1) & 1, p.err, kErrTimeoutEmpty);
                    if (ok) {
                        const uint32_t bar = s_full + 8 * st;
                        const uint32_t dk = s_base + st * G::kStage;
                        const uint32_t dv = dk + G::kTile;
                        const int t = ph * p.nkv + kh;
                        mbar_arrive_expect_tx(bar, G::kStage);
                        if (p.whole_tile_box) {
                            tma_load_4d(dk, &tm_k, bar, 0, 0, 0, t);
                            tma_load_4d(dv, &tm_v, bar, 0, 0, 0, t);
                        } else {
#pragma unroll
                            for (int c = 0; c < kChunks; ++c) {
                                tma_load_3d(dk + c * kBoxBytes, &tm_k, bar, c * kBoxElems, 0, t);
                                tma_load_3d(dv + c * kBoxBytes, &tm_v, bar, c * kBoxElems, 0, t);
                            }
                        }
                    }
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        return;
    }

    // ---------------------------------------------------- consumer warps
    float oacc[NTL][4];              // O: rows gid / gid+8, dims dq0 + 8nt + 2tig, +1
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt)
        oacc[nt][0] = oacc[nt][1] = oacc[nt][2] = oacc[nt][3] = 0.f;
    float m_a = -INFINITY, m_b = -INFINITY;   // running max of rows gid, gid+8 (log2 units)
    float l_a = 0.f, l_b = 0.f;               // this lane's share of their running sums

    const int lm_i = lane >> 3, lm_r = lane & 7;
    const int k_tok = (lm_i >> 1) * 8 + lm_r;     // K (QK B operand): (tok lo/hi) x (dims lo/hi)
    const int k_half = lm_i & 1;
    const int v_tok = (lm_i & 1) * 8 + lm_r;      // V (PV B operand, .trans): (dims lo/hi) x (tok lo/hi)
    const int v_half = lm_i >> 1;
    float4 *sx = reinterpret_cast<float4 *>(smem + G::kXOff) + blk * (2 * WPG * 32 * 2);

    bool ok = true;
    int na = 0;                      // pages this block has processed (exchange buffer parity)
    for (int i = 0; i < npages; ++i) {
        const int st = i % NS;
        if (ok)
            ok = mbar_wait_bounded(s_full + 8 * st, (i / NS) & 1, p.err, kErrTimeoutFull);
        const uint32_t sk = s_base + st * G::kStage;
        const uint32_t sv = sk + G::kTile;
        const int tok0 = (p_first + i) * kPage;
        if (tok0 <= blk_hi && tok0 + kPage - 1 >= blk_lo) {   // uniform over the block's warps
            // partial S over this warp's dims: [n-tile: tokens 0-7, 8-15][c0..c3]
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            if (ok) {
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const int d = dq0 + ks * 16 + k_half * 8;
                    uint32_t b00, b01, b10, b11;
                    ldsm_x4(sk + (d >> 6) * kBoxBytes + swz(k_tok, (d & 63) >> 3), b00, b01, b10, b11);
                    mma_bf16_16816(sc[0], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b00, b01);
                    mma_bf16_16816(sc[1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b10, b11);
                }
            }
            if (WPG > 1) {
                // full S = sum of the block's partials, in warp order
                // (buffers alternate over processed pages: a warp reuses one
                // only after the block's barrier of the page in between)
                float4 *xb = sx + (na & 1) * (WPG * 32 * 2);
                xb[(wib * 32 + lane) * 2] = make_float4(sc[0][0], sc[0][1], sc[0][2], sc[0][3]);
                xb[(wib * 32 + lane) * 2 + 1] = make_float4(sc[1][0], sc[1][1], sc[1][2], sc[1][3]);
                group_bar_sync(1 + blk, WPG * 32);
                float4 u0 = xb[lane * 2], u1 = xb[lane * 2 + 1];
#pragma unroll
                for (int w = 1; w < WPG; ++w) {
                    const float4 v0 = xb[(w * 32 + lane) * 2], v1 = xb[(w * 32 + lane) * 2 + 1];
                    u0.x += v0.x;
                    u0.y += v0.y;
                    u0.z += v0.z;
                    u0.w += v0.w;
                    u1.x += v1.x;
                    u1.y += v1.y;
                    u1.z += v1.z;
                    u1.w += v1.w;
                }
                sc[0][0] = u0.x;
                sc[0][1] = u0.y;
                sc[0][2] = u0.z;
                sc[0][3] = u0.w;
                sc[1][0] = u1.x;
                sc[1][1] = u1.y;
                sc[1][2] = u1.z;
                sc[1][3] = u1.w;
            }

            // mask to each query row's [lo, hi], scale to log2 units:
            // sc[nt][0/1] row gid, tokens 8nt + 2tig, +1; sc[nt][2/3] row gid+8
            float x[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int t = tok0 + nt * 8 + 2 * tig;
                x[nt][0] = (t >= lo_a && t <= hi_a) ? sc[nt][0] * kLog2e : -INFINITY;
                x[nt][1] = (t + 1 >= lo_a && t + 1 <= hi_a) ? sc[nt][1] * kLog2e : -INFINITY;
                x[nt][2] = (t >= lo_b && t <= hi_b) ? sc[nt][2] * kLog2e : -INFINITY;
                x[nt][3] = (t + 1 >= lo_b && t + 1 <= hi_b) ? sc[nt][3] * kLog2e : -INFINITY;
            }
            // online softmax: the 4 lanes of a quad hold a row's 16 scores
            float mxa = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
            float mxb = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
            for (int k = 1; k < 4; k <<= 1) {
                mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, k));
                mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, k));
            }
            const float mna = fmaxf(m_a, mxa), mnb = fmaxf(m_b, mxb);
            float al_a = 1.f, al_b = 1.f;
            float pr[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            if (mna != -INFINITY) {
                al_a = exp2f(m_a - mna);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    pr[nt][0] = bf16_round(exp2f(x[nt][0] - mna));
                    pr[nt][1] = bf16_round(exp2f(x[nt][1] - mna));
                }
            }
            if (mnb != -INFINITY) {
                al_b = exp2f(m_b - mnb);
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    pr[nt][2] = bf16_round(exp2f(x[nt][2] - mnb));
                    pr[nt][3] = bf16_round(exp2f(x[nt][3] - mnb));
                }
            }
            m_a = mna;
            m_b = mnb;
            l_a = __fmaf_rn(l_a, al_a, (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
            l_b = __fmaf_rn(l_b, al_b, (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]));
            if (__any_sync(0xffffffffu, al_a != 1.f || al_b != 1.f)) {
#pragma unroll
                for (int nt = 0; nt < NTL; ++nt) {
                    oacc[nt][0] *= al_a;
                    oacc[nt][1] *= al_a;
                    oacc[nt][2] *= al_b;
                    oacc[nt][3] *= al_b;
                }
            }
            // P as the PV A operand: rows gid / gid+8, tokens 2tig.. (n-tile 0), 8+2tig.. (n-tile 1)
            const uint32_t pa0 = pack_bf16x2(pr[0][0], pr[0][1]);
            const uint32_t pa1 = pack_bf16x2(pr[0][2], pr[0][3]);
            const uint32_t pa2 = pack_bf16x2(pr[1][0], pr[1][1]);
            const uint32_t pa3 = pack_bf16x2(pr[1][2], pr[1][3]);

            // V B fragments hold tokens (2tig, 2tig+1) and (8+2tig, 9+2tig);
            // on a page that reaches outside the CTA's union window, tokens
            // outside it are zeroed (their slots may hold anything, NaN
            // included, and P is 0 there)
            uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
            if (tok0 < lo_u || tok0 + kPage - 1 > hi_u) {
                const int t = tok0 + 2 * tig;
                vm0 = ((t >= lo_u && t <= hi_u) ? 0x0000ffffu : 0u) | ((t + 1 >= lo_u && t + 1 <= hi_u) ? 0xffff0000u : 0u);
                vm1 = ((t + 8 >= lo_u && t + 8 <= hi_u) ? 0x0000ffffu : 0u) |
                      ((t + 9 >= lo_u && t + 9 <= hi_u) ? 0xffff0000u : 0u);
            }
            if (ok) {
#pragma unroll
                for (int n2 = 0; n2 < NTL / 2; ++n2) {
                    const int d = dq0 + n2 * 16 + v_half * 8;
                    uint32_t b0a, b1a, b0b, b1b;
                    ldsm_x4_trans(sv + (d >> 6) * kBoxBytes + swz(v_tok, (d & 63) >> 3), b0a, b1a, b0b, b1b);
                    mma_bf16_16816(oacc[2 * n2], pa0, pa1, pa2, pa3, b0a & vm0, b1a & vm1);
                    mma_bf16_16816(oacc[2 * n2 + 1], pa0, pa1, pa2, pa3, b0b & vm0, b1b & vm1);
                }
            }
            ++na;
        }
        __syncwarp();
        if (lane == 0)
            mbar_arrive(s_empty + 8 * st);
    }

    // ---- finish: full row sums, O / l, bf16 (round to nearest)
#pragma unroll
    for (int k = 1; k < 4; k <<= 1) {
        l_a += __shfl_xor_sync(0xffffffffu, l_a, k);
        l_b += __shfl_xor_sync(0xffffffffu, l_b, k);
    }
#pragma unroll
    for (int nt = 0; nt < NTL; ++nt) {
        const int d = dq0 + nt * 8 + 2 * tig;
        if (va) {
            __nv_bfloat162 v;
            v.x = merge_finish(oacc[nt][0], l_a);
            v.y = merge_finish(oacc[nt][1], l_a);
            *reinterpret_cast<__nv_bfloat162 *>(p.o + rh_a * HD + d) = v;
        }
        if (vb) {
            __nv_bfloat162 v;
            v.x = merge_finish(oacc[nt][2], l_b);
            v.y = merge_finish(oacc[nt][3], l_b);
            *reinterpret_cast<__nv_bfloat162 *>(p.o + rh_b * HD + d) = v;
        }
    }
}

struct PrefillLaunchArgs {
    PrefillParams p;
    const CUtensorMap *tm_k;
    const CUtensorMap *tm_v;
    int ntiles;
    int max_tile_rows;    // no tile holds more rows (<= rows_per_tile): sets the chunks per tile
    int num_sms;          // persistent kernels: one CTA per SM
    cudaStream_t stream;
};

// Query-row chunks per tile: enough CTAs for the longest allowed tile.
template <int HD>
constexpr int prefill_chunks(int g)
{
    return (PfCfg<HD>::kRowsPerTile * g + PfGeo<HD>::kQueryRows - 1) / PfGeo<HD>::kQueryRows;
}

template <int HD>
cudaError_t launch_prefill(const PrefillLaunchArgs &a, bool set_attr)
{
    if (set_attr) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             PfGeo<HD>::kAlloc);
        if (e != cudaSuccess)
            return e;
    }
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.ntiles, a.p.nkv, prefill_chunks<HD>(a.p.g));
    cfg.blockDim = dim3(PfGeo<HD>::kThreads);
    cfg.dynamicSmemBytes = PfGeo<HD>::kAlloc;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prefill_kernel<HD>, *a.tm_k, *a.tm_v, a.p);
}

cudaError_t launch_prefill_hd64(const PrefillLaunchArgs &a, bool set_attr);
cudaError_t launch_prefill_hd128(const PrefillLaunchArgs &a, bool set_attr);
cudaError_t launch_prefill_hd256(const PrefillLaunchArgs &a, bool set_attr);
cudaError_t launch_prefill_hd512(const PrefillLaunchArgs &a, bool set_attr);

}  // namespace pgqa
