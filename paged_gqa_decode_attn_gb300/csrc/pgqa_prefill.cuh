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
// This header holds what the host and the tcgen05 kernel
// (pgqa_prefill_tc.cuh) share: the parameters, the rows per tile and each
// row's visible range.
#pragma once

#include "pgqa_device.cuh"

namespace pgqa {

constexpr unsigned int kErrTileRows = 8u;    // a tile longer than rows_per_tile

// Rows per tile, at every head dim: the tcgen05 kernel's M = 128 query rows
// (row, head) take a tile's rows for one kv head in ceil(rows * g / 128) chunks.
constexpr int kPrefillRowsPerTile = 128;

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
    int k_halves;              // K by one 5-D box per tile ([half][chunk][8][64]), else by 64-dim boxes
    // split-KV: with splits > 1 each (row, head) writes
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

struct PrefillLaunchArgs {
    PrefillParams p;
    const CUtensorMap *tm_k;
    const CUtensorMap *tm_v;
    const CUtensorMap *tm_q;    // Q as [rows][nh][hd], boxes of 64 dims x g heads x 128/g rows; null: no Q by TMA
    int ntiles;
    int max_tile_rows;    // no tile holds more rows (<= rows_per_tile): sets the chunks per tile
    int num_sms;          // persistent grids: one CTA per SM (pairs: as many as are resident)
    cudaStream_t stream;
};

// The tcgen05 kernel per head dim (pgqa_prefill_hd*.cu, compiled apart).
cudaError_t launch_prefill_hd64(const PrefillLaunchArgs &a, bool set_attr);
cudaError_t launch_prefill_hd128(const PrefillLaunchArgs &a, bool set_attr);
cudaError_t launch_prefill_hd256(const PrefillLaunchArgs &a, bool set_attr);
cudaError_t launch_prefill_hd512(const PrefillLaunchArgs &a, bool set_attr);
// CTA pairs of the hd-512 kernel that can be resident at once on the current device (0: none).
int prefill_pair_capacity_hd512();

}  // namespace pgqa
