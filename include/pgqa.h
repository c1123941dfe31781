/*
 * pgqa — split-KV paged GQA decode attention for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libpgqa.so.  Plain pointers and sizes only; every pointer named
 * "device" must be a CUDA device (or managed) address on the current device,
 * every other pointer is host memory.  The caller owns all buffers.
 *
 * The operation is the decode attention exercised by span-02
 * `engine/crates/kernels/tests/gpu.rs` (`attn::attn_decode`,
 * `attn::choose_splits`, `attn::decode_part_bytes` in its `run` function, and
 * the f64 `reference` function that defines the result):
 *
 *   for every query row r and head h, kv head kh = h / (nh / nkv):
 *     lo   = window > 0 ? max(0, qpos[r] + 1 - window) : 0
 *     hi   = kvpos ? min(qpos[r], kvpos[r]) : qpos[r]     (causal)
 *     o[r,h,:] = softmax_p( q[r,h,:] . K[p,kh,:] ) @ V[p,kh,:],  p in [lo, hi]
 *
 * with scale 1.0 (no 1/sqrt(hd)).  KV position p of row r is slot p % 16 of
 * physical page  phys = block_table[off[r] + p / 16]  (then
 * phys = page_map[phys] when page_map is given).  The pools are
 * [page][nkv][16][hd] bf16, so the (page, kv head) tile is 16*hd contiguous
 * elements.  A row with hi < lo has no visible position and gets zeros.
 *
 * Status codes: every function returning int returns PGQA_OK (0) or one of
 * the negative PGQA_ERR_* codes below; pgqa_strerror() names them.
 */
#ifndef PGQA_H
#define PGQA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PGQA_OK 0
#define PGQA_ERR_INVALID_ARGUMENT (-1)   /* null pointer, bad size, nh % nkv != 0, ... */
#define PGQA_ERR_UNSUPPORTED_HD (-2)     /* hd not in {64, 128, 256, 512} */
#define PGQA_ERR_MISALIGNED (-3)         /* o, part, q or a pool is not 16-byte aligned */
#define PGQA_ERR_CUDA (-4)               /* a CUDA runtime call or launch failed */
#define PGQA_ERR_TENSOR_MAP (-5)         /* the driver refused the TMA descriptor */
#define PGQA_ERR_DEVICE_TIMEOUT (-6)     /* a kernel gave up a bounded wait (see pgqa_device_status) */
#define PGQA_ERR_TOO_MANY_SPLITS (-7)    /* splits > PGQA_MAX_SPLITS */
#define PGQA_ERR_NOALLOC_TOO_LARGE (-8)  /* call needs more scratch than pgqa_attn_decode_noalloc has */
#define PGQA_ERR_TILE_TOO_LONG (-9)      /* (device) a prefill tile held more rows than rows_per_tile */

#define PGQA_PAGE_TOKENS 16
#define PGQA_MAX_SPLITS 256

/*
 * Split-KV paged decode attention (`attn::attn_decode` of the test file
 * above; the result is its f64 `reference`).
 *
 * Device buffers:
 *   o           [rows][nh][hd] bf16, written (never read), 16-byte aligned.
 *   part        scratch of at least pgqa_decode_part_bytes(rows, nh, splits, hd)
 *               bytes, 16-byte aligned; contents need no initialisation and are
 *               dead after the call.  May be NULL when splits == 1.
 *   q           [rows][nh][hd] bf16, 16-byte aligned.
 *   k_pool,
 *   v_pool      [npages][nkv][16][hd] bf16, 16-byte aligned.  Only the pages
 *               holding positions [lo, hi] of some row are read, so pages wholly
 *               outside every row's window may point anywhere, e.g. a NaN-filled
 *               null page.  Slots of a read page outside every row's [lo, hi]
 *               may hold any bits (NaN included): they never reach o.
 *   block_table int32; row r's logical page j is block_table[off[r] + j].
 *   off         [rows] int32, per-row start in block_table.
 *   qpos        [rows] int32, query position of each row (>= 0).
 *   kvpos       [rows] int32 last KV position written for each row, or NULL
 *               for kvpos = qpos.  The attention is causal, so a value past
 *               qpos[r] changes nothing; a smaller one ends the range early.
 *   counters    merge counters, NULL or at least
 *               pgqa_decode_counter_count(rows, nh, nkv) uint32 slots.  Zero
 *               them once before first use; every successful call leaves them
 *               zero again.  Non-NULL with 2 <= splits <= 8: the split
 *               partials merge inside the kernel -- on chip, through the
 *               distributed shared memory of a thread-block cluster holding a
 *               tile's splits, when splits is 2, 4 or 8 and the device can
 *               co-schedule such a cluster; otherwise in the tile's last CTA,
 *               found through the counters.  NULL, or more than 8 splits: a
 *               separate combine kernel merges them (in two levels of up to 8
 *               splits above 8), and the counters are not touched.  All give
 *               bit-identical o.
 *   page_map    int32 map from block-table entries to physical pages, or NULL.
 *
 * Host scalars: rows >= 0, nh, nkv > 0 with nh % nkv == 0, hd in
 * {64, 128, 256, 512}, window >= 0 (0 = full causal), 1 <= splits <=
 * PGQA_MAX_SPLITS.  Grid limits: rows <= 65535, nkv * ceil((nh / nkv) / 8)
 * <= 65535 and, with splits > 1, rows * nh <= INT_MAX; beyond them the call
 * returns PGQA_ERR_INVALID_ARGUMENT.  The output for a given (inputs, splits)
 * does not depend on which physical pages hold the data.
 *
 * Row packing: consecutive rows in groups of max(1, 8 / (nh / nkv)) that share
 * their block-table span (equal off) and whose visible ranges pairwise
 * overlap are served together, so their common KV is read once.  Which rows
 * pack depends only on off, qpos, kvpos and window.
 *
 * stream: a cudaStream_t (NULL = the legacy default stream).  The call only
 * enqueues work: it never synchronises and never allocates.  Calls sharing
 * `part` or `counters` must be ordered on the GPU (same stream or events).
 *
 * Ordering with the kernel before it in the stream: the kernels may start
 * while that kernel ends (programmatic dependent launch) and wait for it to
 * complete before they use any input.  A call that merges in the combine
 * kernel also reads off, qpos, kvpos, block_table and page_map before that
 * wait, through L2 only, to prefetch its first K/V pages into L2.  Those
 * reads may see values the earlier kernel is still writing; they only steer
 * the prefetch, and every index they produce is checked against the extent
 * of the allocation it points into (cuMemGetAddressRange), so nothing
 * outside the caller's allocations is touched.  Where the driver cannot size
 * an allocation (virtual-memory mappings, for example) the prefetch is off.
 */
int pgqa_attn_decode(void *o, void *part, const void *q, const void *k_pool, const void *v_pool,
                     const int32_t *block_table, const int32_t *off, const int32_t *qpos,
                     const int32_t *kvpos, int rows, int nh, int nkv, int hd, int window,
                     int splits, uint32_t *counters, const int32_t *page_map, void *stream);

/*
 * Number of KV splits per (row, kv head) tile (`attn::choose_splits` of the
 * test file; its body is not given there, this rule is this library's own).
 * kv_len_eff is the visible KV length, min(ctx, window) for sliding layers.
 * rows and nseq are the query rows and the distinct sequences among them;
 * nkv the kv heads.  Uses the current device's SM count.  Returns >= 1.
 */
int pgqa_choose_splits(int kv_len_eff, int rows, int nkv, int nseq);

/* pgqa_choose_splits for an explicit SM count (pure host arithmetic). */
int pgqa_choose_splits_for(int kv_len_eff, int rows, int nkv, int nseq, int num_sms);

/*
 * Splits per tile when the caller also knows the head count nh and head
 * dimension hd: not in the pages, whose `choose_splits` takes neither.  It
 * knows how many rows of a sequence share a CTA (max(1, 8 / (nh / nkv))), so
 * how many CTAs one split launches, and, from the current device, how many of
 * the hd kernel's CTAs and clusters can be resident at once.  With fewer tiles
 * than SMs it fills the GPU in one wave -- one CTA per SM at hd 256 and 512,
 * about 2.5 per SM at hd 64 and 128, whose CTAs are a third of an SM -- unless
 * each CTA's share of K and V stays within 16 pages and 128 KB per two query
 * rows it serves (q = min(8, rows packed per CTA x nh / nkv); 128 KB x
 * max(1, q / 2)) with
 * the largest cluster size (2, 4 or 8) whose clusters all fit, which then
 * merges on chip: the combine kernel's cost grows with the rows it merges.  With at
 * least one tile per SM it returns pgqa_choose_splits's count.  The rule was
 * fitted to measured decode times over hd, kv heads and context lengths.
 * Returns >= 1, PGQA_ERR_UNSUPPORTED_HD for another hd, or
 * PGQA_ERR_INVALID_ARGUMENT unless nh and nkv are positive with nh % nkv == 0.
 */
int pgqa_choose_splits_ex(int kv_len_eff, int rows, int nkv, int nseq, int nh, int hd);

/*
 * pgqa_choose_splits_ex for an explicit device (pure host arithmetic): its SM
 * count, the split kernel's resident CTAs per SM at hd, and how many clusters
 * of 2, 4 and 8 of them can be resident at once.
 */
int pgqa_choose_splits_ex_for(int kv_len_eff, int rows, int nkv, int nseq, int nh, int hd, int num_sms,
                              int ctas_per_sm, int clusters2, int clusters4, int clusters8);

/*
 * Bytes of the `part` scratch (`attn::decode_part_bytes` of the test file):
 * rows * nh * splits * (hd + 2) * 4 (f32 O, running max and sum per split).
 */
size_t pgqa_decode_part_bytes(int rows, int nh, int splits, int hd);

/* uint32 merge-counter slots one call needs: rows * nkv * ceil((nh / nkv) / 8), one per tile. */
size_t pgqa_decode_counter_count(int rows, int nh, int nkv);

/*
 * Kernels one pgqa_attn_decode call with rows > 0 launches: 1 (the split
 * kernel, merging in the kernel) when splits == 1, or when counters are given
 * (with_counters != 0) and splits <= 8; else 2 (plus the combine kernel).
 * 0 for splits outside [1, PGQA_MAX_SPLITS].  Pure host arithmetic.
 */
int pgqa_decode_kernel_count(int splits, int with_counters);

/*
 * Reads and clears the device-side error word of the current device
 * (synchronises the device).  Returns PGQA_OK, or PGQA_ERR_DEVICE_TIMEOUT if a
 * kernel gave up one of its bounded waits since the last read; merge counters
 * must then be zeroed again.
 */
int pgqa_device_status(void);

/*
 * Self-test of the failure path above: enqueues on `stream` one CTA that
 * waits, through the kernels' own bounded wait, on an mbarrier that nothing
 * arrives on.  After about one second of SM clock it gives up and records a
 * timeout, so the next pgqa_device_status returns PGQA_ERR_DEVICE_TIMEOUT;
 * nothing faults, traps or hangs, and later calls run normally.  Returns
 * PGQA_OK once enqueued, or PGQA_ERR_CUDA.
 */
int pgqa_selftest_bounded_wait(void *stream);

/*
 * Debug tracing.  In a library built with PGQA_TRACE defined, every split-kernel
 * CTA of later calls writes 32 uint64 slots into device_buffer: the global
 * timer (ns) at up to 16 phase boundaries in slots 0-15 and the SM cycle
 * counter at the same moments in slots 16-31, at [cta][slot] with
 * cta = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x, when
 * the buffer holds the whole grid; NULL turns it off.  Returns PGQA_OK in a
 * trace build and PGQA_ERR_INVALID_ARGUMENT (with no effect on kernels) in a
 * normal one.
 */
int pgqa_trace_buffer(void *device_buffer, size_t bytes);

/*
 * pgqa_attn_decode without caller scratch.  The pages describe no such entry
 * point; this one exists for callers that cannot allocate device memory for
 * `part` and `counters` (a plugin inside a host runtime that owns all device
 * allocations, or a caller that must not call cudaMalloc on its path).
 *
 * Same arguments and result as pgqa_attn_decode given merge counters (the
 * split kernel merges up to 8 splits, the combine kernel more), minus part
 * and counters: those live in one static device array of this
 * library (PGQA_NOALLOC_MAX_COUNTERS uint32 counters followed by
 * PGQA_NOALLOC_MAX_PART_BYTES of partials, about 8.1 MiB), which every GPU
 * that loads the library holds until the process exits.  Calls needing more
 * (pgqa_decode_part_bytes or pgqa_decode_counter_count above those limits)
 * return PGQA_ERR_NOALLOC_TOO_LARGE.  Every argument check of
 * pgqa_attn_decode runs first too, and a rejected call enqueues nothing.
 *
 * It allocates nothing.  Each call clears the counters it uses with
 * cudaMemsetAsync on `stream`, then enqueues the decode there.  The first
 * call on a device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current); make that first call before any stream capture.
 * After a device reset (cudaDeviceReset) the next call sees a new context and
 * looks the address up again, so that call, too, belongs outside a capture.
 * Every call on a device shares the one array and finds it as the previous
 * call left it, so calls that may overlap on the GPU (different streams
 * without ordering between them) race and must not be issued.
 */
#define PGQA_NOALLOC_MAX_COUNTERS 16384
#define PGQA_NOALLOC_MAX_PART_BYTES (8 * 1024 * 1024)
int pgqa_attn_decode_noalloc(void *o, const void *q, const void *k_pool, const void *v_pool,
                             const int32_t *block_table, const int32_t *off, const int32_t *qpos,
                             const int32_t *kvpos, int rows, int nh, int nkv, int hd, int window,
                             int splits, const int32_t *page_map, void *stream);

/*
 * Paged causal prefill: `attn::attn_prefill`, with `attn::make_tiles` and
 * `attn::prefill_rows_per_tile`, of span-02 engine/crates/kernels/tests/gpu.rs,
 * `run` ("prefill: all ctx rows causal").
 *
 * Every row r of the tiles, for every head h, attends exactly as a decode row
 * does (pgqa_attn_decode): scale 1.0, kv head h / (nh/nkv), the positions
 * [lo(r), min(qpos[r], kvpos[r])] with lo(r) = window > 0 ?
 * max(0, qpos[r] + 1 - window) : 0, read through
 * block_table[off[r] + pos/16] and the optional page_map.
 *   o        [rows][nh][hd] bf16, written (round to nearest), never read
 *   q        [rows][nh][hd] bf16
 *   k_pool, v_pool, block_table, off, qpos, kvpos, page_map: as for decode
 *            (kvpos may be NULL, meaning qpos; page_map may be NULL)
 *   tile_t0, tile_tn  [ntiles] int32, device: tile i is rows
 *            tile_t0[i] .. tile_t0[i] + tile_tn[i] - 1, all with the same off
 *            and at most pgqa_prefill_rows_per_tile(hd) of them (pgqa_make_tiles
 *            builds such tiles); rows not in any tile are not written
 * All buffers are caller-owned device memory; q, o and the pools must be
 * 16-byte aligned.  Asynchronous on `stream`; no host synchronisation, no
 * allocation.  Returns PGQA_OK (also for ntiles == 0) or PGQA_ERR_* for bad
 * arguments (checked before any CUDA call) or a launch failure.  A tile
 * longer than rows_per_tile is skipped and reported by pgqa_device_status as
 * PGQA_ERR_TILE_TOO_LONG.  The result does not depend on the physical page
 * ids: a permuted pool behind a page map gives the same bits.
 */
int pgqa_attn_prefill(void *o, const void *q, const void *k_pool, const void *v_pool,
                      const int32_t *block_table, const int32_t *off, const int32_t *qpos,
                      const int32_t *kvpos, const int32_t *tile_t0, const int32_t *tile_tn, int ntiles,
                      int nh, int nkv, int hd, int window, const int32_t *page_map, void *stream);

/*
 * pgqa_attn_prefill with split-KV, for tiles whose rows share a long context:
 * chunked prefill, or the multi-token decode of one sequence (speculative
 * verification), whose rows are many query rows per kv head -- more than the
 * 8 that pgqa_attn_decode packs into one CTA.  Each (tile chunk, kv head) work
 * item of the tcgen05 kernel is cut into `splits` page ranges of its window;
 * each writes an unnormalised partial (as pgqa_attn_decode's scratch holds
 * them) and the decode combine kernel merges them into o.  The result is the
 * same attention as pgqa_attn_prefill's (equal within the page's gate: the
 * sums run in another order).
 *   part   device scratch of at least pgqa_decode_part_bytes(rows, nh, splits, hd)
 *          bytes, 16-byte aligned, caller-owned (not read before written)
 *   rows   the number of rows; every row must be in exactly one tile; with
 *          splits > 1, rows * nh <= INT_MAX (else PGQA_ERR_INVALID_ARGUMENT)
 *   splits 1..PGQA_MAX_SPLITS; 1 is pgqa_attn_prefill (part unused)
 * Other arguments as for pgqa_attn_prefill.  Asynchronous on `stream`; two
 * kernels.
 */
int pgqa_attn_prefill_split(void *o, void *part, const void *q, const void *k_pool, const void *v_pool,
                            const int32_t *block_table, const int32_t *off, const int32_t *qpos,
                            const int32_t *kvpos, const int32_t *tile_t0, const int32_t *tile_tn, int ntiles,
                            int rows, int nh, int nkv, int hd, int window, int splits, const int32_t *page_map,
                            void *stream);

/*
 * A split count for pgqa_attn_prefill_split on the current device: enough
 * splits that the live work items (tiles x kv heads x 128-row chunks of
 * (row, head) pairs) fill the SMs once, at least two 64-token blocks of the
 * longest window (kv_len_eff positions) per split; at least 1.
 * PGQA_ERR_INVALID_ARGUMENT for non-positive sizes or nh % nkv != 0.
 */
int pgqa_prefill_split_count(int kv_len_eff, int rows, int ntiles, int nh, int nkv);

/*
 * pgqa_prefill_split_count with the head dimension known (no counterpart in the
 * pages).  At hd 512 a work item runs on a CTA pair, and fewer pairs than SMs
 * are resident at once: while each split keeps at most 32 64-token blocks, the
 * count is the one wave of resident pairs allows (a second wave doubled short
 * calls); otherwise, and at every other hd, it is pgqa_prefill_split_count's.
 * PGQA_ERR_UNSUPPORTED_HD for another hd, and pgqa_prefill_split_count's
 * errors.
 */
int pgqa_prefill_split_count_ex(int kv_len_eff, int rows, int ntiles, int nh, int nkv, int hd);

/* The longest tile pgqa_attn_prefill takes at head dimension hd (128 rows at
 * every supported hd), or PGQA_ERR_UNSUPPORTED_HD. */
int pgqa_prefill_rows_per_tile(int hd);

/*
 * Host-side tiling of `rows` rows (host int32 `seq[rows]`, any per-row key
 * whose changes end a tile: the sequence id or its off): consecutive rows
 * with equal keys, at most rows_per_tile per tile, in row order.  Writes
 * tile_t0/tile_tn (host arrays of max_tiles) and returns the tile count; with
 * both NULL only returns the count.  PGQA_ERR_INVALID_ARGUMENT for bad sizes
 * or too small arrays.
 */
int pgqa_make_tiles(const int32_t *seq, int rows, int rows_per_tile, int32_t *tile_t0, int32_t *tile_tn,
                    int max_tiles);

/*
 * The step before paged attention: QK-RMSNorm, rotary embedding and the paged
 * K/V write.  pegainfer PR #1002 ("reduce the duplicated CPU operator oracles
 * in the HD256/HD512 QK-RoPE smokes") describes this step's device gates --
 * RMSNorm and RoPE of head vectors, rotation over the first rotary_dim dims
 * ("rope-lo", "rope-hi") with the rest passed through, K and V landing at the
 * paged-KV layout address -- but prints no formula; this is the plainest
 * reading.  For every row r and head vector x (hd dims, bf16):
 *   RMSNorm  y_d = x_d / sqrt(mean(x^2) + eps) * w_d   (Q: q_weight, K: k_weight;
 *            V: no weight when norm_v, else copied unchanged)
 *   RoPE     (Q and K) half = rotary_dim / 2, for i < half,
 *            a = pos[r] * theta^(-2i / rotary_dim):
 *            y_i <- y_i cos a - y_{i+half} sin a,  y_{i+half} <- y_{i+half} cos a + y_i sin a
 *   output   q_out[r][h][:]; K and V of kv head kh at element
 *            ((page * nkv + kh) * 16 + pos[r] % 16) * hd of k_pool / v_pool,
 *            page = block_table[off[r] + pos[r] / 16] (then page_map[page] when given)
 * Computed in f32, stored bf16 (round to nearest); the angle is carried in
 * turns from an f64 frequency, so it stays within ~1e-6 rad at any position.
 *   q_in [rows][nh][hd], k_in / v_in [rows][nkv][hd], q_weight / k_weight [hd]: bf16
 *   q_out [rows][nh][hd] bf16, written; k_pool / v_pool: only the rows' slots written
 *   pos, off [rows], block_table, page_map (may be NULL): int32, device;
 *            0 <= pos[r] < 2^24 and every looked-up entry in range (not checked)
 * hd is 64, 128, 256 or 512; rotary_dim in [0, hd], a multiple of hd / 16;
 * theta > 0, eps >= 0.  Device buffers are caller-owned and 16-byte aligned.
 * Asynchronous on `stream`; no allocation.  Returns PGQA_OK or PGQA_ERR_* for
 * bad arguments (checked before any CUDA call) or a launch failure.
 */
int pgqa_qk_norm_rope_write(void *q_out, void *k_pool, void *v_pool, const void *q_in, const void *k_in,
                            const void *v_in, const void *q_weight, const void *k_weight, const int32_t *pos,
                            const int32_t *block_table, const int32_t *off, const int32_t *page_map, int rows,
                            int nh, int nkv, int hd, int rotary_dim, float theta, float eps, int norm_v,
                            void *stream);

/* Static, human-readable name of a status code. */
const char *pgqa_strerror(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int pgqa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PGQA_H */
