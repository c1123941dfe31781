// Paged causal prefill on the 5th-generation tensor cores (tcgen05) of GB300,
// for head dims 64, 128, 256 and 512 (the page's `attn::attn_prefill`: every
// tile row attends like a decode row at its position), computed as a
// flash-attention loop with the accumulators in tensor memory:
//
//   * one CTA serves 128 query rows (row, head) of one tile and kv head --
//     the M = 128 of every MMA -- with heads fastest; their Q sits in tensor
//     memory (the A operand of S), which leaves 192 KB of shared memory to
//     the K/V ring (128 KB beside the S exchange buffers at hd 512);
//   * warp 16 streams the chunk's union window in blocks of 4 pages (64
//     tokens) by TMA into that ring, page ids read 32 at a time ahead of the
//     copies, one box per (page, kv head) tile each: K in a 5-D view that
//     lands as [2 halves][hd/64][8 tokens][128 B], so one chunk's 8-token
//     swizzle atoms sit hd * 16 bytes apart over the block's 4 pages and one
//     N = 64 MMA per 16 dims reads them (per-page 64-dim boxes, four times as
//     many copies, where the driver refuses the view); V as
//     [hd/64][16 tokens][128 B]; a stage's K and V have barriers of their
//     own, so K_{j+NST} streams in as soon as S_j is done;
//   * warp 17 issues S_j = Q K_j^T into one of two TMEM buffers (64 columns
//     each) and warp 19 O += P_j V_j (TMEM, a column per head dim of the CTA,
//     one MMA per page), each batch committed to mbarriers;
//   * warp 18 computes the work items ahead and publishes them;
//   * at hd 512, where O of 128 rows would fill all of tensor memory, a pair
//     of CTAs (a cluster of two) serves each item, each CTA over half of the
//     head dims of Q, K, V and O: both compute their half of S_j, swap the
//     halves through distributed shared memory (st.async, one mbarrier per
//     buffer) and add them, so both run the same softmax on the same S_j;
//   * warps 0-15 run the softmax, four threads per query row (warps w, w+4,
//     w+8, w+12 share TMEM lanes 32(w%4)..: lane = row), each over a quarter
//     of the block's columns: they read S_j from TMEM, mask it to the row's
//     window, agree on the row max through shared memory, run the online
//     softmax in log2 units, rescale their quarter of O in TMEM only when the
//     row's running max grows by more than 2^8 (exact in real arithmetic: P
//     then stays below 256), write their quarter of P_j as bf16 (the A
//     operand of the PV MMA), and at the end divide their quarter of O by the
//     row sum and store bf16 -- or, split-KV, the unnormalised partial;
//   * P_j goes into the first half of S_j's own TMEM buffer, the PV MMA's A
//     operand: the buffer takes S_{j+2} once PV_j is done, and P_j waits for
//     no PV (a single shared-memory P buffer had to wait for PV_{j-1}).
//
// Every wait is bounded; a thread that gives up skips its later waits and
// every role still reaches the final barrier, which frees the tensor memory.
#pragma once

#include <algorithm>
#include <climits>

#include "pgqa_prefill.cuh"

namespace pgqa {

// ---------------------------------------------------------------- tcgen05 helpers

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets, the fixed 0b001 at bits 46-48, 128-byte swizzle (mode 2, bits 61-63).
__device__ __forceinline__ uint64_t umma_sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// Instruction descriptor of kind::f16: f32 accumulate, bf16 A and B, A / B
// K-major (0) or MN-major (1), N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t umma_idesc_bf16(int m, int n, int a_mn, int b_mn)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
           (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(n >> 3) << 17) |
           (static_cast<uint32_t>(m >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// The same with A in tensor memory: row m in lane m, its K elements two to a
// 32-bit column (the lower-indexed one in the low half).
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                 uint32_t acc)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
        : "memory");
}

// Arrive once on `bar` when every tcgen05.mma this thread issued so far is complete.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

template <int kCols>
__device__ __forceinline__ void tmem_alloc(uint32_t slot)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot), "n"(kCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

template <int kCols>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(kCols) : "memory");
}

// 32 lanes x 16 consecutive 32-bit columns: thread t gets lane (warp's base + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
                 : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void fence_async_shared() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// 2^x by the SFU's approximation (relative error about 2^-22; 2^-inf = +0):
// one instruction per score, whose result is rounded to bf16 for P anyway.
__device__ __forceinline__ float ex2_sfu(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// L2 prefetches (hints: nothing is written, nothing waits): a contiguous
// range of `bytes` (16-byte aligned and sized), and one TMA box of a tensor map.
__device__ __forceinline__ void l2_prefetch_bytes(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(src)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void l2_prefetch_box_3d(const CUtensorMap *map, int x, int y, int z)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void l2_prefetch_box_4d(const CUtensorMap *map, int x, int y, int z, int w)
{
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

__device__ __forceinline__ void l2_prefetch_box_5d(const CUtensorMap *map, int c, int t)
{
    asm volatile("cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %1, %2, %1, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(0), "r"(c), "r"(t)
                 : "memory");
}

// One TMA box of a 5-D tensor map at (0, 0, c, 0, t): the (page, kv head)
// tile t in the halves view, from 64-dim chunk c on (the box's chunk count).
__device__ __forceinline__ void tma_load_5d_tile(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c, int t)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %3, %4, %3, %5}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(0), "r"(c), "r"(t)
        : "memory");
}

// A CTA pair: this CTA's rank in its cluster, and the cluster barrier's
// arrive with release semantics.
__device__ __forceinline__ int cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return static_cast<int>(r);
}

__device__ __forceinline__ void cluster_arrive_release() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }

// Non-blocking test of an mbarrier phase (try_wait may suspend the thread for
// a while before it answers, which would hold up a poller watching two barriers).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// 32 bytes to global memory in one instruction (a whole L2 sector); dst must be
// 32-byte aligned.
__device__ __forceinline__ void st_global_32B(void *dst, const uint32_t (&w)[8])
{
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(reinterpret_cast<uint64_t>(dst)),
                 "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// ---------------------------------------------------------------- geometry

template <int HD>
struct TcGeo {
    // hd 512: O of 128 rows would fill all of tensor memory, so a pair of CTAs
    // (a cluster of two) serves each item, each CTA over half of the head
    // dims, and they add their halves of S through distributed shared memory
    static constexpr bool kSplitDims = HD > 256;
    static constexpr int kHdc = kSplitDims ? HD / 2 : HD;     // head dims per CTA
    static constexpr int kRows = 128;                  // query rows per CTA (MMA M)
    static constexpr int kBlockPages = 4;
    static constexpr int kBlockTokens = kBlockPages * kPage;   // 64: S columns per block
    static constexpr int kChunks = kHdc / 64;          // 128-byte swizzle rows per head vector (this CTA's dims)
    static constexpr int kKBytes = kChunks * kBlockTokens * 128;           // [chunk][64 tokens][128 B]
    static constexpr int kVPage = kChunks * kPage * 128;                   // [chunk][16 tokens][128 B]
    static constexpr int kVBytes = kBlockPages * kVPage;
    static constexpr int kStageBytes = kKBytes + kVBytes;
    // 192 KB of K/V in flight; 128 KB beside the S exchange buffers of a pair
    static constexpr int kStages = ((kSplitDims ? 128 : 192) * 1024) / kStageBytes;
    static constexpr int kStageOff = 0;
    static constexpr int kSoftmaxWarps = 16;           // four threads per query row
    static constexpr int kParts = kSoftmaxWarps / 4;   // threads per row, each over 1/kParts of the columns
    static constexpr int kXOff = kStageOff + kStages * kStageBytes;   // row max [2][parts][128], row sum [parts][128]
    // the scheduler's published items: [2] TcItem, then [2][kRows] int2 row windows
    static constexpr int kInfoOff = kXOff + (2 * kParts * kRows + kParts * kRows) * 4;
    static constexpr int kInfoBytes = 2 * 64;          // two slots of kItemSlot bytes
    static constexpr int kWinOff = kInfoOff + kInfoBytes;
    // split dims: the peer's half of S_j, [2 buffers][parts][4][kRows] float4
    // (a thread's 16 columns as 4 float4, rows adjacent)
    static constexpr int kSxOff = kWinOff + 2 * kRows * 8;
    static constexpr int kSxBytes = kSplitDims ? 2 * kRows * kBlockTokens * 4 : 0;
    static constexpr int kBarOff = kSxOff + kSxBytes;
    // k_full[stages], k_empty[stages], v_full[stages], v_empty[stages], s_full[2], s_free[2],
    // p_full[2], o_done, q_ready, o_free, info_full[2], info_empty[2], o_item, then (split dims) x_full[2]
    static constexpr int kBars = 4 * kStages + 14 + (kSplitDims ? 2 : 0);
    static constexpr int kSlotOff = kBarOff + kBars * 8;
    static constexpr int kTotal = kSlotOff + 16;
    static constexpr int kAlloc = kTotal + 1024;
    static constexpr int kProducerWarp = kSoftmaxWarps;
    static constexpr int kMmaWarp = kSoftmaxWarps + 1;
    static constexpr int kSchedWarp = kSoftmaxWarps + 2;
    static constexpr int kPvWarp = kSoftmaxWarps + 3;
    static constexpr int kThreads = (kSoftmaxWarps + 4) * 32;   // + producer, S issuer, scheduler, PV issuer
    static constexpr int kTmemCols = kHdc == 64 ? 256 : 512;   // S0, S1, O (dims), Q (dims / 2)
    static constexpr int kOCol = 2 * kBlockTokens;
    static constexpr int kQCol = kOCol + kHdc;
    static_assert(kQCol + kHdc / 2 <= kTmemCols, "tensor memory");
    static_assert(kAlloc <= 227 * 1024, "shared memory");
    static_assert(kStageBytes % 1024 == 0, "swizzle atoms");
};

// One work item: the 128 query rows of chunk `chunk` of tile `tile` for kv
// head `kh`, and the union window of their positions.  The scheduler warp
// computes each item once and publishes it, with every query row's window,
// through shared memory.
struct TcItem {
    int t0, tn, kh, qbase, lo_u, hi_u, p_first, npages, nblocks, off0, split;
    bool live;     // the chunk has rows
    bool qslot;    // the chunk's Q comes by TMA through a ring stage ahead of its blocks
};
constexpr int kItemSlot = 64;     // bytes of one published item in shared memory
static_assert(sizeof(TcItem) <= kItemSlot && kItemSlot % 16 == 0, "published item slot");

// Item `it` (by one whole warp, four query rows per lane), and the visible
// range (lo, hi) of each of its 128 query rows into win[] ((1, 0): no row).
template <int HD, bool kQTma>
__device__ __forceinline__ TcItem tc_item_rows(const PrefillParams &p, int it, int ntiles, int nchunks, int lane,
                                               int2 *win)
{
    using G = TcGeo<HD>;
    TcItem I;
    // tiles outermost, last tiles first (they hold the longest windows), then
    // kv head, then chunk, then split
    const int S = p.splits;
    I.split = it % S;
    it /= S;
    const int per_tile = p.nkv * nchunks;
    const int tile = ntiles - 1 - it / per_tile;
    const int rest = it - (it / per_tile) * per_tile;
    I.kh = rest / nchunks;
    const int chunk = rest - I.kh * nchunks;
    I.t0 = __ldg(p.tile_t0 + tile);
    I.tn = __ldg(p.tile_tn + tile);
    I.qbase = chunk * G::kRows;
    I.live = false;
    I.lo_u = 0;
    I.hi_u = -1;
    I.p_first = 0;
    I.npages = 0;
    I.nblocks = 0;
    I.off0 = 0;
    I.qslot = false;
    const bool too_long = I.tn > p.rows_per_tile;
    if (too_long && lane == 0)
        atomicOr(p.err, kErrTileRows);
    const int g = p.g;
    const int nqr = too_long ? 0 : I.tn * g;
    int lo_m = INT_MAX, hi_m = INT_MIN;
#pragma unroll
    for (int k = 0; k < G::kRows / 32; ++k) {
        const int r = lane + 32 * k;
        const int qr = I.qbase + r;
        int lo = 1, hi = 0;
        if (qr < nqr)
            prefill_window(p, I.t0 + qr / g, lo, hi);
        win[r] = make_int2(lo, hi);
        if (hi >= lo) {
            lo_m = min(lo_m, lo);
            hi_m = max(hi_m, hi);
        }
    }
    if (I.tn <= 0 || I.qbase >= nqr)
        return I;
    I.live = true;
#pragma unroll
    for (int k = 16; k; k >>= 1) {
        lo_m = min(lo_m, __shfl_xor_sync(0xffffffffu, lo_m, k));
        hi_m = max(hi_m, __shfl_xor_sync(0xffffffffu, hi_m, k));
    }
    if (hi_m != INT_MIN) {
        I.lo_u = lo_m;
        I.hi_u = hi_m;
    }
    I.p_first = I.lo_u >> 4;
    I.npages = I.hi_u >= I.lo_u ? (I.hi_u >> 4) - I.p_first + 1 : 0;
    if (S > 1) {       // this split's share of the window's pages, in whole blocks
        const int nb = (I.npages + G::kBlockPages - 1) / G::kBlockPages;
        const int per = (nb + S - 1) / S * G::kBlockPages;
        const int first = I.split * per;
        I.p_first += first;
        I.npages = max(0, min(per, I.npages - first));
    }
    I.nblocks = (I.npages + G::kBlockPages - 1) / G::kBlockPages;
    I.off0 = __ldg(p.off + I.t0);
    // Q through the ring: its 128 rows are whole positions of the tile (g
    // divides 128 wherever the kernel takes this path), so one box per 64
    // dims reads nothing past the tile
    I.qslot = kQTma && I.nblocks > 0 && I.qbase + G::kRows <= nqr;
    return I;
}

// L2 prefetch, by one warp, of an item's Q rows (every head of its kv head, a
// superset of the chunk's) and of the K and V tiles of its first
// kPrefetchPages pages.
template <int HD>
__device__ __forceinline__ void tc_prefetch_item(const PrefillParams &p, const TcItem &I, const CUtensorMap *tm_k,
                                                 const CUtensorMap *tm_v, int dofs, int lane)
{
    using G = TcGeo<HD>;
    constexpr int kPrefetchPages = 2 * G::kBlockPages;
    if (!I.live || I.nblocks == 0)
        return;
    const int g = p.g;
    const int pr_first = I.qbase / g;
    const int pr_last = min(I.tn - 1, (I.qbase + G::kRows - 1) / g);
    for (int pr = pr_first + lane; pr <= pr_last; pr += 32)
        l2_prefetch_bytes(p.q + (static_cast<size_t>(I.t0 + pr) * p.nh + I.kh * g) * HD,
                          static_cast<uint32_t>(g * HD * 2));
    if (lane < min(kPrefetchPages, I.npages)) {
        int phys = __ldg(p.block_table + I.off0 + I.p_first + lane);
        if (p.page_map)
            phys = __ldg(p.page_map + phys);
        const int t = phys * p.nkv + I.kh;
        if (p.k_halves) {
            l2_prefetch_box_5d(tm_k, dofs / kBoxElems, t);
        } else {
#pragma unroll
            for (int c = 0; c < G::kChunks; ++c)
                l2_prefetch_box_3d(tm_k, dofs + c * kBoxElems, 0, t);
        }
        if (p.whole_tile_box) {
            l2_prefetch_box_4d(tm_v, 0, 0, dofs / kBoxElems, t);
        } else {
#pragma unroll
            for (int c = 0; c < G::kChunks; ++c)
                l2_prefetch_box_3d(tm_v, dofs + c * kBoxElems, 0, t);
        }
    }
}

// Persistent: in round k CTA c serves item k G + c (k even) or k G + G - 1 - c
// (k odd) of the ntiles * nkv * nchunks items, G = gridDim.x: with the items
// in roughly falling size, the snake pairs long items with short ones.  The ring, the S buffers and the mbarrier phases run on
// counters that continue across items, so the next item's K/V stream in
// while the current one finishes, and its Q goes into tensor memory (after
// the current item's last S) before the current item's O is read out.
// kQTma: a chunk whose 128 rows are whole positions of its tile takes its Q
// by TMA (tm_q: a [rows][nh][hd] view with boxes of 64 dims x g heads x
// 128 / g positions) into a ring stage ahead of its blocks, instead of by
// loads from every softmax thread when the item starts.
template <int HD, bool kQTma>
__global__ void __launch_bounds__(TcGeo<HD>::kThreads, 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                      const __grid_constant__ CUtensorMap tm_q, const PrefillParams p, int ntiles, int nchunks)
{
    using G = TcGeo<HD>;
    constexpr int NST = G::kStages;
    constexpr int NCH = G::kChunks;
    constexpr int HDC = G::kHdc;                       // head dims of this CTA
    constexpr bool kSplit = G::kSplitDims;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_bar = s_base + G::kBarOff;
    // a stage's K and V halves fill and free apart: K is free once its S
    // batch is done, about a block before the PV batch frees V
    const uint32_t b_kfull = s_bar;                    // [NST]
    const uint32_t b_kempty = s_bar + 8 * NST;         // [NST]
    const uint32_t b_vfull = s_bar + 16 * NST;         // [NST]
    const uint32_t b_vempty = s_bar + 24 * NST;        // [NST]
    const uint32_t b_sfull = s_bar + 32 * NST;         // [2]
    const uint32_t b_sfree = b_sfull + 16;             // [2]
    // P_j is in S_j's buffer: one p_full per buffer.  A softmax warp that runs a
    // block ahead of the others (nothing holds it to PV_{j-1}) then arrives on
    // the other buffer's barrier; it reaches this one again (block j + 2) only
    // after S_{j+2}, so after PV_j has taken this phase.
    const uint32_t b_pfull = b_sfree + 16;             // [2]
    const uint32_t b_odone = b_pfull + 16;
    const uint32_t b_qready = b_odone + 8;
    const uint32_t b_ofree = b_qready + 8;
    const uint32_t b_ifull = b_ofree + 8;              // [2] a published item is in its slot
    const uint32_t b_iempty = b_ifull + 16;            // [2] every role has read it
    // an item's last PV batch is done (one phase per item with blocks): the
    // read-out of O waits on it.  o_done, a phase per block, cannot serve: by
    // then it may be one phase past the item, and a parity wait would alias.
    const uint32_t b_oitem = b_iempty + 16;
    const uint32_t b_xfull = b_oitem + 8;              // [2] split dims: the peer's half of S_j is here
    const int2 *win = reinterpret_cast<const int2 *>(smem + G::kWinOff);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + G::kSlotOff);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // split dims: the pair is one scheduling unit; rank r takes dims [r HDC, (r + 1) HDC)
    const int crank = kSplit ? cluster_ctarank() : 0;
    const int dofs = crank * HDC;
    const int nitems = ntiles * p.nkv * nchunks * p.splits;
    const int ncta = kSplit ? gridDim.x / 2 : gridDim.x;
    const int cta = kSplit ? blockIdx.x / 2 : blockIdx.x;
    auto first_item = [&](int) { return cta < nitems ? cta : nitems; };
    // the item after `it` (round k = it / ncta) for this CTA, or nitems
    auto next_item = [&](int it) {
        for (int k = it / ncta + 1; k * ncta < nitems; ++k) {
            const int n = k * ncta + ((k & 1) ? ncta - 1 - cta : cta);
            if (n < nitems)
                return n;
        }
        return nitems;
    };

    if (tid == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(b_kfull + 8 * s, 1);
            mbar_init(b_kempty + 8 * s, 1);
            mbar_init(b_vfull + 8 * s, 1);
            mbar_init(b_vempty + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(b_sfull + 8 * b, 1);
            mbar_init(b_sfree + 8 * b, 1);          // PV_j's commit: S_j and P_j read
        }
        for (int b = 0; b < 2; ++b)
            mbar_init(b_pfull + 8 * b, G::kSoftmaxWarps);
        mbar_init(b_odone, 1);
        mbar_init(b_oitem, 1);
        mbar_init(b_qready, G::kSoftmaxWarps);
        mbar_init(b_ofree, G::kSoftmaxWarps);
        for (int b = 0; b < 2; ++b) {
            mbar_init(b_ifull + 8 * b, 1);
            mbar_init(b_iempty + 8 * b, G::kSoftmaxWarps + 3);   // softmax warps, producer, S and PV issuers
        }
        if (kSplit) {
            // each phase: the peer's 128 x 64 f32 half of one S block; the next
            // phase is armed by thread 0 as soon as it has seen this one
            for (int b = 0; b < 2; ++b) {
                mbar_init(b_xfull + 8 * b, 1);
                mbar_arrive_expect_tx(b_xfull + 8 * b, G::kRows * G::kBlockTokens * 4);
            }
        }
        mbar_init_fence();
    }
    // split dims: the peer's barriers are set up before anything is sent to them
    if (kSplit)
        cluster_arrive_relaxed();
    grid_dependency_wait();
    grid_launch_dependents();
    if (warp == 0)
        tmem_alloc<G::kTmemCols>(smem_u32(tslot));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (kSplit)
        cluster_wait();
    const uint32_t tbase = *tslot;
    // The k-th item of this CTA, published by the scheduler in slot k % 2;
    // the reading warp takes a copy and frees the slot (one arrival per warp).
    bool iok = true;
    auto take_item = [&](int k) {
        const int sl = k & 1;
        if (iok)
            iok = mbar_wait_bounded(b_ifull + 8 * sl, (k >> 1) & 1, p.err, kErrTimeoutFull);
        const TcItem I = *reinterpret_cast<const TcItem *>(smem + G::kInfoOff + sl * kItemSlot);
        return I;
    };
    auto release_item = [&](int k) {
        __syncwarp();
        if (lane == 0)
            mbar_arrive(b_iempty + 8 * (k & 1));
    };

    if (warp == G::kSchedWarp) {
        // ------------------------------------------------ scheduler: items ahead of time
        // Each item's metadata and row windows take a few dependent global
        // loads; computed here, up to two items ahead, no other role waits for
        // them at an item's start.  Each published item's Q rows and first
        // K/V pages are also prefetched into L2: items of all CTAs end about
        // together, and their first loads would otherwise meet in one burst.
        int kit = 0;
        for (int it = first_item(0); it < nitems; it = next_item(it), ++kit) {
            const int sl = kit & 1;
            if (kit >= 2 && lane == 0 && iok)
                iok = mbar_wait_bounded(b_iempty + 8 * sl, ((kit >> 1) - 1) & 1, p.err, kErrTimeoutEmpty);
            __syncwarp();
            int2 *w = reinterpret_cast<int2 *>(smem + G::kWinOff) + sl * G::kRows;
            const TcItem I = tc_item_rows<HD, kQTma>(p, it, ntiles, nchunks, lane, w);
            if (lane == 0)
                *reinterpret_cast<TcItem *>(smem + G::kInfoOff + sl * kItemSlot) = I;
            __syncwarp();
            if (lane == 0)
                mbar_arrive(b_ifull + 8 * sl);
            tc_prefetch_item<HD>(p, I, &tm_k, &tm_v, dofs, lane);
        }
    } else if (warp == G::kProducerWarp) {
        // ------------------------------------------------ producer: blocks of 4 pages
        if (lane == 0) {
            tma_prefetch_map(&tm_k);
            tma_prefetch_map(&tm_v);
            if (kQTma)
                tma_prefetch_map(&tm_q);
        }
        bool ok = true;
        int js = 0;                                    // ring slots filled (Q tiles and blocks), over all items
        int kit = 0;
        for (int it = first_item(0); it < nitems; it = next_item(it), ++kit) {
            const TcItem I = take_item(kit);
            release_item(kit);
            if (!I.live || I.nblocks == 0)
                continue;
            if (kQTma && I.qslot) {
                // the chunk's Q, [hd/64][128 rows][128 B] under the 128-byte
                // swizzle, takes a whole stage ahead of its blocks; V's barrier
                // passes the slot with a bare arrival
                const int st = js % NST;
                if (lane == 0 && ok && js >= NST) {
                    ok = mbar_wait_bounded(b_kempty + 8 * st, ((js / NST) - 1) & 1, p.err, kErrTimeoutEmpty);
                    if (ok)
                        ok = mbar_wait_bounded(b_vempty + 8 * st, ((js / NST) - 1) & 1, p.err, kErrTimeoutEmpty);
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (ok && lane == 0) {
                    const uint32_t sQ = s_base + G::kStageOff + st * G::kStageBytes;
                    mbar_arrive_expect_tx(b_kfull + 8 * st, G::kStageBytes);
#pragma unroll
                    for (int c = 0; c < NCH; ++c)
                        tma_load_3d(sQ + c * (G::kRows * 128), &tm_q, b_kfull + 8 * st, dofs + c * kBoxElems,
                                    I.kh * p.g, I.t0 + I.qbase / p.g);
                    mbar_arrive(b_vfull + 8 * st);
                }
                ++js;
            }
            const int32_t *tbl = p.block_table + I.off0 + I.p_first;
            for (int c0 = 0; c0 < I.npages; c0 += 32) {       // 32 is a multiple of the block's pages
                int phys = 0;
                if (c0 + lane < I.npages) {
                    phys = __ldg(tbl + c0 + lane);
                    if (p.page_map)
                        phys = __ldg(p.page_map + phys);
                }
                const int nc = min(32, I.npages - c0);
                for (int i = 0; i < nc; i += G::kBlockPages, ++js) {
                    const int np = min(G::kBlockPages, nc - i);
                    const int st = js % NST;
                    const uint32_t sK = s_base + G::kStageOff + st * G::kStageBytes;
                    const uint32_t sV = sK + G::kKBytes;
                    const uint32_t half_tx = np * kPage * HDC * 2;
                    // K of this block, once the slot's last use is released (its S batch)
                    if (lane == 0 && ok && js >= NST)
                        ok = mbar_wait_bounded(b_kempty + 8 * st, ((js / NST) - 1) & 1, p.err, kErrTimeoutEmpty);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (ok && lane == 0)
                        mbar_arrive_expect_tx(b_kfull + 8 * st, half_tx);
                    for (int pp = 0; pp < G::kBlockPages; ++pp) {
                        const int ph = __shfl_sync(0xffffffffu, phys, (i + pp) & 31);
                        if (ok && lane == 0 && pp < np) {
                            const int t = ph * p.nkv + I.kh;
                            if (p.k_halves) {      // one box: [half][chunk][8 slots][128 B] per page
                                tma_load_5d_tile(sK + pp * G::kVPage, &tm_k, b_kfull + 8 * st, dofs / kBoxElems, t);
                            } else {               // [chunk][64 tokens][128 B]
#pragma unroll
                                for (int c = 0; c < NCH; ++c)
                                    tma_load_3d(sK + c * (G::kBlockTokens * 128) + pp * (kPage * 128), &tm_k,
                                                b_kfull + 8 * st, dofs + c * kBoxElems, 0, t);
                            }
                        }
                    }
                    // V of this block, once the slot's last use is released (its PV batch)
                    if (lane == 0 && ok && js >= NST)
                        ok = mbar_wait_bounded(b_vempty + 8 * st, ((js / NST) - 1) & 1, p.err, kErrTimeoutEmpty);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (ok && lane == 0)
                        mbar_arrive_expect_tx(b_vfull + 8 * st, half_tx);
                    for (int pp = 0; pp < G::kBlockPages; ++pp) {
                        const int ph = __shfl_sync(0xffffffffu, phys, (i + pp) & 31);
                        if (ok && lane == 0 && pp < np) {
                            const int t = ph * p.nkv + I.kh;
                            if (p.whole_tile_box) {
                                tma_load_4d(sV + pp * G::kVPage, &tm_v, b_vfull + 8 * st, 0, 0, dofs / kBoxElems, t);
                            } else {
#pragma unroll
                                for (int c = 0; c < NCH; ++c)
                                    tma_load_3d(sV + pp * G::kVPage + c * (kPage * 128), &tm_v, b_vfull + 8 * st,
                                                dofs + c * kBoxElems, 0, t);
                            }
                        }
                    }
                }
            }
        }
    } else if (warp == G::kMmaWarp) {
        // ------------------------------------------------ S issuer (one thread)
        // The S and PV batches come from two threads of two warps: issuing an
        // MMA batch takes the issuing thread a good fraction of a microsecond,
        // and with one thread PV_j waited for the S batch in its way.  Their
        // MMAs touch disjoint tensor memory (S buffers, O) and meet only
        // through the barriers below.
        constexpr uint32_t kIdS = umma_idesc_bf16(128, G::kBlockTokens, 0, 0);
        // K of a block as the B operand (64 token rows, K-major): in the
        // halves layout a chunk's 8-row swizzle atoms are 1 KB into each
        // (page, half) and hd * 16 bytes apart; in the chunk layout they are
        // contiguous, 1 KB apart, within the chunk's 8 KB
        const uint32_t k_chunk = p.k_halves ? 1024u : static_cast<uint32_t>(G::kBlockTokens * 128);
        const uint32_t k_sbo = p.k_halves ? static_cast<uint32_t>(NCH * 1024) : 1024u;
        bool ok = true;
        int jg = 0, kq = 0;                            // blocks and items with blocks, over all items
        int qs = 0;                                    // Q tiles that came through the ring
        int kit = 0;
        for (int it = first_item(0); it < nitems; it = next_item(it), ++kit) {
            const TcItem I = take_item(kit);
            release_item(kit);
            if (!I.live || I.nblocks == 0)
                continue;
            if (kQTma && I.qslot)
                ++qs;
            if (lane == 0) {
                if (ok)
                    ok = mbar_wait_bounded(b_qready, kq & 1, p.err, kErrTimeoutFull);
                tc_fence_after();
                for (int j = 0; j < I.nblocks; ++j) {
                    const int jj = jg + j, js = jj + qs;    // block and ring slot
                    const int st = js % NST, b = jj & 1;
                    if (ok)
                        ok = mbar_wait_bounded(b_kfull + 8 * st, (js / NST) & 1, p.err, kErrTimeoutFull);
                    if (ok && jj >= 2)
                        ok = mbar_wait_bounded(b_sfree + 8 * b, ((jj - 2) >> 1) & 1, p.err, kErrTimeoutFull);
                    tc_fence_after();
                    if (ok) {
                        const uint32_t sK = s_base + G::kStageOff + st * G::kStageBytes;
#pragma unroll
                        for (int ks = 0; ks < HDC / 16; ++ks) {
                            const int c = ks >> 2, kk = ks & 3;
                            umma_bf16_tmem_a(tbase + b * G::kBlockTokens, tbase + G::kQCol + ks * 8,
                                             umma_sdesc(sK + c * k_chunk + kk * 32, 16, k_sbo), kIdS, ks > 0);
                        }
                    }
                    umma_commit(b_sfull + 8 * b);
                    umma_commit(b_kempty + 8 * st);
                }
            }
            __syncwarp();
            jg += I.nblocks;
            ++kq;
        }
    } else if (warp == G::kPvWarp) {
        // ------------------------------------------------ PV issuer (one thread)
        constexpr uint32_t kIdO = umma_idesc_bf16(128, HDC, 0, 1);
        bool ok = true;
        int jg = 0, kq = 0, qs = 0;
        int kit = 0;
        for (int it = first_item(0); it < nitems; it = next_item(it), ++kit) {
            const TcItem I = take_item(kit);
            release_item(kit);
            if (!I.live || I.nblocks == 0)
                continue;
            if (kQTma && I.qslot)
                ++qs;
            if (lane == 0) {
                for (int j = 0; j < I.nblocks; ++j) {
                    const int jj = jg + j, js = jj + qs, st = js % NST;
                    if (ok)
                        ok = mbar_wait_bounded(b_pfull + 8 * (jj & 1), (jj >> 1) & 1, p.err, kErrTimeoutFull);
                    if (ok && j == 0 && kq >= 1)            // the previous item's O has been read out
                        ok = mbar_wait_bounded(b_ofree, (kq - 1) & 1, p.err, kErrTimeoutFull);
                    // V_j has landed (the softmax has waited for it already where it
                    // zeroes V_j's edge rows)
                    if (ok)
                        ok = mbar_wait_bounded(b_vfull + 8 * st, (js / NST) & 1, p.err, kErrTimeoutFull);
                    tc_fence_after();
                    if (ok) {
                        const uint32_t sV = s_base + G::kStageOff + st * G::kStageBytes + G::kKBytes;
                        const int np = min(G::kBlockPages, I.npages - j * G::kBlockPages);
                        // P_j: 16 tokens of page pp are 8 columns of S_j's buffer
                        const uint32_t tP = tbase + (jj & 1) * G::kBlockTokens;
                        for (int pp = 0; pp < np; ++pp)
                            umma_bf16_tmem_a(tbase + G::kOCol, tP + pp * 8,
                                             umma_sdesc(sV + pp * G::kVPage, kPage * 128, 1024), kIdO,
                                             j > 0 || pp > 0);
                    }
                    umma_commit(b_odone);
                    umma_commit(b_vempty + 8 * st);
                    umma_commit(b_sfree + 8 * (jj & 1));    // S_j's buffer, P_j with it, is free
                    if (j == I.nblocks - 1)
                        umma_commit(b_oitem);
                }
            }
            __syncwarp();
            jg += I.nblocks;
            ++kq;
        }
    } else {
        // ------------------------------------------------ softmax warps: kParts threads per query row
        constexpr int NP = G::kParts;
        constexpr int HC = G::kBlockTokens / NP;           // columns of S per thread
        constexpr int HO = HDC / NP;                       // columns of O per thread
        constexpr int kRs = HO >= 32 ? 32 : 16;            // O columns per rescale step
        const int row = (warp & 3) * 32 + lane;            // query row of the item; TMEM lane
        const int part = warp >> 2;                        // column part
        const uint32_t trow = tbase + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        float *xmax = reinterpret_cast<float *>(smem + G::kXOff);          // [2][NP][128]
        float *xsum = xmax + 2 * NP * G::kRows;                             // [NP][128]
        const int pair_bar = 1 + (warp & 3);                               // warps w, w + 4, w + 8, ...
        bool ok = true;
        int jg = 0;
        int qs = 0;                 // Q tiles that came through the ring

        // the finish of an item: the row sum over the parts, O / l in bf16
        // (this part's dims) -- or, split, the unnormalised partial (m, L, O)
        // -- then O is free for the next item
        int kfin = 0;               // items whose O has been read out
        auto finish = [&](size_t frh, bool fva, float fl, float fm, int fsplit) {
            xsum[part * G::kRows + row] = fl;
            group_bar_sync(pair_bar, 32 * NP);
            float lt = xsum[row];
#pragma unroll
            for (int k = 1; k < NP; ++k)
                lt += xsum[k * G::kRows + row];
            // every PV of the item is done (phase kfin of o_item: the items with
            // blocks in order; the next item's cannot end before this read-out)
            if (ok)
                ok = mbar_wait_bounded(b_oitem, kfin & 1, p.err, kErrTimeoutFull);
            ++kfin;
            tc_fence_after();
            const bool split_out = p.splits > 1;
            const size_t prow = frh * p.splits + fsplit;
            if (split_out && fva && part == 0 && crank == 0)     // a pair's two (m, L) are equal
                p.part_ml[prow] = make_float2(fm, lt);
            // one division per row, then a multiply per element (64 IEEE
            // divisions per thread took about 4 us per item)
            const float inv = lt > 0.f ? __frcp_rn(lt) : 0.f;
            const bool o_sector_aligned = (reinterpret_cast<uintptr_t>(p.o) & 31) == 0;
            const bool part_sector_aligned = (reinterpret_cast<uintptr_t>(p.part_o) & 31) == 0;
            // the row's O in pieces of kFinLd x 16 columns: the loads of a piece
            // are in flight together, then converted and stored
            constexpr int kFinLd = HO / 16 >= 2 ? 2 : 1;
#pragma unroll 1
            for (int c1 = part * HO; c1 < (part + 1) * HO; c1 += 16 * kFinLd) {
              uint32_t rr[kFinLd][16];
#pragma unroll
              for (int h = 0; h < kFinLd; ++h)
                  tmem_ld16(trow + G::kOCol + c1 + 16 * h, rr[h]);
              tmem_wait_ld();
#pragma unroll
              for (int h = 0; h < kFinLd; ++h) {
                const int c0 = c1 + 16 * h;
                const uint32_t (&r)[16] = rr[h];
                if (fva && split_out) {
                    float *dst = p.part_o + prow * HD + dofs + c0;
                    if (part_sector_aligned) {          // two whole sectors
                        const uint32_t (&lo)[8] = *reinterpret_cast<const uint32_t (*)[8]>(&r[0]);
                        const uint32_t (&hi)[8] = *reinterpret_cast<const uint32_t (*)[8]>(&r[8]);
                        st_global_32B(dst, lo);
                        st_global_32B(dst + 8, hi);
                    } else {
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            reinterpret_cast<float4 *>(dst)[k] =
                                make_float4(__uint_as_float(r[4 * k]), __uint_as_float(r[4 * k + 1]),
                                            __uint_as_float(r[4 * k + 2]), __uint_as_float(r[4 * k + 3]));
                    }
                } else if (fva) {
                    uint32_t w[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        __nv_bfloat162 v;
                        v.x = __float2bfloat16_rn(__fmul_rn(__uint_as_float(r[2 * k]), inv));
                        v.y = __float2bfloat16_rn(__fmul_rn(__uint_as_float(r[2 * k + 1]), inv));
                        w[k] = *reinterpret_cast<uint32_t *>(&v);
                    }
                    // one whole sector per lane where o allows it: the 32 lanes
                    // write 32 rows, so two 16-byte halves would each cost a
                    // partial-sector write
                    __nv_bfloat16 *dst = p.o + frh * HD + dofs + c0;
                    if (o_sector_aligned) {
                        st_global_32B(dst, w);
                    } else {
                        reinterpret_cast<uint4 *>(dst)[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        reinterpret_cast<uint4 *>(dst)[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
              }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(b_ofree);
        };

        bool pend = false;          // an item whose O has not been read out yet
        size_t pend_rh = 0;
        bool pend_va = false;
        float pend_l = 0.f, pend_m = -INFINITY;
        int pend_split = 0;
        int kit = 0;
        for (int it = first_item(0); it < nitems; it = next_item(it), ++kit) {
            const TcItem I = take_item(kit);
            const int2 wr = win[(kit & 1) * G::kRows + row];     // this query row's visible range
            release_item(kit);
            if (!I.live)
                continue;
            bool va = false;
            int lo_a = 1, hi_a = 0;
            size_t rh = 0;
            {
                const int qr = I.qbase + row;
                if (qr < I.tn * p.g) {
                    const int pr = qr / p.g, h = qr - pr * p.g;
                    lo_a = wr.x;
                    hi_a = wr.y;
                    rh = static_cast<size_t>(I.t0 + pr) * p.nh + I.kh * p.g + h;
                    va = true;
                }
            }
            if (I.nblocks == 0) {           // no position visible to any row: zeros, or an empty partial
                if (va && p.splits > 1) {
                    const size_t prow = rh * p.splits + I.split;
                    if (part == 0 && crank == 0)
                        p.part_ml[prow] = make_float2(-INFINITY, 0.f);
                    for (int c0 = part * HO; c0 < (part + 1) * HO; c0 += 4)
                        *reinterpret_cast<float4 *>(p.part_o + prow * HD + dofs + c0) =
                            make_float4(0.f, 0.f, 0.f, 0.f);
                } else if (va) {
                    for (int c0 = part * HO; c0 < (part + 1) * HO; c0 += 8)
                        *reinterpret_cast<uint4 *>(p.o + rh * HD + dofs + c0) = make_uint4(0u, 0u, 0u, 0u);
                }
                continue;
            }
            // this item's Q -> tensor memory columns kQCol + [0, hd/2), 16 columns
            // (32 elements) at a time, the parts taking turns; the previous
            // item's S MMAs, the only readers of Q, are all complete
            if (kQTma && I.qslot) {
                // from its ring stage: row r's 64-dim chunk c at c * 16 KB + 128 r,
                // 16-byte unit u at u ^ (r % 8)
                const int js = jg + qs;
                ++qs;
                const int st = js % NST;
                if (ok)
                    ok = mbar_wait_bounded(b_kfull + 8 * st, (js / NST) & 1, p.err, kErrTimeoutFull);
                const uint8_t *sq = smem + G::kStageOff + st * G::kStageBytes + row * 128;
                const uint32_t tq = trow + G::kQCol;
#pragma unroll
                for (int c0 = part * 16; c0 < HDC / 2; c0 += 16 * NP) {
                    const int e0 = 2 * c0;                          // first element of the piece
                    const uint8_t *src = sq + (e0 >> 6) * (G::kRows * 128);
                    const int u0 = (e0 & 63) >> 3;
                    uint32_t r[16];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(src + (((u0 + k) ^ (row & 7)) << 4));
                        r[4 * k] = v.x;
                        r[4 * k + 1] = v.y;
                        r[4 * k + 2] = v.z;
                        r[4 * k + 3] = v.w;
                    }
                    tmem_st16(tq + c0, r);
                }
                tmem_wait_st();
                tc_fence_before();
                group_bar_sync(5, 32 * G::kSoftmaxWarps);          // every softmax thread has read the tile
                if (tid == 0) {
                    mbar_arrive(b_kempty + 8 * st);
                    mbar_arrive(b_vempty + 8 * st);
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(b_qready);
            } else {
                // every load of this thread's part goes out before the first store
                constexpr int kQIt = (HDC / 2 + 16 * NP - 1) / (16 * NP);   // 16-column pieces per thread
                const uint4 *src = reinterpret_cast<const uint4 *>(p.q + rh * HD + dofs);
                const uint32_t tq = trow + G::kQCol;
                uint4 qv[kQIt][4];
#pragma unroll
                for (int i = 0; i < kQIt; ++i) {
                    const int c0 = part * 16 + i * 16 * NP;
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        qv[i][k] = va && c0 < HDC / 2 ? __ldg(src + c0 / 4 + k) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int i = 0; i < kQIt; ++i) {
                    const int c0 = part * 16 + i * 16 * NP;
                    if (c0 < HDC / 2) {
                        uint32_t r[16];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            r[4 * k] = qv[i][k].x;
                            r[4 * k + 1] = qv[i][k].y;
                            r[4 * k + 2] = qv[i][k].z;
                            r[4 * k + 3] = qv[i][k].w;
                        }
                        tmem_st16(tq + c0, r);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(b_qready);
            }
            if (pend)
                finish(pend_rh, pend_va, pend_l, pend_m, pend_split);

            float m = -INFINITY, l = 0.f;
            for (int j = 0; j < I.nblocks; ++j) {
                const int jj = jg + j;
                const int b = jj & 1;
                if (ok)
                    ok = mbar_wait_bounded(b_sfull + 8 * b, (jj >> 1) & 1, p.err, kErrTimeoutFull);
                tc_fence_after();
                uint32_t sr[HC];
#pragma unroll
                for (int q4 = 0; q4 < HC / 16; ++q4)
                    tmem_ld16(trow + b * G::kBlockTokens + part * HC + q4 * 16,
                              *reinterpret_cast<uint32_t(*)[16]>(sr + q4 * 16));
                tmem_wait_ld();
                tc_fence_before();
                if constexpr (kSplit) {
                    // The pair's halves of S_j: this thread's 16 columns go to the
                    // peer, the peer's come here, and the two are added.  a + b is
                    // b + a bit for bit, so both CTAs hold the same S_j and run the
                    // same softmax.  The peer writes buffer b again (block jj + 2)
                    // only after it has every thread's half of block jj + 1 from
                    // here, which each thread sends after reading block jj's.
                    static_assert(HC == 16, "exchange layout: four float4 per thread");
                    const uint32_t xoff = G::kSxOff + static_cast<uint32_t>(((b * NP + part) * 4 * G::kRows + row) * 16);
                    const int peer = crank ^ 1;
                    const uint32_t rbar = map_to_cta(b_xfull + 8 * b, peer);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        st_async_f32x4(map_to_cta(s_base + xoff + k * G::kRows * 16, peer),
                                       make_float4(__uint_as_float(sr[4 * k]), __uint_as_float(sr[4 * k + 1]),
                                                   __uint_as_float(sr[4 * k + 2]), __uint_as_float(sr[4 * k + 3])),
                                       rbar);
                    if (ok)
                        ok = mbar_wait_bounded(b_xfull + 8 * b, (jj >> 1) & 1, p.err, kErrTimeoutFull);
                    if (tid == 0 && ok)    // arm the buffer's next phase (block jj + 2)
                        mbar_arrive_expect_tx(b_xfull + 8 * b, G::kRows * G::kBlockTokens * 4);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float4 v = *reinterpret_cast<const float4 *>(smem + xoff + k * G::kRows * 16);
                        sr[4 * k] = __float_as_uint(__uint_as_float(sr[4 * k]) + v.x);
                        sr[4 * k + 1] = __float_as_uint(__uint_as_float(sr[4 * k + 1]) + v.y);
                        sr[4 * k + 2] = __float_as_uint(__uint_as_float(sr[4 * k + 2]) + v.z);
                        sr[4 * k + 3] = __float_as_uint(__uint_as_float(sr[4 * k + 3]) + v.w);
                    }
                }

                const int tok0 = (I.p_first + j * G::kBlockPages) * kPage + part * HC;
                // mask to the row's window; this part's max in four chains, then the row's
                float x[HC];
                float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
                if (tok0 >= lo_a && tok0 + HC - 1 <= hi_a) {
#pragma unroll
                    for (int c = 0; c < HC; ++c) {
                        x[c] = __uint_as_float(sr[c]);
                        mq[c & 3] = fmaxf(mq[c & 3], x[c]);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < HC; ++c) {
                        const int t = tok0 + c;
                        x[c] = (t >= lo_a && t <= hi_a) ? __uint_as_float(sr[c]) : -INFINITY;
                        mq[c & 3] = fmaxf(mq[c & 3], x[c]);
                    }
                }
                const float mh = fmaxf(fmaxf(mq[0], mq[1]), fmaxf(mq[2], mq[3]));
                xmax[(b * NP + part) * G::kRows + row] = mh;
                group_bar_sync(pair_bar, 32 * NP);
                float mr = mh;
#pragma unroll
                for (int k = 0; k < NP; ++k)
                    mr = fmaxf(mr, xmax[(b * NP + k) * G::kRows + row]);
                const float mx = mr * kLog2e;   // log2 units
                // stale-max rescale: keep m unless the block's max exceeds it by more than 8
                float m_use = m, alpha = 1.f;
                if (mx > m + 8.f || (m == -INFINITY && mx != -INFINITY)) {
                    m_use = mx;
                    alpha = (m == -INFINITY) ? 0.f : exp2f(m - mx);
                }
                const bool live = m_use != -INFINITY;
                const float nm = live ? -m_use : 0.f;
                float lq[4] = {0.f, 0.f, 0.f, 0.f};
                uint32_t pk[HC / 2];
#pragma unroll
                for (int c = 0; c < HC; c += 2) {
                    // P rounded to bf16 once, by the pair conversion; the row sum
                    // takes the rounded values back out of the packed word
                    const float e0 = live ? ex2_sfu(__fmaf_rn(x[c], kLog2e, nm)) : 0.f;
                    const float e1 = live ? ex2_sfu(__fmaf_rn(x[c + 1], kLog2e, nm)) : 0.f;
                    const uint32_t w = pack_bf16x2(e0, e1);
                    pk[c / 2] = w;
                    lq[(c >> 1) & 3] += __uint_as_float(w << 16) + __uint_as_float(w & 0xffff0000u);
                }
                l = __fmaf_rn(l, alpha, (lq[0] + lq[1]) + (lq[2] + lq[3]));     // this part's share
                m = m_use;

                // O may be rescaled once the previous block's PV is done.  P_j goes
                // where S_j was, so it waits for nothing more: PV_{j-2}, the
                // buffer's last reader, was done before S_j was issued into it, and
                // every part of the row has read S_j (the row-max barrier above).
                // PV_j needs P_j, so b_odone has not passed PV_{j-1} here.
                const bool rescale = j >= 1 && __any_sync(0xffffffffu, alpha != 1.f);
                if (rescale && ok)
                    ok = mbar_wait_bounded(b_odone, (jj - 1) & 1, p.err, kErrTimeoutFull);
                tc_fence_after();
                if (rescale) {
#pragma unroll 1
                    for (int c0 = part * HO; c0 < (part + 1) * HO; c0 += kRs) {
                        uint32_t ra[kRs / 16][16];
#pragma unroll
                        for (int h = 0; h < kRs / 16; ++h)
                            tmem_ld16(trow + G::kOCol + c0 + 16 * h, ra[h]);
                        tmem_wait_ld();
#pragma unroll
                        for (int h = 0; h < kRs / 16; ++h)
#pragma unroll
                            for (int k = 0; k < 16; ++k)
                                ra[h][k] = __float_as_uint(__uint_as_float(ra[h][k]) * alpha);
#pragma unroll
                        for (int h = 0; h < kRs / 16; ++h)
                            tmem_st16(trow + G::kOCol + c0 + 16 * h, ra[h]);
                    }
                    tmem_wait_st();
                }
                // this part of the P row -> tensor memory, tokens (2c, 2c + 1) of the
                // block in column c of S_j's buffer (the low half the lower token)
                static_assert(HC == 16, "P: eight columns per part");
                tmem_st8(trow + b * G::kBlockTokens + part * (HC / 2), pk);
                tmem_wait_st();
                // V rows of tokens outside the union window may hold anything (NaN
                // included) and P is 0 there: zero them before the PV MMA reads them
                const int btok0 = (I.p_first + j * G::kBlockPages) * kPage;
                if (btok0 < I.lo_u || btok0 + G::kBlockTokens - 1 > I.hi_u) {
                    const int js = jj + qs, st = js % NST;
                    if (ok)           // V_j lands apart from K_j: zero nothing before the copy has
                        ok = mbar_wait_bounded(b_vfull + 8 * st, (js / NST) & 1, p.err, kErrTimeoutFull);
                    uint8_t *sV = smem + G::kStageOff + st * G::kStageBytes + G::kKBytes;
                    const int np = min(G::kBlockPages, I.npages - j * G::kBlockPages);
                    for (int e = tid; e < np * kPage * NCH * 8; e += G::kSoftmaxWarps * 32) {
                        const int u = e & 7, rc = e >> 3;
                        const int c = rc % NCH, tk = rc / NCH;     // token of the block, chunk
                        const int t = btok0 + tk;
                        if (t < I.lo_u || t > I.hi_u)
                            *reinterpret_cast<uint4 *>(sV + (tk >> 4) * G::kVPage + c * (kPage * 128) +
                                                       (tk & 15) * 128 + u * 16) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                fence_async_shared();
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(b_pfull + 8 * b);
            }
            pend = true;
            pend_rh = rh;
            pend_va = va;
            pend_l = l;
            pend_m = m;
            pend_split = I.split;
            jg += I.nblocks;
        }
        if (pend)
            finish(pend_rh, pend_va, pend_l, pend_m, pend_split);
    }
    // split dims: neither CTA of the pair leaves while the other may still
    // write into its shared memory
    if (kSplit) {
        cluster_arrive_release();
        cluster_wait();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc<G::kTmemCols>(tbase);
    }
}

// Clusters of two CTAs of the split-dims kernel that can be resident at once
// on the current device (0: none), asked once per device after the kernel's
// shared-memory attribute is set.
template <int HD>
int prefill_tc_pair_capacity()
{
    static int cap[64];
    static bool known[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
        return 0;
    if (known[dev])
        return cap[dev];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(TcGeo<HD>::kThreads);
    cfg.dynamicSmemBytes = TcGeo<HD>::kAlloc;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, prefill_tc_kernel<HD, false>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cap[dev] = n;
    known[dev] = true;
    return n;
}

template <int HD>
cudaError_t launch_prefill_tc(const PrefillLaunchArgs &a, bool set_attr)
{
    using G = TcGeo<HD>;
    if (set_attr) {
        cudaError_t e = cudaSuccess;
        for (auto kern : {prefill_tc_kernel<HD, false>, prefill_tc_kernel<HD, true>})
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, G::kAlloc);
        if (e != cudaSuccess)
            return e;
    }
    const int tile_rows = a.max_tile_rows > 0 ? std::min(a.max_tile_rows, a.p.rows_per_tile) : a.p.rows_per_tile;
    const int nchunks = (tile_rows * a.p.g + G::kRows - 1) / G::kRows;
    const long long items = static_cast<long long>(a.ntiles) * a.p.nkv * nchunks * a.p.splits;
    if (items > INT_MAX)
        return cudaErrorInvalidValue;
    // one unit (a CTA, or at hd 512 a pair) per item while they fit in about
    // two waves (the hardware then hands the second wave to the first units
    // free); persistent, as many units as are resident at once, beyond that
    long long resident = a.num_sms > 0 ? a.num_sms : 1;
    if (G::kSplitDims) {
        resident = prefill_tc_pair_capacity<HD>();
        if (resident < 1)
            return cudaErrorInvalidConfiguration;
    }
    const long long units = items <= 2 * resident ? items : resident;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    int na = 1;
    if (G::kSplitDims) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = 2;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        na = 2;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(G::kSplitDims ? 2 * units : units));
    cfg.blockDim = dim3(G::kThreads);
    cfg.dynamicSmemBytes = G::kAlloc;
    cfg.stream = a.stream;
    cfg.attrs = attr;
    cfg.numAttrs = na;
    // without a Q map the kernel never reads tm_q: K's map fills the parameter
    const CUtensorMap &tq = a.tm_q ? *a.tm_q : *a.tm_k;
    auto kern = a.tm_q ? prefill_tc_kernel<HD, true> : prefill_tc_kernel<HD, false>;
    return cudaLaunchKernelEx(&cfg, kern, *a.tm_k, *a.tm_v, tq, a.p, a.ntiles, nchunks);
}

}  // namespace pgqa
