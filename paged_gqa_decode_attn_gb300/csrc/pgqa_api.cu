// C ABI of libpgqa.so (declared in include/pgqa.h): argument checks, the
// split heuristic, scratch sizing, TMA descriptors and the launches.
//
// The entry points mirror the calls of span-02
// `engine/crates/kernels/tests/gpu.rs`: `attn::attn_decode`,
// `attn::choose_splits` and `attn::decode_part_bytes` in its `run` function.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "pgqa.h"
#include "pgqa_launch.cuh"
#include "pgqa_prefill.cuh"

namespace pgqa {
int current_context_id(unsigned long long *id);
}

namespace {

// Device-side error word: bounded waits OR their code into it.
__device__ unsigned int g_pgqa_error_word;

constexpr int kMaxDevices = 64;

struct DeviceState {
    bool ready = false;
    unsigned long long ctx_id = 0;   // the context everything below belongs to
    int num_sms = 0;
    unsigned int *err = nullptr;
    bool attr_set[4] = {false, false, false, false};
    bool prefill_attr_set[4] = {false, false, false, false};
    int cluster_cap[4][5] = {{-1, -1, -1, -1, -1}, {-1, -1, -1, -1, -1}, {-1, -1, -1, -1, -1},
                             {-1, -1, -1, -1, -1}};   // [hd][log2 cluster]: resident clusters, -1 unknown
    int cps[4] = {-1, -1, -1, -1};   // [hd]: split CTAs resident per SM, -1 unknown
};

// Cluster size for the on-chip merge of `splits` CTAs, or 0 to merge through
// global memory.  Clusters of 2 and 4 are taken whenever any fit (for the
// short loops that choose them, a second wave of clusters measured faster
// than the last-CTA merge); clusters of 8 only when all `live` ones (one per
// tile that does work) are resident at once: the split rule picks 8 beside
// fewer resident clusters only for long loops, where a waiting cluster would
// double its tile's time.  Caller holds g_mutex.
int on_chip_cluster(DeviceState *s, int hi, int hd, int splits, long long live)
{
    int lg = -1;
    switch (splits) {
    case 2: lg = 1; break;
    case 4: lg = 2; break;
    case 8: lg = 3; break;
    default: return 0;          // 16-CTA clusters rarely all fit beside each other
    }
    int &cap = s->cluster_cap[hi][lg];
    if (cap < 0) {
        switch (hd) {
        case 64: cap = pgqa::cluster_capacity_hd64(splits); break;
        case 128: cap = pgqa::cluster_capacity_hd128(splits); break;
        case 256: cap = pgqa::cluster_capacity_hd256(splits); break;
        default: cap = pgqa::cluster_capacity_hd512(splits); break;
        }
    }
    return cap >= 1 && (splits <= 4 || cap >= live) ? splits : 0;
}

std::mutex g_mutex;
DeviceState g_dev[kMaxDevices];
unsigned long long *g_trace = nullptr;    // trace builds: per-CTA timestamps
size_t g_trace_bytes = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_current = nullptr;
CtxGetIdFn g_ctx_id = nullptr;

using MemGetAddressRangeFn = CUresult (*)(CUdeviceptr *, size_t *, CUdeviceptr);
MemGetAddressRangeFn g_mem_range = nullptr;

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

int hd_index(int hd)
{
    switch (hd) {
    case 64: return 0;
    case 128: return 1;
    case 256: return 2;
    case 512: return 3;
    default: return -1;
    }
}

// Per-device set-up (SM count, error-word address).  Caller holds g_mutex.
// Everything cached here belongs to one CUDA context: a device reset
// (cudaDeviceReset) destroys the context, and the next one may place the
// module's device symbols elsewhere and has none of the kernel attributes, so
// the state is rebuilt whenever the current context's id changes.
int device_state(DeviceState **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PGQA_ERR_CUDA;
    unsigned long long ctx = 0;
    if (pgqa::current_context_id(&ctx) != PGQA_OK)
        return PGQA_ERR_CUDA;
    DeviceState &s = g_dev[dev];
    if (s.ready && s.ctx_id != ctx)
        s = DeviceState();
    if (!s.ready) {
        s.ctx_id = ctx;
        if (cudaDeviceGetAttribute(&s.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return PGQA_ERR_CUDA;
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pgqa_error_word) != cudaSuccess)
            return PGQA_ERR_CUDA;
        s.err = static_cast<unsigned int *>(p);
        s.ready = true;
    }
    *out = &s;
    return PGQA_OK;
}

// Bytes from `ptr` to the end of the device allocation that holds it, or 0
// when the driver cannot tell (memory it did not allocate with cuMemAlloc or
// cudaMalloc, such as virtual-memory mappings, or a null pointer).
long long bytes_to_allocation_end(const void *ptr)
{
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_mem_range = reinterpret_cast<MemGetAddressRangeFn>(fn);
    });
    if (!g_mem_range || !ptr)
        return 0;
    CUdeviceptr base = 0;
    size_t size = 0;
    const CUdeviceptr d = reinterpret_cast<CUdeviceptr>(ptr);
    if (g_mem_range(&base, &size, d) != CUDA_SUCCESS || d < base || d - base >= size)
        return 0;
    return static_cast<long long>(base + size - d);
}

// The speculative prefetch's extents for a decode launch (pgqa_device.cuh):
// every field stays 0, and the prefetch off, unless all allocations are known.
void set_speculation(pgqa::DecodeParams &p, const void *k_pool, const void *v_pool, int hd)
{
    const long long tile_bytes = static_cast<long long>(pgqa::kPage) * hd * 2;
    const long long kb = bytes_to_allocation_end(k_pool), vb = bytes_to_allocation_end(v_pool);
    const long long bb = bytes_to_allocation_end(p.block_table);
    const long long mb = p.page_map ? bytes_to_allocation_end(p.page_map) : 0;
    if (kb < tile_bytes || vb < tile_bytes || bb < 4 || (p.page_map && mb < 4))
        return;
    p.spec_tiles = std::min(kb, vb) / tile_bytes;
    p.spec_bt_len = bb / 4;
    p.spec_pm_len = mb / 4;
}

int get_encoder()
{
    if (g_encode)
        return PGQA_OK;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
        return PGQA_ERR_TENSOR_MAP;
    g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    return PGQA_OK;
}

// TMA descriptors of a [pages][nkv][16][hd] bf16 pool.  The pool's page
// count is not known here, so the tile dimension spans the int32 coordinate
// range; only tiles the block table names are ever addressed.  Three views,
// all under the 128-byte swizzle:
//   kMapWhole  -- 4-D (64 dims, 16 slots, hd/64 dim chunks, tile = phys*nkv + kh):
//                 one box per (page, kv head) tile, in shared memory as
//                 [chunk][slot][64];
//   kMapHalves -- 5-D (64 dims, 8 slots, hd/64 chunks, 2 slot halves, tile):
//                 one box per tile, in shared memory as [half][chunk][8 slots][64],
//                 so that the 8-slot swizzle atoms of one chunk sit hd * 16
//                 bytes apart across consecutive tiles (the tcgen05 prefill's
//                 K operand);
//   kMapChunks -- 3-D (dims, slots, tiles) with 64-dim boxes: hd/64 copies per
//                 tile, and the fallback where the driver refuses the others.
enum MapKind { kMapWhole = 1, kMapHalves = 2, kMapChunks = 0 };

struct MapCacheEntry {
    const void *base = nullptr;
    int hd = 0;
    int want = -1;           // the view asked for
    int box_chunks = 0;      // 64-dim chunks per box (the whole and halves views)
    int kind = 0;            // the view built
    CUtensorMap map;
};
MapCacheEntry g_map_cache[128];
unsigned g_map_next = 0;

// `box_chunks` (0: hd / 64) sets how many 64-dim chunks of a tile one box of
// the whole or halves view takes: half of them serves one CTA of the hd-512
// prefill's pairs.
int pool_map(const void *base, int hd, CUtensorMap *out, int *kind, int want = kMapWhole, int box_chunks = 0)
{
    if (box_chunks <= 0)
        box_chunks = hd / 64;
    for (auto &e : g_map_cache)
        if (e.base == base && e.hd == hd && e.want == want && e.box_chunks == box_chunks) {
            *out = e.map;
            *kind = e.kind;
            return PGQA_OK;
        }
    int st = get_encoder();
    if (st != PGQA_OK)
        return st;
    CUtensorMap m;
    int w = want;
    if (w == kMapWhole) {
        const cuuint64_t dims[4] = {64u, 16u, static_cast<cuuint64_t>(hd / 64), 0x7fffffffull};
        const cuuint64_t strides[3] = {static_cast<cuuint64_t>(hd) * 2u, 128u, static_cast<cuuint64_t>(hd) * 32u};
        const cuuint32_t box[4] = {64u, 16u, static_cast<cuuint32_t>(box_chunks), 1u};
        const cuuint32_t estride[4] = {1u, 1u, 1u, 1u};
        CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides, box,
                              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            w = kMapChunks;
    } else if (w == kMapHalves) {
        const cuuint64_t dims[5] = {64u, 8u, static_cast<cuuint64_t>(hd / 64), 2u, 0x7fffffffull};
        const cuuint64_t strides[4] = {static_cast<cuuint64_t>(hd) * 2u, 128u, static_cast<cuuint64_t>(hd) * 16u,
                                       static_cast<cuuint64_t>(hd) * 32u};
        const cuuint32_t box[5] = {64u, 8u, static_cast<cuuint32_t>(box_chunks), 2u, 1u};
        const cuuint32_t estride[5] = {1u, 1u, 1u, 1u, 1u};
        CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims, strides, box,
                              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            w = kMapChunks;
    }
    if (w == kMapChunks) {
        const cuuint64_t dims[3] = {static_cast<cuuint64_t>(hd), 16u, 0x7fffffffull};
        const cuuint64_t strides[2] = {static_cast<cuuint64_t>(hd) * 2u, static_cast<cuuint64_t>(hd) * 32u};
        const cuuint32_t box[3] = {64u, 16u, 1u};
        const cuuint32_t estride[3] = {1u, 1u, 1u};
        CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                              estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS)
            return PGQA_ERR_TENSOR_MAP;
    }
    MapCacheEntry &e = g_map_cache[g_map_next++ % 128];
    e.base = base;
    e.hd = hd;
    e.want = want;
    e.box_chunks = box_chunks;
    e.kind = w;
    e.map = m;
    *out = m;
    *kind = w;
    return PGQA_OK;
}

// A TMA descriptor of a [rows][nh][hd] bf16 Q whose box is one tcgen05 prefill
// chunk's 64 dims: 64 dims x g heads (one kv head's) x 128 / g rows, under the
// 128-byte swizzle.  The row count is not known here, so the row dimension
// spans the int32 range; the kernel loads only chunks whose rows all lie in a
// tile.  Needs g to divide 128.
struct QMapEntry {
    const void *base = nullptr;
    int nh = 0, hd = 0, g = 0;
    CUtensorMap map;
};
QMapEntry g_qmap_cache[32];
unsigned g_qmap_next = 0;

int q_map(const void *base, int nh, int hd, int g, CUtensorMap *out)
{
    if (g < 1 || g > 128 || 128 % g != 0)
        return PGQA_ERR_INVALID_ARGUMENT;
    for (auto &e : g_qmap_cache)
        if (e.base == base && e.nh == nh && e.hd == hd && e.g == g) {
            *out = e.map;
            return PGQA_OK;
        }
    int st = get_encoder();
    if (st != PGQA_OK)
        return st;
    CUtensorMap m;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(hd), static_cast<cuuint64_t>(nh), 0x7fffffffull};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(hd) * 2u, static_cast<cuuint64_t>(nh) * hd * 2u};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(128 / g)};
    const cuuint32_t estride[3] = {1u, 1u, 1u};
    CUresult r = g_encode(&m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                          estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
        return PGQA_ERR_TENSOR_MAP;
    QMapEntry &e = g_qmap_cache[g_qmap_next++ % 32];
    e.base = base;
    e.nh = nh;
    e.hd = hd;
    e.g = g;
    e.map = m;
    *out = m;
    return PGQA_OK;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

namespace pgqa {
// Unique id of the CUDA context current on this thread (the runtime's primary
// context of the current device unless the caller made another current).  A
// thread with no current context gets the current device's primary context
// first: cudaSetDevice initialises it, and allocates nothing.
int current_context_id(unsigned long long *id)
{
    static std::once_flag once;
    std::call_once(once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_current = reinterpret_cast<CtxGetCurrentFn>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_id = reinterpret_cast<CtxGetIdFn>(fn);
    });
    if (!g_ctx_current || !g_ctx_id)
        return PGQA_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS)
        return PGQA_ERR_CUDA;
    if (ctx == nullptr) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || cudaSetDevice(dev) != cudaSuccess ||
            g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr)
            return PGQA_ERR_CUDA;
    }
    return g_ctx_id(ctx, id) == CUDA_SUCCESS ? PGQA_OK : PGQA_ERR_CUDA;
}

// SM count and error-word address of the current device, for the entry
// points defined in other translation units.
int device_info(int *num_sms, unsigned int **err)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState *s = nullptr;
    const int st = device_state(&s);
    if (st != PGQA_OK)
        return st;
    *num_sms = s->num_sms;
    *err = s->err;
    return PGQA_OK;
}

int split_kernel_smem_bytes(int hd)
{
    switch (hd) {
    case 64: return Smem<64>::kAlloc;
    case 128: return Smem<128>::kAlloc;
    case 256: return Smem<256>::kAlloc;
    case 512: return Smem<512>::kAlloc;
    default: return 0;
    }
}

cudaError_t launch_bounded_wait_probe(unsigned int *err, cudaStream_t stream);   // pgqa_selftest.cu
}  // namespace pgqa

extern "C" {

int pgqa_version(void) { return 100; }

int pgqa_trace_buffer(void *device_buffer, size_t bytes)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    g_trace = static_cast<unsigned long long *>(device_buffer);
    g_trace_bytes = device_buffer ? bytes : 0;
#ifdef PGQA_TRACE
    return PGQA_OK;
#else
    return PGQA_ERR_INVALID_ARGUMENT;
#endif
}

const char *pgqa_strerror(int status)
{
    switch (status) {
    case PGQA_OK: return "ok";
    case PGQA_ERR_INVALID_ARGUMENT: return "invalid argument";
    case PGQA_ERR_UNSUPPORTED_HD: return "unsupported head dimension (64, 128, 256 or 512)";
    case PGQA_ERR_MISALIGNED: return "buffer not 16-byte aligned";
    case PGQA_ERR_CUDA: return "CUDA runtime error";
    case PGQA_ERR_TENSOR_MAP: return "TMA descriptor rejected by the driver";
    case PGQA_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    case PGQA_ERR_TOO_MANY_SPLITS: return "splits above PGQA_MAX_SPLITS";
    case PGQA_ERR_NOALLOC_TOO_LARGE: return "call needs more scratch than the no-allocation entry point holds";
    case PGQA_ERR_TILE_TOO_LONG: return "a prefill tile held more rows than pgqa_prefill_rows_per_tile";
    default: return "unknown status";
    }
}

size_t pgqa_decode_part_bytes(int rows, int nh, int splits, int hd)
{
    if (rows <= 0 || nh <= 0 || splits <= 0 || hd <= 0)
        return 0;
    return static_cast<size_t>(rows) * nh * splits * (static_cast<size_t>(hd) + 2) * 4;
}

size_t pgqa_decode_counter_count(int rows, int nh, int nkv)
{
    if (rows <= 0 || nh <= 0 || nkv <= 0 || nh % nkv != 0)
        return 0;
    const int g = nh / nkv;
    return static_cast<size_t>(rows) * nkv * ((g + pgqa::kQRows - 1) / pgqa::kQRows);
}

int pgqa_decode_kernel_count(int splits, int with_counters)
{
    if (splits < 1 || splits > PGQA_MAX_SPLITS)
        return 0;
    return splits == 1 || (with_counters && splits <= pgqa::kGroupSplits) ? 1 : 2;
}

namespace {

// Clusters of 2, 4 and 8 CTAs (index log2) resident at once with one CTA per
// SM -- the split kernel's shape at head dims 256 and 512 -- measured on a
// 152-SM GB300.  A cluster must fit in one GPC, so 8-CTA clusters fit only
// 15 times, not 19.
constexpr int kClusters152[4] = {152, 76, 36, 15};

// The split-count rule; `clusters` (index log2 of the size) is the device's
// cluster residency, or null for the 152-SM table scaled to num_sms.
int choose_splits_rule(int kv_len_eff, int rows, int nkv, int nseq, int num_sms, const int *clusters)
{
    if (kv_len_eff < 1)
        kv_len_eff = 1;
    if (rows < 1)
        rows = 1;
    if (nseq < 1 || nseq > rows)
        nseq = rows;
    if (nkv < 1)
        nkv = 1;
    if (num_sms < 1)
        num_sms = 1;
    const long long pages = (kv_len_eff + PGQA_PAGE_TOKENS - 1) / PGQA_PAGE_TOKENS;
    // Rows of one sequence share CTAs (row packing), so the CTAs of one split
    // are about nseq * nkv.  Few tiles: split until the grid is one wave of
    // one CTA per SM.  Many tiles: about four CTAs per SM, for balance.
    const long long tiles = static_cast<long long>(nseq) * nkv;
    long long s = tiles < num_sms ? (num_sms + tiles - 1) / tiles : (4LL * num_sms + tiles - 1) / tiles;
    long long cap = pages / 2;       // at least two pages per split
    if (cap < 1)
        cap = 1;
    if (s > cap)
        s = cap;
    // Up to 24 splits, take a power of two no larger than 8: 2, 4 and 8
    // splits merge on chip, in one thread-block cluster per tile.  Prefer the
    // largest such size whose clusters, one per tile, are all resident at
    // once; if none is, the largest power of two.  When the size that fits is
    // smaller than wanted and a split's loop is long, the wanted count wins
    // instead, merged by the last CTA in one level (a few microseconds more
    // than on chip, about kMergePages pages of one CTA's loop) -- the launch
    // takes the on-chip merge only where all clusters are resident.
    if (s <= 24) {
        long long p2 = 1;
        while (p2 * 2 <= s && p2 < 8)
            p2 *= 2;
        long long fit = 1;
        for (int lg = 1; (1LL << lg) <= p2; ++lg) {
            const long long res = clusters ? clusters[lg] : static_cast<long long>(kClusters152[lg]) * num_sms / 152;
            if (res >= tiles)
                fit = 1LL << lg;
        }
        // (only while the grid stays one wave even unpacked: how many rows a
        // CTA packs depends on the group size, which this rule is not given)
        constexpr long long kMergePages = 16;
        if (fit > 1 && fit < p2 && pages / fit - pages / p2 > kMergePages &&
            static_cast<long long>(rows) * nkv * p2 <= num_sms)
            s = p2;
        else
            s = fit > 1 ? fit : p2;
    }
    if (s > PGQA_MAX_SPLITS)
        s = PGQA_MAX_SPLITS;
    if (s < 1)
        s = 1;
    return static_cast<int>(s);
}

// The split rule with the kernel's shape known (pgqa_choose_splits_ex).  Every
// sequence's rows pack into CTAs of max(1, 8 / g) rows (g = nh / nkv), so a
// split has `tiles` CTAs.  With at least one tile per SM the grid is many
// waves and the page-signature rule above stands.  With fewer, the count was
// fitted to decode timings over hd {128, 256, 512} x nkv {2..32} x context
// {1K..64K} on a GB300:
//  * fill the GPU in one wave: one CTA per SM where one fits per SM (hd 256,
//    512), about 2.5 per SM where three fit (hd 64, 128: each CTA's ring is
//    then half an SM's, and more CTAs keep more bytes in flight);
//  * but while a CTA's loop stays short -- at most kShortLoopBytes of K and V
//    per two query rows the CTA serves, with the largest cluster size whose
//    clusters all fit -- take that cluster size: its on-chip merge costs less
//    than the combine kernel's second launch saves, and the combine kernel's
//    share grows with the (row, head) pairs it merges (4 packed rows at g = 2
//    took 11.6 us through it against 8.8 on chip, where one row was even).
constexpr long long kShortLoopBytes = 128 * 1024;
// ... and at most 16 pages: at hd 128 a one-CTA-per-SM cluster grid keeps
// fewer bytes in flight per SM than the fill (4 rows over 256 pages: 12.9 us
// on chip against 11.8 through the combine kernel).
constexpr long long kShortLoopPages = 16;

int choose_splits_ex_rule(int kv_len_eff, int rows, int nkv, int nseq, int nh, int hd, int num_sms, int cps,
                          const int *clusters)
{
    if (kv_len_eff < 1)
        kv_len_eff = 1;
    if (rows < 1)
        rows = 1;
    if (nseq < 1 || nseq > rows)
        nseq = rows;
    if (num_sms < 1)
        num_sms = 1;
    if (cps < 1)
        cps = 1;
    const int g = nh / nkv;
    const long long pack = g <= pgqa::kQRows ? pgqa::kQRows / g : 1;
    const long long hsg = (g + pgqa::kQRows - 1) / pgqa::kQRows;
    const long long per_seq = (rows + nseq - 1) / nseq;
    const long long tiles = static_cast<long long>(nseq) * ((per_seq + pack - 1) / pack) * nkv * hsg;
    if (tiles >= num_sms)
        return choose_splits_rule(kv_len_eff, rows, nkv, nseq, num_sms, clusters);
    const long long pages = (kv_len_eff + PGQA_PAGE_TOKENS - 1) / PGQA_PAGE_TOKENS;
    const long long target = cps > 1 ? 5LL * num_sms / 2 : num_sms;
    long long fill = target / tiles;
    fill = std::min<long long>(fill, std::max<long long>(1, pages / 2));    // at least two pages per split
    fill = std::max<long long>(1, std::min<long long>(fill, PGQA_MAX_SPLITS));
    long long c = 1;                                                      // on-chip merge that fits
    for (int lg = 1; lg <= 3; ++lg)
        if ((1LL << lg) <= fill && clusters[lg] >= tiles)
            c = 1LL << lg;
    const long long qrows = std::min<long long>(pgqa::kQRows, std::min(per_seq, pack) * g);   // per CTA
    long long s;
    if (fill <= 8)
        s = c > 1 ? c : fill;
    else if (c > 1 && (pages + c - 1) / c <= kShortLoopPages &&
             (pages + c - 1) / c * 64LL * hd <= kShortLoopBytes * std::max<long long>(1, qrows / 2))
        s = c;
    else
        s = fill;
    return static_cast<int>(s);
}

bool ex_args_ok(int nh, int nkv, int hd)
{
    return nh > 0 && nkv > 0 && nh % nkv == 0 && hd_index(hd) >= 0;
}

}  // namespace

int pgqa_choose_splits_ex_for(int kv_len_eff, int rows, int nkv, int nseq, int nh, int hd, int num_sms,
                              int ctas_per_sm, int clusters2, int clusters4, int clusters8)
{
    if (!ex_args_ok(nh, nkv, hd))
        return hd_index(hd) < 0 ? PGQA_ERR_UNSUPPORTED_HD : PGQA_ERR_INVALID_ARGUMENT;
    const int clusters[4] = {num_sms, clusters2, clusters4, clusters8};
    return choose_splits_ex_rule(kv_len_eff, rows, nkv, nseq, nh, hd, num_sms, ctas_per_sm, clusters);
}

int pgqa_choose_splits_ex(int kv_len_eff, int rows, int nkv, int nseq, int nh, int hd)
{
    if (!ex_args_ok(nh, nkv, hd))
        return hd_index(hd) < 0 ? PGQA_ERR_UNSUPPORTED_HD : PGQA_ERR_INVALID_ARGUMENT;
    const int hi = hd_index(hd);
    int sms = 0, cps = 0;
    int clusters[4] = {};
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        DeviceState *s = nullptr;
        const int st = device_state(&s);
        if (st != PGQA_OK)
            return st;
        sms = s->num_sms;
        if (s->cps[hi] < 0) {
            switch (hd) {
            case 64: s->cps[hi] = pgqa::ctas_per_sm_hd64(); break;
            case 128: s->cps[hi] = pgqa::ctas_per_sm_hd128(); break;
            case 256: s->cps[hi] = pgqa::ctas_per_sm_hd256(); break;
            default: s->cps[hi] = pgqa::ctas_per_sm_hd512(); break;
            }
        }
        cps = s->cps[hi];
        clusters[0] = sms;
        for (int lg = 1; lg <= 3; ++lg) {
            int &cap = s->cluster_cap[hi][lg];
            if (cap < 0) {
                switch (hd) {
                case 64: cap = pgqa::cluster_capacity_hd64(1 << lg); break;
                case 128: cap = pgqa::cluster_capacity_hd128(1 << lg); break;
                case 256: cap = pgqa::cluster_capacity_hd256(1 << lg); break;
                default: cap = pgqa::cluster_capacity_hd512(1 << lg); break;
                }
            }
            clusters[lg] = cap;
        }
    }
    return choose_splits_ex_rule(kv_len_eff, rows, nkv, nseq, nh, hd, sms, cps, clusters);
}

int pgqa_choose_splits_for(int kv_len_eff, int rows, int nkv, int nseq, int num_sms)
{
    return choose_splits_rule(kv_len_eff, rows, nkv, nseq, num_sms, nullptr);
}

int pgqa_choose_splits(int kv_len_eff, int rows, int nkv, int nseq)
{
    int sms = 152;
    int clusters[4] = {};
    bool have = false;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        DeviceState *s = nullptr;
        if (device_state(&s) == PGQA_OK) {
            sms = s->num_sms;
            have = true;
            for (int lg = 1; lg <= 3; ++lg) {    // the one-CTA-per-SM shape: head dim 256
                int &cap = s->cluster_cap[2][lg];
                if (cap < 0)
                    cap = pgqa::cluster_capacity_hd256(1 << lg);
                clusters[lg] = cap;
            }
        }
    }
    return choose_splits_rule(kv_len_eff, rows, nkv, nseq, sms, have ? clusters : nullptr);
}

int pgqa_device_status(void)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState *s = nullptr;
    int st = device_state(&s);
    if (st != PGQA_OK)
        return st;
    unsigned int word = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&word, s->err, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PGQA_ERR_CUDA;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(s->err, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return PGQA_ERR_CUDA;
        return (word & pgqa::kErrTileRows) ? PGQA_ERR_TILE_TOO_LONG : PGQA_ERR_DEVICE_TIMEOUT;
    }
    return PGQA_OK;
}

int pgqa_selftest_bounded_wait(void *stream)
{
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState *s = nullptr;
    const int st = device_state(&s);
    if (st != PGQA_OK)
        return st;
    return pgqa::launch_bounded_wait_probe(s->err, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? PGQA_OK
               : PGQA_ERR_CUDA;
}

}  // extern "C"

namespace pgqa {
// Every host-side check of pgqa_attn_decode's arguments, in its order; no CUDA
// call.  PGQA_OK for rows == 0 too (the call then does nothing).
int check_decode_args(const void *o, const void *part, const void *q, const void *k_pool, const void *v_pool,
                      const int32_t *block_table, const int32_t *off, const int32_t *qpos, int rows, int nh,
                      int nkv, int hd, int window, int splits)
{
    if (rows < 0 || nh <= 0 || nkv <= 0 || nh % nkv != 0 || window < 0 || splits < 1)
        return PGQA_ERR_INVALID_ARGUMENT;
    if (hd_index(hd) < 0)
        return PGQA_ERR_UNSUPPORTED_HD;
    if (splits > PGQA_MAX_SPLITS)
        return PGQA_ERR_TOO_MANY_SPLITS;
    if (rows == 0)
        return PGQA_OK;
    if (!o || !q || !k_pool || !v_pool || !block_table || !off || !qpos || (splits > 1 && !part))
        return PGQA_ERR_INVALID_ARGUMENT;
    const int g = nh / nkv;
    const int hsg = (g + kQRows - 1) / kQRows;
    if (rows > 65535 || static_cast<long long>(nkv) * hsg > 65535)
        return PGQA_ERR_INVALID_ARGUMENT;
    if (splits > 1 && static_cast<long long>(rows) * nh > INT_MAX)    // the combine kernel's grid
        return PGQA_ERR_INVALID_ARGUMENT;
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(q, 16) || !aligned(o, 16) ||
        (splits > 1 && !aligned(part, 16)))
        return PGQA_ERR_MISALIGNED;
    return PGQA_OK;
}
}  // namespace pgqa

extern "C" {

int pgqa_attn_decode(void *o, void *part, const void *q, const void *k_pool, const void *v_pool,
                     const int32_t *block_table, const int32_t *off, const int32_t *qpos, const int32_t *kvpos,
                     int rows, int nh, int nkv, int hd, int window, int splits, uint32_t *counters,
                     const int32_t *page_map, void *stream)
{
    const int cs = pgqa::check_decode_args(o, part, q, k_pool, v_pool, block_table, off, qpos, rows, nh, nkv, hd,
                                           window, splits);
    if (cs != PGQA_OK || rows == 0)
        return cs;
    const int hi = hd_index(hd);
    const int g = nh / nkv;
    const int hsg = (g + pgqa::kQRows - 1) / pgqa::kQRows;

    pgqa::LaunchArgs a;
    pgqa::DecodeParams &p = a.p;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.part_o = static_cast<float *>(part);
    p.part_ml = splits > 1 ? reinterpret_cast<float2 *>(static_cast<char *>(part) +
                                                        static_cast<size_t>(rows) * nh * splits * hd * 4)
                           : nullptr;
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.block_table = block_table;
    p.off = off;
    p.qpos = qpos;
    p.kvpos = kvpos;
    p.page_map = page_map;
    // in-kernel merges take up to kGroupSplits splits; more go to the combine
    // kernel, whose loads spread over rows * nh * hd / 128 CTAs
    p.counters = splits <= pgqa::kGroupSplits ? counters : nullptr;
    p.rows = rows;
    p.nh = nh;
    p.nkv = nkv;
    p.window = window;
    p.splits = splits;
    p.g = g;
    p.hsg = hsg;
    p.pack = g <= pgqa::kQRows ? pgqa::kQRows / g : 1;
    p.trace = nullptr;
    p.cluster = 0;
    p.whole_tile_box = 0;
    p.spec_tiles = p.spec_bt_len = p.spec_pm_len = 0;
    p.k_pool = static_cast<const __nv_bfloat16 *>(k_pool);
    p.v_pool = static_cast<const __nv_bfloat16 *>(v_pool);
    a.stream = static_cast<cudaStream_t>(stream);

    // The lock covers set-up and the (asynchronous) launch itself, so the
    // one-time shared-memory attribute is in place before any launch.
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState *s = nullptr;
    int st = device_state(&s);
    if (st != PGQA_OK)
        return st;
    CUtensorMap tk, tv;
    int whole_k = 0, whole_v = 0;
    if ((st = pool_map(k_pool, hd, &tk, &whole_k)) != PGQA_OK || (st = pool_map(v_pool, hd, &tv, &whole_v)) != PGQA_OK)
        return st;
    if (whole_k != whole_v)
        return PGQA_ERR_TENSOR_MAP;
    p.whole_tile_box = whole_k;
    p.err = s->err;
    // tiles that do work: one per packing group of rows (the rows of a group
    // that is packed leave at once), kv head and head subgroup
    const long long live = static_cast<long long>((rows + p.pack - 1) / p.pack) * nkv * hsg;
    p.cluster = p.counters ? on_chip_cluster(s, hi, hd, splits, live) : 0;
    // Launches that merge in the combine kernel (more than 8 splits, or no
    // counters) are long ones.  Their split CTAs prefetch their first pages
    // while the kernel ahead of them in the stream ends: in a loop of calls,
    // the previous call's combine kernel, during which they take the SMs its
    // split CTAs leave.  When nothing ahead is still running, the guess costs
    // a few dependent loads.  One wave of split CTAs at most: later waves
    // start after the wait anyway.
    if (splits > 1 && p.counters == nullptr && live * splits <= 2LL * s->num_sms)
        set_speculation(p, k_pool, v_pool, hd);
    if (g_trace && static_cast<size_t>(splits) * nkv * hsg * rows * pgqa::kTraceEvents * 8 <= g_trace_bytes)
        p.trace = g_trace;
    a.tm_k = &tk;
    a.tm_v = &tv;
    const bool set_attr = !s->attr_set[hi];
    cudaError_t e;
    switch (hd) {
    case 64: e = pgqa::launch_decode_hd64(a, set_attr); break;
    case 128: e = pgqa::launch_decode_hd128(a, set_attr); break;
    case 256: e = pgqa::launch_decode_hd256(a, set_attr); break;
    default: e = pgqa::launch_decode_hd512(a, set_attr); break;
    }
    if (e != cudaSuccess)
        return PGQA_ERR_CUDA;
    s->attr_set[hi] = true;
    return PGQA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------- prefill

int pgqa_prefill_rows_per_tile(int hd)
{
    switch (hd) {
    case 64:
    case 128:
    case 256:
    case 512: return pgqa::kPrefillRowsPerTile;
    default: return PGQA_ERR_UNSUPPORTED_HD;
    }
}

int pgqa_make_tiles(const int32_t *seq, int rows, int rows_per_tile, int32_t *tile_t0, int32_t *tile_tn,
                    int max_tiles)
{
    if (rows < 0 || rows_per_tile < 1 || (rows > 0 && !seq))
        return PGQA_ERR_INVALID_ARGUMENT;
    int n = 0;
    for (int r = 0, len = 0; r < rows; ++r) {
        if (r == 0 || seq[r] != seq[r - 1] || len == rows_per_tile) {
            ++n;
            len = 0;
        }
        ++len;
    }
    if (!tile_t0 && !tile_tn)
        return n;
    if (!tile_t0 || !tile_tn || max_tiles < n)
        return PGQA_ERR_INVALID_ARGUMENT;
    int t = -1;
    for (int r = 0; r < rows; ++r) {
        if (r == 0 || seq[r] != seq[r - 1] || tile_tn[t] == rows_per_tile) {
            ++t;
            tile_t0[t] = r;
            tile_tn[t] = 0;
        }
        ++tile_tn[t];
    }
    return n;
}

namespace {

// pgqa_attn_prefill and, with splits > 1, pgqa_attn_prefill_split: the tiled
// kernel, then (split) the decode combine kernel over the rows' partials.
int prefill_call(void *o, void *part, const void *q, const void *k_pool, const void *v_pool,
                 const int32_t *block_table, const int32_t *off, const int32_t *qpos, const int32_t *kvpos,
                 const int32_t *tile_t0, const int32_t *tile_tn, int ntiles, int rows, int nh, int nkv, int hd,
                 int window, int splits, const int32_t *page_map, void *stream)
{
    if (ntiles < 0 || nh <= 0 || nkv <= 0 || nh % nkv != 0 || window < 0 || splits < 1)
        return PGQA_ERR_INVALID_ARGUMENT;
    if (splits > PGQA_MAX_SPLITS)
        return PGQA_ERR_TOO_MANY_SPLITS;
    const int hi = hd_index(hd);
    if (hi < 0)
        return PGQA_ERR_UNSUPPORTED_HD;
    if (ntiles == 0)
        return PGQA_OK;
    if (!o || !q || !k_pool || !v_pool || !block_table || !off || !qpos || !tile_t0 || !tile_tn)
        return PGQA_ERR_INVALID_ARGUMENT;
    if (splits > 1 && (!part || rows < 1 || static_cast<long long>(rows) * nh > INT_MAX))
        return PGQA_ERR_INVALID_ARGUMENT;
    if (splits > 1 && !aligned(part, 16))
        return PGQA_ERR_MISALIGNED;
    const int g = nh / nkv;
    const int rpt = pgqa_prefill_rows_per_tile(hd);
    const int qr = 128;     // query rows per CTA (pair, at hd 512)
    if (nkv > 65535 || (static_cast<long long>(rpt) * g + qr - 1) / qr > 65535)
        return PGQA_ERR_INVALID_ARGUMENT;
    if (!aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(q, 16) || !aligned(o, 16))
        return PGQA_ERR_MISALIGNED;

    pgqa::PrefillLaunchArgs a;
    pgqa::PrefillParams &p = a.p;
    p.o = static_cast<__nv_bfloat16 *>(o);
    p.q = static_cast<const __nv_bfloat16 *>(q);
    p.block_table = block_table;
    p.off = off;
    p.qpos = qpos;
    p.kvpos = kvpos;
    p.page_map = page_map;
    p.tile_t0 = tile_t0;
    p.tile_tn = tile_tn;
    p.nh = nh;
    p.nkv = nkv;
    p.g = g;
    p.window = window;
    p.rows_per_tile = rpt;
    p.splits = splits;
    p.part_o = splits > 1 ? static_cast<float *>(part) : nullptr;
    p.part_ml = splits > 1 ? reinterpret_cast<float2 *>(static_cast<char *>(part) +
                                                        static_cast<size_t>(rows) * nh * splits * hd * 4)
                           : nullptr;
    a.ntiles = ntiles;
    a.max_tile_rows = rows > 0 ? std::min(rows, rpt) : rpt;
    a.stream = static_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState *s = nullptr;
    int st = device_state(&s);
    if (st != PGQA_OK)
        return st;
    CUtensorMap tk, tv;
    int kind_k = 0, kind_v = 0;
    // The tcgen05 kernel copies K by one box per tile in the halves view and
    // V by one whole-tile box, each of this CTA's dims (all of them, or half at
    // hd 512), or by 64-dim boxes where the driver refuses those views.
    const int box_chunks = hd > 256 ? hd / 128 : hd / 64;
    if ((st = pool_map(k_pool, hd, &tk, &kind_k, kMapHalves, box_chunks)) != PGQA_OK ||
        (st = pool_map(v_pool, hd, &tv, &kind_v, kMapWhole, box_chunks)) != PGQA_OK)
        return st;
    p.whole_tile_box = kind_v == kMapWhole;
    p.k_halves = kind_k == kMapHalves;
    // Q by TMA where g divides the 128-row chunk and a tile can fill a chunk
    // (else, or if the driver refuses the map, by loads from the softmax
    // threads, in the kernel built without that path)
    CUtensorMap tq;
    a.tm_q = (128 % g == 0 && static_cast<long long>(a.max_tile_rows) * g >= 128 &&
              q_map(q, nh, hd, g, &tq) == PGQA_OK)
                 ? &tq
                 : nullptr;
    p.err = s->err;
    a.num_sms = s->num_sms;
    a.tm_k = &tk;
    a.tm_v = &tv;
    const bool set_attr = !s->prefill_attr_set[hi];
    cudaError_t e;
    switch (hd) {
    case 64: e = pgqa::launch_prefill_hd64(a, set_attr); break;
    case 128: e = pgqa::launch_prefill_hd128(a, set_attr); break;
    case 256: e = pgqa::launch_prefill_hd256(a, set_attr); break;
    default: e = pgqa::launch_prefill_hd512(a, set_attr); break;
    }
    if (e != cudaSuccess)
        return PGQA_ERR_CUDA;
    s->prefill_attr_set[hi] = true;
    if (splits > 1) {
        pgqa::DecodeParams c;
        std::memset(&c, 0, sizeof c);
        c.o = p.o;
        c.part_o = p.part_o;
        c.part_ml = p.part_ml;
        c.rows = rows;
        c.nh = nh;
        c.nkv = nkv;
        c.splits = splits;
        c.err = s->err;
        switch (hd) {
        case 64: e = pgqa::launch_combine_hd64(c, a.stream); break;
        case 128: e = pgqa::launch_combine_hd128(c, a.stream); break;
        case 256: e = pgqa::launch_combine_hd256(c, a.stream); break;
        default: e = pgqa::launch_combine_hd512(c, a.stream); break;
        }
        if (e != cudaSuccess)
            return PGQA_ERR_CUDA;
    }
    return PGQA_OK;
}

}  // namespace

int pgqa_attn_prefill(void *o, const void *q, const void *k_pool, const void *v_pool, const int32_t *block_table,
                      const int32_t *off, const int32_t *qpos, const int32_t *kvpos, const int32_t *tile_t0,
                      const int32_t *tile_tn, int ntiles, int nh, int nkv, int hd, int window,
                      const int32_t *page_map, void *stream)
{
    return prefill_call(o, nullptr, q, k_pool, v_pool, block_table, off, qpos, kvpos, tile_t0, tile_tn, ntiles, 0,
                        nh, nkv, hd, window, 1, page_map, stream);
}

int pgqa_prefill_split_count(int kv_len_eff, int rows, int ntiles, int nh, int nkv)
{
    if (kv_len_eff < 1 || rows < 1 || ntiles < 1 || nh < 1 || nkv < 1 || nh % nkv != 0)
        return PGQA_ERR_INVALID_ARGUMENT;
    int sms = 152;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        DeviceState *s = nullptr;
        if (device_state(&s) == PGQA_OK)
            sms = s->num_sms;
    }
    // live work items: tiles x kv heads x 128-row chunks of the average tile
    const long long tile_rows = std::min<long long>((rows + ntiles - 1) / ntiles, 128);
    const long long chunks = (tile_rows * (nh / nkv) + 127) / 128;
    const long long items = static_cast<long long>(ntiles) * nkv * chunks;
    // one wave: as many splits as fill the SMs, each at least two 64-token blocks
    long long s = std::max<long long>(1, sms / items);
    const long long blocks = (kv_len_eff + 63) / 64;
    s = std::min(s, std::max<long long>(1, blocks / 2));
    return static_cast<int>(std::min<long long>(s, PGQA_MAX_SPLITS));
}

int pgqa_prefill_split_count_ex(int kv_len_eff, int rows, int ntiles, int nh, int nkv, int hd)
{
    const int base = pgqa_prefill_split_count(kv_len_eff, rows, ntiles, nh, nkv);
    if (base < 1 || hd != 512)
        return base < 1 ? base : (hd_index(hd) < 0 ? PGQA_ERR_UNSUPPORTED_HD : base);
    // At hd 512 a work item takes a CTA pair, and only so many pairs are
    // resident: beyond one wave of them a second wave doubles a short call.
    // While each split keeps at most 32 blocks, size the splits to one wave.
    int pairs = 0;
    {
        std::lock_guard<std::mutex> lock(g_mutex);
        DeviceState *s = nullptr;
        if (device_state(&s) == PGQA_OK)
            pairs = pgqa::prefill_pair_capacity_hd512();
    }
    const long long tile_rows = std::min<long long>((rows + ntiles - 1) / ntiles, 128);
    const long long items = static_cast<long long>(ntiles) * nkv * ((tile_rows * (nh / nkv) + 127) / 128);
    const long long one_wave = std::max<long long>(1, pairs / items);
    const long long blocks = (kv_len_eff + 63) / 64;
    if (pairs > 0 && one_wave < base && (blocks + one_wave - 1) / one_wave <= 32)
        return static_cast<int>(one_wave);
    return base;
}

int pgqa_attn_prefill_split(void *o, void *part, const void *q, const void *k_pool, const void *v_pool,
                            const int32_t *block_table, const int32_t *off, const int32_t *qpos,
                            const int32_t *kvpos, const int32_t *tile_t0, const int32_t *tile_tn, int ntiles,
                            int rows, int nh, int nkv, int hd, int window, int splits, const int32_t *page_map,
                            void *stream)
{
    return prefill_call(o, part, q, k_pool, v_pool, block_table, off, qpos, kvpos, tile_t0, tile_tn, ntiles, rows,
                        nh, nkv, hd, window, splits, page_map, stream);
}
