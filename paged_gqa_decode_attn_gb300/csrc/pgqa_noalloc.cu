// pgqa_attn_decode_noalloc: the split-KV decode with its scratch in this
// library's own static device memory instead of caller-provided buffers.
//
// Some callers cannot hand the library device scratch: a plugin loaded into
// a host runtime that owns every device allocation and exposes no allocator
// to it, or a caller on a path where it must not call cudaMalloc (which can
// synchronise the device) and has no pool to borrow from.  For them the
// partials and merge counters live in the fixed array below, which every GPU
// that loads the library holds until the process exits.  The caller still
// provides all inputs and the output.
//
// This entry point allocates nothing: no cudaMalloc, no cudaFree, no
// allocating library routine.  It checks its arguments as pgqa_attn_decode
// does, clears the merge counters it will use with cudaMemsetAsync on the
// caller's stream, then enqueues the ordinary pgqa_attn_decode with merge
// counters, pointed at the static scratch.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "pgqa.h"

namespace pgqa {
int current_context_id(unsigned long long *id);    // pgqa_api.cu
int check_decode_args(const void *o, const void *part, const void *q, const void *k_pool, const void *v_pool,
                      const int32_t *block_table, const int32_t *off, const int32_t *qpos, int rows, int nh,
                      int nkv, int hd, int window, int splits);
}  // namespace pgqa

namespace {

constexpr size_t kCounterBytes = static_cast<size_t>(PGQA_NOALLOC_MAX_COUNTERS) * sizeof(uint32_t);
constexpr size_t kScratchBytes = kCounterBytes + static_cast<size_t>(PGQA_NOALLOC_MAX_PART_BYTES);

// The shared scratch: merge counters first, then the split partials.  In host
// code this name is only a stand-in for the device array; its device address
// comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
unsigned char *g_scratch_ptr[kMaxDevices] = {};
unsigned long long g_scratch_ctx[kMaxDevices] = {};   // the context each address belongs to

// Device address of the scratch on the current device; looked up by the first
// call on each device, with that device current, and again after the device's
// context has been replaced (cudaDeviceReset destroys it, and the module may
// then load at another address).
int scratch_address(unsigned char **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return PGQA_ERR_CUDA;
    unsigned long long ctx = 0;
    if (pgqa::current_context_id(&ctx) != PGQA_OK)
        return PGQA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (g_scratch_ptr[dev] == nullptr || g_scratch_ctx[dev] != ctx) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return PGQA_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<unsigned char *>(ptr);
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_ptr[dev];
    return PGQA_OK;
}

}  // namespace

extern "C" int pgqa_attn_decode_noalloc(void *o, const void *q, const void *k_pool, const void *v_pool,
                                        const int32_t *block_table, const int32_t *off, const int32_t *qpos,
                                        const int32_t *kvpos, int rows, int nh, int nkv, int hd, int window,
                                        int splits, const int32_t *page_map, void *stream)
{
    if (rows < 0 || nh <= 0 || nkv <= 0 || nh % nkv != 0 || splits < 1)
        return PGQA_ERR_INVALID_ARGUMENT;
    if (rows == 0)
        return PGQA_OK;
    const size_t part_bytes = pgqa_decode_part_bytes(rows, nh, splits, hd);
    const size_t counters = pgqa_decode_counter_count(rows, nh, nkv);
    if (part_bytes > static_cast<size_t>(PGQA_NOALLOC_MAX_PART_BYTES) ||
        counters > static_cast<size_t>(PGQA_NOALLOC_MAX_COUNTERS))
        return PGQA_ERR_NOALLOC_TOO_LARGE;

    // every other check of pgqa_attn_decode, before any CUDA call (part: an
    // aligned host stand-in for the static scratch, which is 256-byte aligned)
    alignas(16) static const unsigned char part_stand_in[16] = {};
    int st = pgqa::check_decode_args(o, part_stand_in, q, k_pool, v_pool, block_table, off, qpos, rows, nh, nkv, hd,
                                     window, splits);
    if (st != PGQA_OK)
        return st;
    unsigned char *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != PGQA_OK)
        return st;
    uint32_t *cnt = reinterpret_cast<uint32_t *>(scratch);
    void *part = scratch + kCounterBytes;

    // The counters keep whatever the previous call left; they must start at zero.
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(cnt, 0, counters * sizeof(uint32_t), s) != cudaSuccess)
        return PGQA_ERR_CUDA;
    return pgqa_attn_decode(o, part, q, k_pool, v_pool, block_table, off, qpos, kvpos, rows, nh, nkv, hd, window,
                            splits, cnt, page_map, stream);
}
