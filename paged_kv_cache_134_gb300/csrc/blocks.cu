// Whole-block copies of the paged pool: copy-on-write and swap.
//
// What it computes ("PagedAttention 与前缀缓存", 2kiu.com, section 2.2: production managers add
// copy-on-write for prefix blocks shared by beam search or parallel sampling, and swap a
// preempted request's block contents out to CPU memory; section 4.3 step 3: a shared block is
// never rewritten in place, the path that diverges gets its own copy; section 5.2: swapping
// frees GPU blocks for other requests): for i < n, destination block i := source block i,
// all of it.  In the pool layout [block][K|V][head][slot][dim] one block is a single
// contiguous run of 2 * Hkv * bs * D * elt bytes, so a block copy is a contiguous move.
//
// HBM-bound gather/scatter.  Work items are (block pair, 16 KB chunk); CTAs of 256 threads take
// them in a grid-stride loop and move 4 x 16 bytes per thread with streaming (evict-first)
// loads and stores, all four loads issued before the first store.  A block id outside its pool
// skips the pair and sets PKV_DEVERR_BLOCK_ID.  Programmatic dependent launch as elsewhere.
#include <algorithm>

#include "device_common.cuh"
#include "pkv_internal.h"

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;
constexpr int64_t kChunksPerItem = kThreads * kUnroll; // 16-byte chunks per work item (16 KB)

struct CopyArgs {
    const char *src;
    const int32_t *src_ids; // NULL: pair i reads block i of `src`
    int64_t src_blocks;
    char *dst;
    const int32_t *dst_ids; // NULL: pair i writes block i of `dst`
    int64_t dst_blocks;
    int64_t n, block_bytes; // block_bytes % 16 == 0
    unsigned int *err;
};

__global__ void __launch_bounds__(kThreads) copy_blocks_kernel(const CopyArgs a) {
    pdl_trigger();
    pdl_wait();
    const int64_t chunks = a.block_bytes / 16;
    const int64_t items_per_block = (chunks + kChunksPerItem - 1) / kChunksPerItem;
    const int64_t total = a.n * items_per_block;
    for (int64_t w = blockIdx.x; w < total; w += gridDim.x) {
        const int64_t i = w / items_per_block, part = w - i * items_per_block;
        const int64_t sb = a.src_ids ? (int64_t)a.src_ids[i] : i;
        const int64_t db = a.dst_ids ? (int64_t)a.dst_ids[i] : i;
        if (sb < 0 || sb >= a.src_blocks || db < 0 || db >= a.dst_blocks) {
            if (threadIdx.x == 0 && part == 0) set_error(a.err, PKV_DEVERR_BLOCK_ID);
            continue;
        }
        const uint4 *s = reinterpret_cast<const uint4 *>(a.src + sb * a.block_bytes) + part * kChunksPerItem;
        uint4 *d = reinterpret_cast<uint4 *>(a.dst + db * a.block_bytes) + part * kChunksPerItem;
        const int64_t left = chunks - part * kChunksPerItem;
        const int64_t lim = left < kChunksPerItem ? left : kChunksPerItem;
        uint4 x[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t c = threadIdx.x + u * kThreads;
            if (c < lim) x[u] = __ldcs(s + c);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int64_t c = threadIdx.x + u * kThreads;
            if (c < lim) __stcs(d + c, x[u]);
        }
    }
}

} // namespace

cudaError_t launch_copy_blocks(pkv_cache *c, const void *src, const int32_t *src_ids, int64_t src_blocks, void *dst,
                               const int32_t *dst_ids, int64_t dst_blocks, int64_t n, cudaStream_t st) {
    CopyArgs a;
    a.src = static_cast<const char *>(src);
    a.src_ids = src_ids;
    a.src_blocks = src_blocks;
    a.dst = static_cast<char *>(dst);
    a.dst_ids = dst_ids;
    a.dst_blocks = dst_blocks;
    a.n = n;
    a.block_bytes = c->pool_bytes / c->num_blocks;
    a.err = c->err;
    const int64_t items = n * ((a.block_bytes / 16 + kChunksPerItem - 1) / kChunksPerItem);
    const int64_t grid = std::max<int64_t>(1, std::min<int64_t>(items, (int64_t)c->num_sms * 8));
    PkvTimer timer(c, PKV_KIND_COPY, st);
    g_pkv_launches++;
    return pdl_launch(copy_blocks_kernel, dim3((unsigned)grid), dim3(kThreads), 0, st, a);
}
