// Slot indexing and paged KV append.
//
// Slot indexing: token t of sequence s goes to physical block block_table[s][t / bs] at
// offset t % bs ("Paged KV Cache 与 Packed Sequence", discosf.com, section 2.2).
// Append: the new token's K/V is written at exactly that (block, offset) and nowhere else
// ("PagedAttention 与前缀缓存", 2kiu.com, section 4.1 step 3 and section 6.3).
//
// Both are HBM-bound scatter/gather work: 16-byte vector loads and stores, one thread per
// 16-byte source chunk, consecutive threads on consecutive chunks of a (token, K|V, head)
// row so that every warp moves whole contiguous 256-byte rows.  The fused variant computes
// each token's slot in the same kernel (and still returns the slots), which saves a launch
// per decode step.  All kernels are launched with programmatic dependent launch: they let the
// next kernel in the stream start its launch early and wait for their own predecessor before
// touching global memory.
#include "device_common.cuh"
#include "pkv_internal.h"

namespace {

PKV_DEV int64_t slot_of(const int32_t *__restrict__ tables, int rows, int max_blocks, int s, int p, int bs) {
    if (s < 0 || s >= rows || p < 0) return -1;
    const int lb = p / bs;
    if (lb >= max_blocks) return -1;
    const int b = tables[(int64_t)s * max_blocks + lb];
    return b < 0 ? -1 : (int64_t)b * bs + p % bs;
}

__global__ void slot_mapping_kernel(const int32_t *__restrict__ tables, int rows, int max_blocks,
                                    const int32_t *__restrict__ seq_ids, const int32_t *__restrict__ positions,
                                    int64_t n, int bs, int64_t *__restrict__ out) {
    pdl_trigger();
    pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
        out[i] = slot_of(tables, rows, max_blocks, seq_ids[i], positions[i], bs);
}

struct AppendArgs {
    const uint4 *k, *v;   // [n][Hkv][D] model dtype, viewed as 16-byte chunks
    const int64_t *slots; // given slots (plain append) ...
    const int32_t *tables, *seq_ids, *positions; // ... or computed here (fused append)
    const int32_t *cu, *ctx; // ... or from packed ranges: token j of [cu[i], cu[i+1]) at position ctx[i] + j - cu[i]
                             // (ctx NULL: position j - cu[i])
    int64_t *slots_out;
    int rows, max_blocks;
    char *pool;
    const float *k_scale, *v_scale;
    unsigned int *err;
    int64_t n, num_slots;
    int hkv, bs, chunks_per_row; // chunks_per_row = D / 8
    int64_t tile_elems;          // bs * D
    int d;
};

// KVT: 0 = 16-bit cache (bit copy), 2 = E4M3 cache; MT = model dtype for the E4M3 path;
// MODE: 0 = slots given, 1 = slot from (table, sequence id, position) per token, 2 = sequence and
// position from packed ranges (cu_seqlens, context lengths), then the slot as in mode 1
enum { SLOTS_GIVEN = 0, SLOTS_AT = 1, SLOTS_RANGES = 2 };
constexpr int kAppendThreads = 256;
constexpr int kAppendUnroll = 4; // chunks a thread loads before it stores any

// The slot of token j (mode-specific), or -1 for "skip".
template <int MODE>
PKV_DEV int64_t append_slot(const AppendArgs &a, int64_t j) {
    if constexpr (MODE == SLOTS_AT) {
        return slot_of(a.tables, a.rows, a.max_blocks, a.seq_ids[j], a.positions[j], a.bs);
    } else if constexpr (MODE == SLOTS_RANGES) {
        // sequence: the largest i with cu[i] <= j (a.rows = number of sequences)
        int lo = 0, hi = a.rows;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (a.cu[mid] <= j)
                lo = mid;
            else
                hi = mid;
        }
        const int64_t st = a.cu[lo], en = a.cu[lo + 1];
        const int c0 = a.ctx ? a.ctx[lo] : 0; // no context lengths: every sequence starts at position 0
        const int64_t pos = (int64_t)c0 + (j - st);
        return (j >= st && j < en && c0 >= 0 && pos <= 0x7FFFFFFF)
                   ? slot_of(a.tables, a.rows, a.max_blocks, lo, (int)pos, a.bs)
                   : -1;
    } else {
        return a.slots[j];
    }
}

// Token-major: a pass of the CTA covers whole tokens, tpg = max(1, threads / chunks per token) of
// them, so a token's slot is found once per thread rather than once per 16-byte chunk, and each
// thread issues the loads of up to kAppendUnroll chunks before it stores any of them.
template <int KVT, int MT, int MODE>
__global__ void __launch_bounds__(kAppendThreads) append_kernel(AppendArgs a) {
    pdl_trigger();
    pdl_wait();
    const int row_chunks = a.hkv * a.chunks_per_row; // one (token, K|V) row over all heads
    const int per_token = 2 * row_chunks;
    const int tpg = per_token >= kAppendThreads ? 1 : kAppendThreads / per_token;
    const int lt = tpg > 1 ? (int)threadIdx.x / per_token : 0; // this thread's token in the pass
    const int r0 = tpg > 1 ? (int)threadIdx.x - lt * per_token : (int)threadIdx.x;
    const int rstep = tpg > 1 ? per_token : kAppendThreads;
    if (lt >= tpg) return; // threads past the last whole token of a pass
    for (int64_t j = (int64_t)blockIdx.x * tpg + lt; j < a.n; j += (int64_t)gridDim.x * tpg) {
        const int64_t slot = append_slot<MODE>(a, j);
        if (MODE != SLOTS_GIVEN && r0 == 0 && a.slots_out) a.slots_out[j] = slot;
        if (slot < 0) continue;
        if (slot >= a.num_slots) {
            if (r0 == 0) set_error(a.err, PKV_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / a.bs;
        const int off = static_cast<int>(slot - blk * a.bs);
        // element index of (blk, kv = 0, h = 0, off, 0) in the [NB][2][Hkv][bs][D] pool
        const int64_t e0 = blk * 2 * a.hkv * a.tile_elems + (int64_t)off * a.d;
        const uint4 *ksrc = a.k + j * row_chunks, *vsrc = a.v + j * row_chunks;
        for (int rb = r0; rb < per_token; rb += kAppendUnroll * rstep) {
            uint4 src[kAppendUnroll];
            int64_t dst[kAppendUnroll];
            int kvs[kAppendUnroll], hs[kAppendUnroll];
#pragma unroll
            for (int u = 0; u < kAppendUnroll; ++u) {
                const int r = rb + u * rstep;
                dst[u] = -1;
                if (r < per_token) {
                    const int kv = r >= row_chunks ? 1 : 0;
                    const int hc = r - kv * row_chunks;
                    const int h = hc / a.chunks_per_row;
                    const int c = hc - h * a.chunks_per_row;
                    src[u] = (kv ? vsrc : ksrc)[hc];
                    dst[u] = e0 + (int64_t)(kv * a.hkv + h) * a.tile_elems + c * 8;
                    kvs[u] = kv;
                    hs[u] = h;
                }
            }
#pragma unroll
            for (int u = 0; u < kAppendUnroll; ++u) {
                if (dst[u] < 0) continue;
                if constexpr (KVT != PKV_FP8_E4M3) {
                    reinterpret_cast<uint4 *>(a.pool)[dst[u] / 8] = src[u];
                } else {
                    float f[8];
                    cvt8<MT>(src[u], f);
                    const float sc = (kvs[u] ? a.v_scale : a.k_scale)[hs[u]];
                    uint2 o;
                    o.x = e4m3x2_from_f32(__fdiv_rn(f[0], sc), __fdiv_rn(f[1], sc)) |
                          (e4m3x2_from_f32(__fdiv_rn(f[2], sc), __fdiv_rn(f[3], sc)) << 16);
                    o.y = e4m3x2_from_f32(__fdiv_rn(f[4], sc), __fdiv_rn(f[5], sc)) |
                          (e4m3x2_from_f32(__fdiv_rn(f[6], sc), __fdiv_rn(f[7], sc)) << 16);
                    reinterpret_cast<uint2 *>(a.pool)[dst[u] / 8] = o;
                }
            }
        }
    }
}

inline int grid_for(int64_t work, int threads, int num_sms) {
    const int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = (int64_t)num_sms * 16;
    return static_cast<int>(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
}

AppendArgs base_args(pkv_cache *c, const void *k, const void *v, int64_t n) {
    AppendArgs a{};
    a.k = static_cast<const uint4 *>(k);
    a.v = static_cast<const uint4 *>(v);
    a.pool = static_cast<char *>(c->pool);
    a.k_scale = c->k_scale;
    a.v_scale = c->v_scale;
    a.err = c->err;
    a.n = n;
    a.num_slots = c->num_blocks * c->block_size;
    a.hkv = c->num_kv_heads;
    a.bs = c->block_size;
    a.chunks_per_row = c->head_dim / 8;
    a.tile_elems = (int64_t)c->block_size * c->head_dim;
    a.d = c->head_dim;
    return a;
}

template <int MODE>
cudaError_t launch_append_t(pkv_cache *c, const AppendArgs &a, cudaStream_t st) {
    // one CTA pass per tpg tokens (see append_kernel), up to 8 resident CTAs per SM
    const int per_token = 2 * a.hkv * a.chunks_per_row;
    const int tpg = per_token >= kAppendThreads ? 1 : kAppendThreads / per_token;
    const int64_t passes = (a.n + tpg - 1) / tpg;
    const int64_t cap = (int64_t)c->num_sms * 8;
    const dim3 grid((unsigned)(passes < 1 ? 1 : (passes > cap ? cap : passes)));
    PkvTimer timer(c, PKV_KIND_APPEND, st);
    cudaError_t e;
    if (c->kv_dtype != PKV_FP8_E4M3)
        e = pdl_launch(append_kernel<PKV_F16, PKV_F16, MODE>, grid, dim3(kAppendThreads), 0, st, a);
    else if (c->model_dtype == PKV_F16)
        e = pdl_launch(append_kernel<PKV_FP8_E4M3, PKV_F16, MODE>, grid, dim3(kAppendThreads), 0, st, a);
    else
        e = pdl_launch(append_kernel<PKV_FP8_E4M3, PKV_BF16, MODE>, grid, dim3(kAppendThreads), 0, st, a);
    g_pkv_launches++;
    return e;
}

} // namespace

cudaError_t launch_slot_mapping(const int32_t *tables, int rows, int max_blocks, const int32_t *seq_ids,
                                const int32_t *positions, int64_t n, int bs, int64_t *out, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    int dev = 0, sms = 148;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const cudaError_t e = pdl_launch(slot_mapping_kernel, dim3(grid_for(n, 256, sms)), dim3(256), 0, st, tables, rows,
                                     max_blocks, seq_ids, positions, n, bs, out);
    g_pkv_launches++;
    return e;
}

cudaError_t launch_append(pkv_cache *c, const void *k, const void *v, const int64_t *slots, int64_t n,
                          cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    AppendArgs a = base_args(c, k, v, n);
    a.slots = slots;
    return launch_append_t<SLOTS_GIVEN>(c, a, st);
}

cudaError_t launch_append_at(pkv_cache *c, const void *k, const void *v, const int32_t *tables, int rows,
                             int max_blocks, const int32_t *seq_ids, const int32_t *positions, int64_t n,
                             int64_t *slots_out, cudaStream_t st) {
    if (n == 0) return cudaSuccess;
    AppendArgs a = base_args(c, k, v, n);
    a.tables = tables;
    a.rows = rows;
    a.max_blocks = max_blocks;
    a.seq_ids = seq_ids;
    a.positions = positions;
    a.slots_out = slots_out;
    return launch_append_t<SLOTS_AT>(c, a, st);
}

cudaError_t launch_append_ranges(pkv_cache *c, const void *k, const void *v, const int32_t *tables, int num_seqs,
                                 int max_blocks, const int32_t *cu, const int32_t *ctx, int64_t n, cudaStream_t st) {
    if (n == 0 || num_seqs <= 0) return cudaSuccess;
    AppendArgs a = base_args(c, k, v, n);
    a.tables = tables;
    a.rows = num_seqs;
    a.max_blocks = max_blocks;
    a.cu = cu;
    a.ctx = ctx;
    return launch_append_t<SLOTS_RANGES>(c, a, st);
}
