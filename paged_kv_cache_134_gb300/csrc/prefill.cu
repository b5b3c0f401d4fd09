// Host side of the tensor-core attention of prefill_impl.cuh: the work-list kernel, the tiled-TMA maps
// and the launches of the packed prefill, the prefill over a cached prefix and the cascade decode's
// prefix phase.  The attention kernel itself is instantiated in prefill_packed.cu, prefill_paged.cu
// and prefill_cascade.cu (one translation unit each, compiled in parallel).
#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "prefill_impl.cuh"

namespace pkv_prefill {

constexpr int kPlanThreads = 1024;

// in-place inclusive prefix sum of x[0, n) by the whole CTA (kPlanThreads threads)
PKV_DEV void cta_inclusive_scan(int *x, int n, int *warp_sums) {
    const int per = (n + kPlanThreads - 1) / kPlanThreads;
    const int b = min((int)threadIdx.x * per, n), e = min(b + per, n);
    int own = 0;
    for (int i = b; i < e; ++i) own += x[i];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int v = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_sums[w] = v;
    __syncthreads();
    if (w == 0) {
        int u = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, u, o);
            if (lane >= o) u += t;
        }
        warp_sums[lane] = u;
    }
    __syncthreads();
    int run = v - own + (w > 0 ? warp_sums[w - 1] : 0);
    for (int i = b; i < e; ++i) {
        run += x[i];
        x[i] = run;
    }
    __syncthreads();
}

// key tiles of pair p of sequence i (its two query tiles' key tiles added), from the item decoding
PKV_DEV int pair_cost(const Args &a, int i, int p) {
    const Item it = decode_item(a, i, p, 0);
    return it.t[0].n + it.t[1].n;
}

// The work list: every (sequence, pair of query tiles), heaviest first (a counting sort on the pair's
// key tiles, clamped to the histogram's range), so that the persistent CTAs, which take items in list
// order, end together.  The order inside one cost class is whatever the atomics give; it only decides
// which CTA computes an item, never what the item computes.  Also resets the next-item counter the
// attention kernel draws from.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const Args a) {
    extern __shared__ int sh[];
    const int R = a.cost_bins;
    int *hist = sh; // hist[c] = #{pairs of cost c}, then #{pairs of cost <= c}
    int *cnt = sh + R;
    int *warp_sums = sh + 2 * R;
    pdl_trigger();
    pdl_wait();
    if (a.nps > 0) {
        // cascade: the items are the (tile of query rows, split pair) pairs, taken in order
        if (threadIdx.x == 0) {
            a.plan[0] = ((a.num_seqs + BM - 1) / BM) * ((a.nps + 1) / 2);
            a.plan[1] = 0;
        }
        return;
    }
    for (int x = threadIdx.x; x < R; x += kPlanThreads) {
        hist[x] = 0;
        cnt[x] = 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < a.num_seqs; i += kPlanThreads) {
        const int np = (seq_tiles(a, i, true) + 1) / 2;
        for (int p = 0; p < np; ++p) atomicAdd(&hist[min(pair_cost(a, i, p), R - 1)], 1);
    }
    __syncthreads();
    cta_inclusive_scan(hist, R, warp_sums); // hist[c] = #{pairs of cost <= c}
    const int total = hist[R - 1];
    int2 *list = reinterpret_cast<int2 *>(a.plan + 4);
    for (int i = threadIdx.x; i < a.num_seqs; i += kPlanThreads) {
        const int np = (seq_tiles(a, i, false) + 1) / 2;
        for (int p = 0; p < np; ++p) {
            const int c = min(pair_cost(a, i, p), R - 1);
            // descending cost: the pairs of cost c come after every pair of higher cost
            const int pos = total - hist[c] + atomicAdd(&cnt[c], 1);
            if (pos < a.plan_cap) list[pos] = make_int2(i, p);
        }
    }
    if (threadIdx.x == 0) {
        // sequences whose rows overlap make more pairs than the tokens allow: reported, list cut short
        if (total > a.plan_cap) set_error(a.err, PKV_DEVERR_CU_SEQLENS);
        a.plan[0] = (int)min((int64_t)total, a.plan_cap);
        a.plan[1] = 0;
    }
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    });
    return fn;
}

// 2-D view [rows][cols] of a row-major matrix; box = 64 columns x box_rows rows, 128-byte swizzle.
// mt = PKV_FP8_E4M3: one-byte elements, boxes of 128 columns (one 128-byte swizzle row).
bool make_map(CUtensorMap *m, const void *base, int mt, int64_t rows, int64_t cols, int box_rows) {
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    const bool bytes = mt == PKV_FP8_E4M3;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * (bytes ? 1 : 2)};
    const cuuint32_t box[2] = {bytes ? 128u : 64u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = bytes                ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : mt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUresult r = enc(m, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// E4M3 pool rows [rows][cols] of bytes, unswizzled: one box = box_rows whole rows (cols <= 256, a
// multiple of 16), landing as box_rows consecutive rows of cols bytes
bool make_code_map(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, int box_rows) {
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols};
    const cuuint32_t box[2] = {(cuuint32_t)cols, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

cudaError_t launch_plan(const Args &a, cudaStream_t st) {
    const int smem = (2 * a.cost_bins + 32) * (int)sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return pdl_launch(plan_kernel, dim3(1), dim3(kPlanThreads), smem, st, a);
}

// the pool's map for the attention's key loads and the packed mode's block stores: 16-bit rows of D
// elements, box = bs rows x 64 dims, swizzled; E4M3 rows of D codes, box = bs whole rows, unswizzled
bool pool_map(CUtensorMap *m, const pkv_cache *c) {
    const int64_t pool_rows = c->num_blocks * 2 * c->num_kv_heads * c->block_size;
    if (c->kv_dtype == PKV_FP8_E4M3) return make_code_map(m, c->pool, pool_rows, c->head_dim, c->block_size);
    return make_map(m, c->pool, c->model_dtype, pool_rows, c->head_dim, c->block_size);
}

template <int MODE, bool KV8>
cudaError_t dispatch(int D, int mt, const Maps &m, const Args &a, int64_t max_ctas, int num_sms, cudaStream_t st) {
    if (D == 128)
        return mt == PKV_BF16 ? launch_attn<128, PKV_BF16, MODE, KV8>(m, a, max_ctas, num_sms, st)
                              : launch_attn<128, PKV_F16, MODE, KV8>(m, a, max_ctas, num_sms, st);
    if (D == 64)
        return mt == PKV_BF16 ? launch_attn<64, PKV_BF16, MODE, KV8>(m, a, max_ctas, num_sms, st)
                              : launch_attn<64, PKV_F16, MODE, KV8>(m, a, max_ctas, num_sms, st);
    return cudaErrorInvalidValue;
}

int lg2(int x) {
    int l = 0;
    while ((1 << l) < x) ++l;
    return l;
}

Args base_args(pkv_cache *c, float scale) {
    Args a{};
    a.pool = static_cast<char *>(c->pool);
    a.k_scale = c->k_scale;
    a.v_scale = c->v_scale;
    a.err = c->err;
    a.num_blocks = c->num_blocks;
    a.tile_elems = (int64_t)c->block_size * c->head_dim;
    a.hkv = c->num_kv_heads;
    a.bs = c->block_size;
    a.lg_bs = lg2(c->block_size);
    a.scale_log2 = scale * 1.4426950408889634f;
    return a;
}

} // namespace pkv_prefill

bool pkv_tmap_2d(CUtensorMap *m, const void *base, int mt, int64_t rows, int64_t cols, int box_rows) {
    return pkv_prefill::make_map(m, base, mt, rows, cols, box_rows);
}

bool pkv_tmap_kv_pairs_e4m3(CUtensorMap *m, const void *pool, int64_t num_blocks, int hkv, int bs) {
    using namespace pkv_prefill;
    EncodeFn enc = encode_fn();
    if (!enc || bs % 8 || bs / 8 > 256 || num_blocks < 1 || (int64_t)hkv * bs / 8 > 0x7FFFFFFFLL) return false;
    // the pool's E4M3 rows [(block, K|V, head, slot)][128 codes] seen as (code, slot % 8, K|V,
    // head * bs / 8 + slot / 8, block): a box of (128, 8, 2, bs / 8, 1) at (0, 0, 0, head * bs / 8,
    // block) is the K tile and the V tile of one (block, head) in one copy, landing as
    // [slot / 8][K, V][8 rows][128 bytes] (each 8-row group of K followed by the same rows of V)
    const cuuint64_t row = 128, kv = (cuuint64_t)hkv * bs * row;
    const cuuint64_t dims[5] = {128, 8, 2, (cuuint64_t)hkv * bs / 8, (cuuint64_t)num_blocks};
    const cuuint64_t strides[4] = {row, kv, 8 * row, 2 * kv};
    const cuuint32_t box[5] = {128u, 8u, 2u, (cuuint32_t)(bs / 8), 1u};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 5, const_cast<void *>(pool), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool pkv_tmap_rows128_grouped(CUtensorMap *m, const void *base, int mt, int64_t rows, int box_rows) {
    using namespace pkv_prefill;
    EncodeFn enc = encode_fn();
    if (!enc || rows % 8 || box_rows % 8 || box_rows > 256 * 8) return false;
    // rows of 128 16-bit elements = 256 bytes, seen as (64 elements, row in its group of 8, half, group):
    // a box of (64, 8, 2, box_rows / 8) lands as [group][half][8 rows][128 bytes]
    const cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)(rows / 8)};
    const cuuint64_t strides[3] = {256, 128, 2048};
    const cuuint32_t box[4] = {64u, 8u, 2u, (cuuint32_t)(box_rows / 8)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = mt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUresult r = enc(m, dt, 4, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static cudaError_t ensure_plan(pkv_cache *c, int64_t bytes) {
    if (bytes <= c->plan_bytes) return cudaSuccess;
    if (c->plan) cudaFree(c->plan);
    c->plan = nullptr;
    c->plan_bytes = 0;
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&c->plan), (size_t)bytes);
    if (e != cudaSuccess) {
        c->plan = nullptr;
        return e;
    }
    c->plan_bytes = bytes;
    return cudaSuccess;
}

cudaError_t launch_prefill(pkv_cache *c, const PrefillLaunch &p, cudaStream_t st) {
    using namespace pkv_prefill;
    if (p.total_tokens <= 0) return cudaSuccess;
    const int D = c->head_dim;
    const int mt = c->model_dtype;
    const bool kv8 = c->kv_dtype == PKV_FP8_E4M3;
    Args a = base_args(c, p.scale);
    a.k = static_cast<const char *>(p.k);
    a.v = static_cast<const char *>(p.v);
    a.out = p.out;
    a.cu = p.cu;
    a.ctx = p.ctx;
    a.tables = p.tables;
    a.total_tokens = p.total_tokens;
    a.num_seqs = p.num_seqs;
    a.max_seqlen = p.max_seqlen;
    a.max_blocks = p.max_blocks;
    a.hq = p.num_q_heads;
    a.write_pool = kv8 ? 0 : 1;
    // (sequence, pair of query tiles) items: sum_i ceil(n_i / 2 BM) <= T / 2 BM + num_seqs
    const int64_t tiles_max = ((int64_t)p.max_seqlen + BM - 1) / BM;
    a.npairs_max = (int)((tiles_max + 1) / 2);
    const int64_t items = std::min<int64_t>((int64_t)a.npairs_max * p.num_seqs, p.total_tokens / (2 * BM) + p.num_seqs);
    if (items == 0) return cudaSuccess;
    if (items * p.num_q_heads > 0x7FFFFFFF) return cudaErrorNotSupported;
    // cost classes of the heaviest-first list: a pair's key tiles, at most 2 ceil((ctx + n) / BN); the
    // histogram's range is clamped (the order then only approximates heaviest first)
    const int64_t max_keys = p.ctx ? (int64_t)p.max_blocks * c->block_size : (int64_t)p.max_seqlen;
    a.cost_bins = (int)std::min<int64_t>(2 * ((max_keys + BN - 1) / BN) + 2, 16384);
    const int64_t plan_bytes = (4 + 2 * items) * (int64_t)sizeof(int);
    a.plan_cap = items;
    cudaError_t e = ensure_plan(c, plan_bytes);
    if (e != cudaSuccess) return e;
    a.plan = c->plan;
    // the pool as rows [(block, K|V, head, slot)][D] for the key loads and the tiled stores of whole
    // blocks; row coordinates are 32-bit
    const int64_t pool_rows = c->num_blocks * 2 * c->num_kv_heads * c->block_size;
    if (pool_rows > 0x7FFFFFFFLL) return cudaErrorNotSupported;
    Maps m;
    if (!make_map(&m.q, p.q, mt, p.total_tokens, (int64_t)p.num_q_heads * D, BM) ||
        !make_map(&m.k, p.k, mt, p.total_tokens, (int64_t)c->num_kv_heads * D, BN) ||
        !make_map(&m.v, p.v, mt, p.total_tokens, (int64_t)c->num_kv_heads * D, BN) || !pool_map(&m.pool, c) ||
        !make_map(&m.out, p.out, mt, p.total_tokens, (int64_t)p.num_q_heads * D, BM))
        return cudaErrorInvalidValue;
    if (p.ctx || kv8) {
        // A cached prefix: the new tokens' K/V go to their slots first, then attention reads every key
        // through the block table.  An FP8 cache: the packed prefill's K/V write is the append's
        // (fp32 division by the head's scale, E4M3 rounding), and the attention reads the packed k, v.
        e = launch_append_ranges(c, p.k, p.v, p.tables, p.num_seqs, p.max_blocks, p.cu, p.ctx, p.total_tokens, st);
        if (e != cudaSuccess) return e;
    }
    PkvTimer timer(c, PKV_KIND_PREFILL, st);
    e = launch_plan(a, st);
    g_pkv_launches++;
    if (e != cudaSuccess) return e;
    const int64_t max_ctas = items * p.num_q_heads;
    if (!p.ctx)
        e = dispatch<MODE_PACKED, false>(D, mt, m, a, max_ctas, c->num_sms, st);
    else if (kv8)
        e = dispatch<MODE_PAGED, true>(D, mt, m, a, max_ctas, c->num_sms, st);
    else
        e = dispatch<MODE_PAGED, false>(D, mt, m, a, max_ctas, c->num_sms, st);
    g_pkv_launches++;
    return e;
}

int cascade_split_tokens(const pkv_cache *c, int num_seqs, int num_q_heads, int prefix_tokens) {
    using namespace pkv_prefill;
    if (const char *v = std::getenv("PAGEDKV_CASCADE_SPLIT_TOKENS")) {
        // keys per prefix split, for tuning sweeps (rounded up to whole 128-key tiles)
        const int x = std::atoi(v);
        if (x > 0) return (x + BN - 1) / BN * BN;
    }
    // The prefix phase runs as one wave of items where it can: as many split pairs per (query-row tile,
    // head) as leave every item a CTA (one per SM; a split past one wave makes the whole phase wait for
    // a second), each split of at least 256 keys so that an item's fixed costs (Q load, epilogue,
    // partial write) stay small next to its key tiles, in whole 128-key tiles.
    const int64_t rows = (int64_t)((num_seqs + BM - 1) / BM) * num_q_heads;
    const int64_t pairs = std::max<int64_t>(1, (int64_t)c->num_sms / std::max<int64_t>(rows, 1));
    const int64_t nps = 2 * pairs;
    int64_t split = (prefix_tokens + nps - 1) / nps;
    split = std::max<int64_t>(split, 256);
    return (int)((split + BN - 1) / BN * BN);
}

cudaError_t launch_cascade_prefix(pkv_cache *c, const CascadePrefixLaunch &p, cudaStream_t st, int part) {
    using namespace pkv_prefill;
    if (p.num_seqs <= 0 || p.prefix_tokens <= 0) return cudaSuccess;
    const int D = c->head_dim;
    const int mt = c->model_dtype;
    const bool kv8 = c->kv_dtype == PKV_FP8_E4M3;
    Args a = base_args(c, p.scale);
    a.tables = p.tables;
    a.total_tokens = p.num_seqs;
    a.num_seqs = p.num_seqs;
    a.max_blocks = p.max_blocks;
    a.hq = p.num_q_heads;
    a.cost_bins = 1;
    a.ws_o = p.ws_o;
    a.ws_ml = p.ws_ml;
    a.max_splits = p.max_splits;
    a.prefix_tokens = p.prefix_tokens;
    a.split_tokens = p.split_tokens;
    a.nps = (p.prefix_tokens + p.split_tokens - 1) / p.split_tokens;
    const int64_t pairs = (int64_t)((p.num_seqs + BM - 1) / BM) * ((a.nps + 1) / 2);
    if (pairs * p.num_q_heads > 0x7FFFFFFF) return cudaErrorNotSupported;
    cudaError_t e = ensure_plan(c, 64);
    if (e != cudaSuccess) return e;
    a.plan = c->plan;
    const int64_t pool_rows = c->num_blocks * 2 * c->num_kv_heads * c->block_size;
    if (pool_rows > 0x7FFFFFFFLL) return cudaErrorNotSupported;
    // q [S][Hq][D] as rows of sequences: a box of 128 sequences x 64 dims of one head
    Maps m; // cascade: q and the pool (k, v, out unused)
    if (!make_map(&m.q, p.q, mt, p.num_seqs, (int64_t)p.num_q_heads * D, BM) || !pool_map(&m.pool, c))
        return cudaErrorInvalidValue;
    if (part == 1) {
        e = launch_plan(a, st);
        g_pkv_launches++;
        return e;
    }
    m.k = m.v = m.out = m.pool;
    e = kv8 ? dispatch<MODE_CASCADE, true>(D, mt, m, a, pairs * p.num_q_heads, c->num_sms, st)
            : dispatch<MODE_CASCADE, false>(D, mt, m, a, pairs * p.num_q_heads, c->num_sms, st);
    g_pkv_launches++;
    return e;
}
