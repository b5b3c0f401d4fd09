// Host side of the tensor-core decode for grouped-query heads (decode_tc.cuh): eligibility, the
// tiled-TMA maps of the pool and of q, and the launch.
#include <cstdlib>

#include "decode_tc.cuh"

namespace {

bool tc_enabled() {
    const char *v = std::getenv("PAGEDKV_DECODE_TC");
    return !(v && v[0] == '0');
}

// the MMAs' operand type: the model dtype, or fp16 for E4M3 caches (widened in shared memory)
int operand_dtype(const pkv_cache *c) {
    return c->kv_dtype == PKV_FP8_E4M3 ? (int)PKV_F16 : c->model_dtype;
}

} // namespace

bool pkv_decode_tc_eligible(const pkv_cache *c, int G, int num_seqs) {
    using namespace pkv_decode_tc;
    if (!tc_enabled()) return false;
    if (c->head_dim != D) return false;
    if (G != 2 && G != 4 && G != 8) return false;
    // TMA row coordinates are 32-bit
    if ((int64_t)c->num_blocks * 2 * c->num_kv_heads * c->block_size > 0x7FFFFFFFLL) return false;
    if ((int64_t)num_seqs * 16 > 0x7FFFFFFFLL) return false;
    return smem_bytes(operand_dtype(c), c->kv_dtype == PKV_FP8_E4M3, num_seqs) <= 232448;
}

cudaError_t pkv_decode_tc_launch(const pkv_cache *c, const pkv_decode::Args &a, const void *q, int G,
                                 cudaStream_t st) {
    using namespace pkv_decode_tc;
    CUtensorMap tkv, tq;
    const int mt = c->model_dtype;
    const bool f8 = c->kv_dtype == PKV_FP8_E4M3;
    if (!pkv_tmap_2d(&tq, q, mt, (int64_t)a.num_seqs * a.hq, D, G)) return cudaErrorInvalidValue;
    // the pool: 16-bit caches, one box per (block, K|V, head) tile of bs rows, as
    // [row group][half][8 rows][128 bytes]; E4M3 caches, one box per (block, head) holding its K and
    // its V tile, as [row group][K, V][8 rows][128 codes] (half the copies of one box per tile)
    const int64_t pool_rows = (int64_t)c->num_blocks * 2 * c->num_kv_heads * c->block_size;
    if (!(f8 ? pkv_tmap_kv_pairs_e4m3(&tkv, c->pool, c->num_blocks, c->num_kv_heads, c->block_size)
             : pkv_tmap_rows128_grouped(&tkv, c->pool, mt, pool_rows, c->block_size)))
        return cudaErrorInvalidValue;
    const size_t smem = smem_bytes(operand_dtype(c), f8, a.num_seqs);
    const int grid = c->num_sms;
#define PKV_TC_CASE(GG)                                                                                                \
    if (G == GG) {                                                                                                     \
        if (f8)                                                                                                        \
            return mt == PKV_BF16 ? launch<GG, PKV_BF16, PKV_FP8_E4M3>(tkv, tq, a, grid, smem, st)                     \
                                  : launch<GG, PKV_F16, PKV_FP8_E4M3>(tkv, tq, a, grid, smem, st);                     \
        return mt == PKV_BF16 ? launch<GG, PKV_BF16, PKV_BF16>(tkv, tq, a, grid, smem, st)                             \
                              : launch<GG, PKV_F16, PKV_F16>(tkv, tq, a, grid, smem, st);                              \
    }
    PKV_TC_CASE(2)
    PKV_TC_CASE(4)
    PKV_TC_CASE(8)
#undef PKV_TC_CASE
    return cudaErrorInvalidValue;
}
