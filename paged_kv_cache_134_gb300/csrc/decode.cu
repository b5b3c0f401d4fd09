// Host side of the paged decode: split size, stage count, grid, workspace, launches.
#include <cstdlib>

#include "decode_impl.cuh"

namespace {

int env_int(const char *name, int dflt) {
    const char *v = std::getenv(name);
    if (!v || !*v) return dflt;
    const int x = std::atoi(v);
    return x > 0 ? x : dflt;
}

PkvDecodeFn pick(const pkv_cache *c) {
    if (c->kv_dtype == PKV_F16) return pkv_decode_f16;
    if (c->kv_dtype == PKV_BF16) return pkv_decode_bf16;
    return c->model_dtype == PKV_F16 ? pkv_decode_fp8_f16 : pkv_decode_fp8_bf16;
}

} // namespace

int decode_split_blocks(const pkv_cache *c) {
    // a unit's block ids must fit one per lane of a warp
    const int tokens = env_int("PAGEDKV_SPLIT_TOKENS", 256);
    const int b = tokens / c->block_size;
    return b < 1 ? 1 : (b > 32 ? 32 : b);
}

int64_t decode_workspace_floats(const pkv_cache *c, int num_seqs, int num_q_heads, int max_splits) {
    // partial o [rows][D], (m, l) [rows][2] with rows = S * Hq * max_splits, then S * Hkv int counters;
    // only needed when a sequence can have more than one split
    if (max_splits <= 1) return 0;
    const int64_t rows = (int64_t)num_seqs * num_q_heads * max_splits;
    return rows * (c->head_dim + 2) + (int64_t)num_seqs * c->num_kv_heads;
}

cudaError_t launch_decode(pkv_cache *c, const DecodeLaunch &d, cudaStream_t st) {
    using namespace pkv_decode;
    const int G = d.num_q_heads / c->num_kv_heads;
    Args a;
    a.q = d.q;
    a.out = d.out;
    a.pool = static_cast<const char *>(c->pool);
    a.k_scale = c->k_scale;
    a.v_scale = c->v_scale;
    a.tables = d.tables;
    a.lens = d.lens;
    a.ws_o = d.ws_o;
    const int64_t rows = (int64_t)d.num_seqs * d.num_q_heads * d.max_splits;
    a.ws_ml = d.ws_o ? d.ws_o + rows * c->head_dim : nullptr;
    a.counters = d.ws_o ? reinterpret_cast<int *>(a.ws_ml + 2 * rows) : nullptr;
    a.err = c->err;
    a.num_blocks = c->num_blocks;
    a.tile_bytes = static_cast<int>(c->tile_bytes);
    a.kv_stride = (int64_t)c->num_kv_heads * c->tile_bytes;
    a.blk_stride = 2 * a.kv_stride;
    a.max_blocks = d.max_blocks;
    a.num_seqs = d.num_seqs;
    a.hq = d.num_q_heads;
    a.hkv = c->num_kv_heads;
    a.bs = c->block_size;
    a.split_blocks = d.split_blocks;
    a.max_splits = d.max_splits;
    a.qk_scale_log2 = d.scale * 1.4426950408889634f;

    const PkvDecodeFn fn = pick(c);
    // per-warp ring: at least 16 KB (2 stages minimum); 4 warps per CTA when a warp's ring is <= 16 KB,
    // else 2, so that at least 3 CTAs fit an SM's shared memory
    const int stage = 2 * a.tile_bytes;
    int nst = env_int("PAGEDKV_DECODE_STAGES", (16384 + stage - 1) / stage);
    if (nst < 2) nst = 2;
    if (nst > 16) nst = 16;
    a.nstages = nst;
    const int nw = (size_t)nst * stage <= 16384 ? kMaxWarps : 2;
    const size_t smem = smem_bytes(nw, nst, a.tile_bytes, d.num_seqs);
    int per_sm = 0;
    fn(a, c->head_dim, G, 0, nw * 32, smem, st, &per_sm);
    if (per_sm < 1) per_sm = 1;
    const int grid = c->num_sms * per_sm;
    PkvTimer timer(c, PKV_KIND_DECODE, st);
    const cudaError_t e = fn(a, c->head_dim, G, grid, nw * 32, smem, st, nullptr);
    g_pkv_launches++;
    return e;
}
