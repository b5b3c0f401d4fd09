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

// target resident CTAs per SM (shared-memory budget per CTA follows from it)
int ctas_per_sm() { return env_int("PAGEDKV_DECODE_CTAS", 4); }

using DecodeFn = cudaError_t (*)(const pkv_decode::Args &, int, int, int, size_t, cudaStream_t, bool);
using OccFn = int (*)(int, int, size_t);

void pick(const pkv_cache *c, DecodeFn *fn, OccFn *occ) {
    if (c->kv_dtype == PKV_F16) {
        *fn = pkv_decode_f16;
        *occ = pkv_decode_occupancy_f16;
    } else if (c->kv_dtype == PKV_BF16) {
        *fn = pkv_decode_bf16;
        *occ = pkv_decode_occupancy_bf16;
    } else if (c->model_dtype == PKV_F16) {
        *fn = pkv_decode_fp8_f16;
        *occ = pkv_decode_occupancy_fp8_f16;
    } else {
        *fn = pkv_decode_fp8_bf16;
        *occ = pkv_decode_occupancy_fp8_bf16;
    }
}

} // namespace

// cascade decode: the prefix kernel runs between the suffix decode and the merge, overlapping the
// decode's last units (the decode lets it launch early; it waits for the decode before it exits)
static cudaError_t launch_prefix_between(pkv_cache *c, const DecodeLaunch &d, cudaStream_t st) {
    if (!d.prefix) return cudaSuccess;
    PkvTimer timer(c, PKV_KIND_PREFILL, st);
    return launch_cascade_prefix(c, *d.prefix, st, 2);
}

int decode_split_blocks(const pkv_cache *c) {
    const int tokens = env_int("PAGEDKV_SPLIT_TOKENS", 256);
    const int b = tokens / c->block_size;
    return b > 0 ? b : 1;
}

int cascade_suffix_split_blocks(const pkv_cache *c) {
    // the suffixes of a cascade batch are short (a few hundred tokens): 128-token splits give the
    // CTAs twice as many, half as long units, which evens out their finish times (prefix13b: step
    // 101.5-102.3 -> 100.2-101.5 us); the tensor-core decode keeps its own longer splits
    const int tokens = env_int("PAGEDKV_CASCADE_SUFFIX_TOKENS", 128);
    const int b = tokens / c->block_size;
    return b > 0 ? b : 1;
}

int decode_seqs_per_launch(const pkv_cache *c, int G) {
    // Both decode kernels keep a per-sequence unit table (3 ints a sequence) in shared memory: the
    // CUDA-core kernel takes up to kMaxSeqs sequences a launch; the tensor-core kernel, whose stage
    // rings fill nearly all of shared memory, fewer (the largest multiple of 64 that still fits).
    int n = pkv_decode::kMaxSeqs;
    if (pkv_decode_tc_eligible(c, G, 64))
        while (n > 64 && !pkv_decode_tc_eligible(c, G, n)) n -= 64;
    return n;
}

int64_t decode_workspace_floats(const pkv_cache *c, int num_seqs, int num_q_heads, int max_splits) {
    // partial o [rows][D] and (m, l) [rows][2], rows = S * Hq * max_splits; only needed when splits > 1
    if (max_splits <= 1) return 0;
    const int64_t rows = (int64_t)num_seqs * num_q_heads * max_splits;
    return rows * (c->head_dim + 2);
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
    a.ws_ml = d.ws_o ? d.ws_o + (int64_t)d.num_seqs * d.num_q_heads * d.max_splits * c->head_dim : nullptr;
    a.err = c->err;
    a.num_blocks = c->num_blocks;
    a.tile_bytes = static_cast<int>(c->tile_bytes);
    // a stage of the CUDA-core kernel holds at most PAGEDKV_DECODE_STAGE_BYTES of K plus V (8 KB:
    // 16 tokens at fp16 and D=128), so that bs=32 blocks go in two stages and as many CTAs fit an
    // SM as with bs=16 (the consumer warps' per-stage work is latency bound; more warps hide it)
    {
        const int64_t cap = env_int("PAGEDKV_DECODE_STAGE_BYTES", 8192);
        int t = c->block_size;
        while (t > 8 && (t & 1) == 0 && 2 * (int64_t)t * c->head_dim * c->elem_bytes > cap) t >>= 1;
        a.sub_tokens = t;
        a.sub_bytes = static_cast<int>((int64_t)t * c->head_dim * c->elem_bytes);
    }
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
    a.start_block = d.start_block;
    a.slot0 = d.slot0;

    DecodeFn fn;
    OccFn occ;
    pick(c, &fn, &occ);
    cudaError_t e;
    if (pkv_decode_tc_eligible(c, G, d.num_seqs)) {
        a.nstages = 0;
        // longer splits than the CUDA-core kernel's: a unit then spans several 128-token MMA steps,
        // which spreads the per-unit work (Q load, epilogue, partial write) over more bytes; the
        // workspace, sized for the default split, only gets more room.  E4M3 caches take twice
        // the tokens: a step of one-byte codes costs about half the time of a 16-bit one, while the
        // per-unit work does not shrink (on log-normal lengths of median 500, 1024-token splits run
        // ~5 % faster than 512-token ones for E4M3 and ~4 % slower for bf16)
        const int tc_default = c->kv_dtype == PKV_FP8_E4M3 ? 1024 : 512;
        const int tc_blocks = env_int("PAGEDKV_SPLIT_TOKENS_TC", tc_default) / c->block_size;
        if (tc_blocks > a.split_blocks) a.split_blocks = tc_blocks;
        {
            PkvTimer timer(c, PKV_KIND_DECODE, st);
            e = pkv_decode_tc_launch(c, a, d.q, G, st);
            g_pkv_launches++;
        }
        if (e != cudaSuccess) return e;
        if ((e = launch_prefix_between(c, d, st)) != cudaSuccess) return e;
        PkvTimer timer(c, PKV_KIND_MERGE, st);
        e = fn(a, c->head_dim, G, 0, 0, st, true);
        g_pkv_launches++;
        return e;
    }
    // stages: fill the per-CTA shared-memory budget
    const size_t fixed = smem_bytes(c->head_dim, G, 0, a.sub_bytes, d.num_seqs);
    const size_t per_stage = smem_bytes(c->head_dim, G, 1, a.sub_bytes, d.num_seqs) - fixed;
    // CTAs per SM: the target, or fewer when registers allow fewer (grouped heads); the stage ring
    // then takes that many CTAs' share of shared memory, so the bytes in flight per SM stay high
    int want = ctas_per_sm();
    {
        const int fit = occ(c->head_dim, G, smem_bytes(c->head_dim, G, kConsumerWarps, a.sub_bytes, d.num_seqs));
        if (fit >= 1 && fit < want) want = fit;
    }
    const size_t budget = (size_t)(233472 / want) - 1024;
    int nst = budget > fixed ? static_cast<int>((budget - fixed) / per_stage) : 0;
    nst = env_int("PAGEDKV_DECODE_STAGES", nst);
    // a whole number of stages per consumer warp (see the tile-to-warp rule in the kernel)
    nst -= nst % kConsumerWarps;
    if (nst > 32) nst = 32;
    if (nst < kConsumerWarps) nst = kConsumerWarps;
    a.nstages = nst;
    const size_t smem = smem_bytes(c->head_dim, G, nst, a.sub_bytes, d.num_seqs);
    int per_sm = occ(c->head_dim, G, smem);
    if (per_sm < 1) per_sm = 1;
    const int grid = c->num_sms * per_sm;
    {
        PkvTimer timer(c, PKV_KIND_DECODE, st);
        e = fn(a, c->head_dim, G, grid, smem, st, false);
        g_pkv_launches++;
    }
    if (e != cudaSuccess) return e;
    if ((e = launch_prefix_between(c, d, st)) != cudaSuccess) return e;
    {
        PkvTimer timer(c, PKV_KIND_MERGE, st);
        e = fn(a, c->head_dim, G, 0, 0, st, true);
        g_pkv_launches++;
    }
    return e;
}
