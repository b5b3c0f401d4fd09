// Host-side internals shared by the translation units of the library.
#pragma once

#include <nvtx3/nvToolsExt.h>
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <mutex>
#include <vector>

#include "pagedkv.h"

struct pkv_cache {
    int device = 0;
    int64_t num_blocks = 0;
    int block_size = 0, num_kv_heads = 0, head_dim = 0;
    pkv_dtype kv_dtype = PKV_F16, model_dtype = PKV_F16;
    int elem_bytes = 2;
    // pool: [num_blocks][2][Hkv][bs][D] elements
    void *pool = nullptr;
    int64_t pool_bytes = 0;
    int64_t tile_bytes = 0;   // one (block, K|V, head) tile: bs * D * elem
    float *k_scale = nullptr; // [Hkv] device (FP8 only)
    float *v_scale = nullptr;
    unsigned int *err = nullptr; // device error word
    // split-K workspace of the decode
    float *ws = nullptr;
    int64_t ws_bytes = 0;
    // work list of the packed prefill (item count, next-item counter, (sequence, query tile) pairs)
    int *plan = nullptr;
    int64_t plan_bytes = 0;
    int num_sms = 0;
    // profiling
    bool profiling = false;
    unsigned profile_kinds = 0; // bit (1 << PKV_KIND_*)
    int profile_every = 1;       // bracket every n-th launch of a kind (see kv_cache_profile_start_sampled)
    int64_t profile_seen[8] = {}; // launches of each kind since the profile started
    struct Ev {
        int kind;
        cudaEvent_t a, b;
    };
    std::vector<Ev> events;
    std::vector<cudaEvent_t> event_pool;
    std::mutex mu;
};

enum { PKV_KIND_DECODE = 0, PKV_KIND_PREFILL = 1, PKV_KIND_APPEND = 2, PKV_KIND_MERGE = 3, PKV_KIND_COPY = 4 };

// status helpers (api.cu)
int pkv_fail(int status, const char *fmt, ...);
int pkv_cuda_fail(cudaError_t e, const char *what);
extern std::atomic<int64_t> g_pkv_launches;

// profiling bracket around one main-kernel launch (api.cu)
struct PkvTimer {
    pkv_cache *c;
    int kind;
    cudaStream_t st;
    cudaEvent_t a = nullptr, b = nullptr;
    PkvTimer(pkv_cache *c_, int kind_, cudaStream_t st_);
    ~PkvTimer();
};

// Launch with the programmatic-stream-serialization attribute (the kernel itself calls
// pdl_wait() before it touches memory a previous kernel may use).
template <typename... KArgs, typename... Args>
cudaError_t pdl_launch(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// launchers (one per translation unit); return cudaError_t of the launch
cudaError_t launch_slot_mapping(const int32_t *tables, int rows, int max_blocks, const int32_t *seq_ids,
                                const int32_t *positions, int64_t n, int bs, int64_t *out, cudaStream_t st);
cudaError_t launch_append(pkv_cache *c, const void *k, const void *v, const int64_t *slots, int64_t n,
                          cudaStream_t st);
cudaError_t launch_append_at(pkv_cache *c, const void *k, const void *v, const int32_t *tables, int rows,
                             int max_blocks, const int32_t *seq_ids, const int32_t *positions, int64_t n,
                             int64_t *slots_out, cudaStream_t st);

// append of packed token ranges: token j of [cu[i], cu[i+1]) goes to position ctx[i] + j - cu[i]
// of sequence i (the tail of a prompt after its cached prefix)
cudaError_t launch_append_ranges(pkv_cache *c, const void *k, const void *v, const int32_t *tables, int num_seqs,
                                 int max_blocks, const int32_t *cu, const int32_t *ctx, int64_t n, cudaStream_t st);

// whole-block copies (blocks.cu): pair i copies block src_ids[i] (or i) of `src` to block
// dst_ids[i] (or i) of `dst`; both regions are made of blocks of the cache's block size
cudaError_t launch_copy_blocks(pkv_cache *c, const void *src, const int32_t *src_ids, int64_t src_blocks, void *dst,
                               const int32_t *dst_ids, int64_t dst_blocks, int64_t n, cudaStream_t st);

struct CascadePrefixLaunch;
struct DecodeLaunch {
    const void *q;
    void *out;
    const int32_t *tables;
    const int32_t *lens;
    int max_blocks, num_seqs, num_q_heads;
    float scale;
    int split_blocks; // blocks per split
    int max_splits;
    float *ws_o;      // [S*Hq*max_splits][D]
    float *ws_ml;     // [S*Hq*max_splits][2]
    // cascade decode: blocks of the shared prefix (covered by launch_cascade_prefix) and the workspace
    // slot of the first suffix split; 0 and 0 for a plain decode
    int start_block = 0, slot0 = 0;
    // cascade decode: the prefix kernel, launched after the decode kernel and before the merge (its
    // plan kernel went before the decode)
    const CascadePrefixLaunch *prefix = nullptr;
};

// One NVTX range per C-ABI call that launches GPU work, named after the call: a profiler attached
// to the process shows the library's calls on its timeline (NVTX v3 is header-only; with no tool
// attached a range costs a branch).
struct PkvRange {
    explicit PkvRange(const char *name) { nvtxRangePushA(name); }
    ~PkvRange() { nvtxRangePop(); }
    PkvRange(const PkvRange &) = delete;
    PkvRange &operator=(const PkvRange &) = delete;
};
#define PKV_RANGE(name) PkvRange pkv_nvtx_range_(name)

// The prefix phase of a cascade decode (prefill.cu): the decode queries of every sequence against the
// first prefix_tokens tokens of table row 0, cut into splits of split_tokens keys (a multiple of 64);
// split p of (sequence s, query head h) goes to workspace slot p of row s * Hq + h.
struct CascadePrefixLaunch {
    const void *q; // [S][Hq][D]
    const int32_t *tables;
    int max_blocks, num_seqs, num_q_heads, prefix_tokens, split_tokens, max_splits;
    float scale;
    float *ws_o, *ws_ml;
};
// part 1: the plan kernel; part 2: the prefix kernel.  The prefix kernel does not wait for the kernel
// before it until it exits, so that kernel must be one that lets it launch only after waiting for its
// own predecessors (the suffix decode, launched between the two parts by launch_decode).
cudaError_t launch_cascade_prefix(pkv_cache *c, const CascadePrefixLaunch &p, cudaStream_t st, int part);
// keys per prefix split of the cascade's prefix phase (a multiple of 64)
int cascade_split_tokens(const pkv_cache *c, int num_seqs, int num_q_heads, int prefix_tokens);
int64_t decode_workspace_floats(const pkv_cache *c, int num_seqs, int num_q_heads, int max_splits);
// Sequences one decode launch takes at most (its kernels hold a per-sequence table in shared memory);
// a call with more runs its sequences in consecutive launches of this many, which reuse one workspace
// (stream order: each launch waits for the previous launch's merge before it writes partials).
int decode_seqs_per_launch(const pkv_cache *c, int G);
// Runs the decode described by d (d.ws_o sized for min(num_seqs, decode_seqs_per_launch) sequences)
// as consecutive launches of at most decode_seqs_per_launch sequences each (api.cu).
cudaError_t launch_decode_chunked(pkv_cache *c, DecodeLaunch d, cudaStream_t st);
// The no-alloc decode's fixed scratch: makes it resident on the current device and records its device
// address (noalloc.cu); kv_cache_create calls it, so the array is in place before a caller's allocator
// takes the rest of the device memory.
int pkv_noalloc_scratch_prepare(int device);
int decode_split_blocks(const pkv_cache *c);
int cascade_suffix_split_blocks(const pkv_cache *c); // blocks per split of a cascade's suffix decode
cudaError_t launch_decode(pkv_cache *c, const DecodeLaunch &d, cudaStream_t st);
// tensor-core decode for grouped-query heads (decode_tc.cu)
namespace pkv_decode {
struct Args;
}
bool pkv_decode_tc_eligible(const pkv_cache *c, int G, int num_seqs);
cudaError_t pkv_decode_tc_launch(const pkv_cache *c, const pkv_decode::Args &a, const void *q, int G, cudaStream_t st);

struct PrefillLaunch {
    const void *q, *k, *v;
    void *out;
    const int32_t *cu;
    const int32_t *ctx; // cached tokens per sequence (paged mode: K/V read from the pool), or NULL
    const int32_t *tables;
    int num_seqs, max_seqlen, max_blocks, num_q_heads;
    int64_t total_tokens;
    float scale;
};
cudaError_t launch_prefill(pkv_cache *c, const PrefillLaunch &p, cudaStream_t st);

// Tiled-TMA map of a row-major fp16/bf16 matrix [rows][cols]: box = 64 columns x box_rows rows,
// 128-byte swizzle, out-of-range elements read as zero (prefill.cu).
bool pkv_tmap_2d(CUtensorMap *m, const void *base, int mt, int64_t rows, int64_t cols, int box_rows);
// rows of 128 16-bit elements (a multiple of 8 of them) as a 4-D map whose box of box_rows rows (a
// multiple of 8) lands as [row group of 8][64-element half][8 rows][128 bytes], 128-byte swizzled:
// one copy per block tile where two 2-D boxes (one per half) were needed
bool pkv_tmap_rows128_grouped(CUtensorMap *m, const void *base, int mt, int64_t rows, int box_rows);
// E4M3 pool: one box = the K and the V tile of one (block, KV head), bs rows of 128 codes each,
// landing as [slot / 8][K, V][8 rows][128 bytes], 128-byte swizzled; coordinates
// (0, 0, 0, head * bs / 8, block) (prefill.cu)
bool pkv_tmap_kv_pairs_e4m3(CUtensorMap *m, const void *pool, int64_t num_blocks, int hkv, int bs);
