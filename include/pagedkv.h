/*
 * pagedkv.h -- C ABI of the GB300 (sm_103a) paged KV cache library.
 *
 * What it computes (the passages each call restates are named per call):
 *   a paged KV cache is one flat device pool cut into num_blocks equal blocks of
 *   block_size tokens; each sequence owns a block table whose entry i names the
 *   physical block holding its logical block i ("PagedAttention 与前缀缓存",
 *   2kiu.com, sections 2.1-2.2).  Token t of sequence s lives in physical block
 *   block_table[s][t / block_size] at offset t % block_size ("Paged KV Cache 与
 *   Packed Sequence", discosf.com, section 2.2).
 *
 * Conventions shared by every call
 *   - Every pointer argument except the cache handle and the outputs of
 *     kv_cache_view / kv_cache_check_error / kv_cache_profile_read is a DEVICE
 *     pointer owned by the caller, 16-byte aligned for q/k/v/out, valid until the
 *     work queued on `stream` has finished.  The library owns only what a cache
 *     handle holds: the block pool, the FP8 scales, a device error word and the
 *     split-K workspace of the decode.
 *   - `stream` is a cudaStream_t passed as void*; 0 is the legacy default stream.
 *     Every call only enqueues work on it and returns; nothing synchronises except
 *     kv_cache_check_error and kv_cache_profile_read.
 *   - Dtypes: PKV_F16 / PKV_BF16 / PKV_FP8_E4M3.  q, k, v and out are in the
 *     cache's model dtype (fp16 or bf16); the pool is in its KV dtype.
 *   - Return value: PKV_OK or a negative pkv_status; pkv_last_error() gives a
 *     message for the calling thread's last failure.  Host-side validation fails
 *     before anything is enqueued.  Data that only the device sees (block ids,
 *     slots, lengths, cu_seqlens) is checked in the kernels: the offending element
 *     is skipped, a bit is or-ed into the cache's device error word, and the
 *     kernel carries on; nothing traps.
 *   - Supported shapes: head_dim in {64, 128}; block_size in {8, 16, 32};
 *     num_q_heads / num_kv_heads in {1, 2, 4, 8}.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_cache *pkv_cache_t; /* opaque; created by kv_cache_create */

typedef enum { PKV_F16 = 0, PKV_BF16 = 1, PKV_FP8_E4M3 = 2 } pkv_dtype;

typedef enum {
    PKV_OK = 0,
    PKV_EINVAL = -1,       /* bad argument (null pointer, size, alignment, dtype mix) */
    PKV_ENOMEM = -2,       /* device allocation failed */
    PKV_ECUDA = -3,        /* a CUDA runtime call or launch failed */
    PKV_EUNSUPPORTED = -4, /* shape outside the supported set */
    PKV_EDEVICE = -5       /* kv_cache_check_error found device-side errors */
} pkv_status;

/* bits of the device error word */
#define PKV_DEVERR_BLOCK_ID 1u   /* a needed block-table entry was outside [0, num_blocks) */
#define PKV_DEVERR_SLOT 2u       /* an append slot was >= num_blocks * block_size */
#define PKV_DEVERR_LENGTH 4u     /* a length needed more than max_blocks_per_seq blocks */
#define PKV_DEVERR_CU_SEQLENS 8u /* cu_seqlens decreasing, or a length above max_seqlen */
#define PKV_DEVERR_TIMEOUT 16u   /* a bounded wait inside a kernel gave up */

/* Create a cache: cudaMalloc a pool of num_blocks blocks, each holding K and V of
 * block_size tokens x num_kv_heads heads x head_dim, in kv_dtype (zero-filled).
 * model_dtype is the dtype of q/k/v/out used with this cache; it must equal
 * kv_dtype unless kv_dtype is PKV_FP8_E4M3.  The pool is the "flat device pool of
 * equal blocks" of 2kiu.com section 2.2 / discosf.com section 2.1.  Pool layout
 * (see kv_cache_view): [num_blocks][2 = K,V][num_kv_heads][block_size][head_dim],
 * so one (block, K|V, head) tile is block_size*head_dim contiguous elements.
 * On failure *out is untouched. */
int kv_cache_create(int64_t num_blocks, int block_size, int num_kv_heads, int head_dim, pkv_dtype kv_dtype,
                    pkv_dtype model_dtype, pkv_cache_t *out);

/* Free everything the handle owns (synchronises the device first).  NULL is a no-op. */
int kv_cache_destroy(pkv_cache_t cache);

/* FP8 caches: copy per-KV-head fp32 scales (device arrays of num_kv_heads floats) into
 * the cache.  Stored code = E4M3(fp32(x) / scale[head]), rounded to nearest-even and
 * saturated to +-448; readers multiply the code's value by the scale (the one-byte
 * cache of 2kiu.com section 1.1).  Scales must be finite and > 0; EINVAL for other caches. */
int kv_cache_set_scales(pkv_cache_t cache, const float *k_scale, const float *v_scale, void *stream);

/* Describe the pool for tests and initialisation: *base = device address of the pool,
 * strides_elems = element strides of the (block, K|V, head, offset, dim) axes,
 * *num_bytes = pool size in bytes.  The library keeps ownership. */
int kv_cache_view(pkv_cache_t cache, void **base, int64_t strides_elems[5], int64_t *num_bytes);

/* Pre-size the decode split-K workspace for up to max_seqs x max_q_heads rows and tables
 * of max_blocks_per_seq entries, so that later decode calls allocate nothing (a batch larger
 * than one launch takes needs only one launch's rows: the launches share the workspace). */
int kv_cache_reserve(pkv_cache_t cache, int max_seqs, int max_q_heads, int max_blocks_per_seq);

/* Synchronise the device, return the device error word's bits in *device_code and clear
 * it.  Returns PKV_EDEVICE when any bit was set, PKV_OK otherwise. */
int kv_cache_check_error(pkv_cache_t cache, int *device_code);

/* Self-test of the kernels' bounded waits (discosf.com section 5.1 and 2kiu.com section 6.1: a
 * failure must degrade, not hang or crash).  Enqueues one small kernel that waits on an mbarrier
 * nothing ever arrives on, with the same wait routines every kernel uses (spinning and
 * suspend-hint forms), for limit_ns nanoseconds (1 .. 1e9); both give up and set
 * PKV_DEVERR_TIMEOUT in the cache's error word, which kv_cache_check_error then reports.  No
 * memory besides that word is touched, nothing traps, and the cache stays usable. */
int kv_cache_selftest_wait_timeout(pkv_cache_t cache, uint64_t limit_ns, void *stream);

/* Message for the calling thread's most recent non-OK return ("" if none). */
const char *pkv_last_error(void);

/* Slot indexing (discosf.com section 2.2; 2kiu.com section 4.1 step 3):
 *   slot_mapping[i] = block_tables[seq_ids[i]][positions[i] / block_size] * block_size
 *                     + positions[i] % block_size                       (int64)
 * or -1 when seq_ids[i] is outside [0, num_rows), positions[i] < 0, the logical block is
 * >= max_blocks_per_seq, or the table entry is negative.
 * block_tables: int32 [num_rows][max_blocks_per_seq], row-major.  seq_ids, positions:
 * int32 [num_tokens].  slot_mapping: int64 [num_tokens] (written).  Exact integer work. */
int paged_slot_mapping(const int32_t *block_tables, int num_rows, int max_blocks_per_seq, const int32_t *seq_ids,
                       const int32_t *positions, int64_t num_tokens, int block_size, int64_t *slot_mapping,
                       void *stream);

/* Paged KV append (2kiu.com section 4.1 step 3 and section 6.3; discosf.com section 4.3
 * step 2): for each token j with slot = slot_mapping[j] >= 0, write k[j] and v[j]
 * ([num_tokens][num_kv_heads][head_dim], model dtype) into block slot / block_size at
 * offset slot % block_size.  fp16/bf16 caches store the bits unchanged; FP8 caches store
 * E4M3(fp32(x) / scale[head]) (see kv_cache_set_scales).  Negative slots are padding and
 * skipped; slots >= num_blocks*block_size are skipped and set PKV_DEVERR_SLOT.  Two
 * tokens with the same slot in one call: which one lands is unspecified. */
int paged_kv_append(pkv_cache_t cache, const void *k, const void *v, const int64_t *slot_mapping,
                    int64_t num_tokens, void *stream);

/* Slot indexing and paged KV append in one launch: for each token j, slot_j is computed as in
 * paged_slot_mapping from (block_tables, seq_ids[j], positions[j]) and k[j], v[j] are written as in
 * paged_kv_append.  slot_mapping, when not NULL, receives the int64 slots (the same values
 * paged_slot_mapping returns).  This is the decode step's "write the new token at its block
 * offset" (discosf.com section 4.3 steps 1-2) without a separate indexing launch. */
int paged_kv_append_at(pkv_cache_t cache, const void *k, const void *v, const int32_t *block_tables, int num_rows,
                       int max_blocks_per_seq, const int32_t *seq_ids, const int32_t *positions, int64_t num_tokens,
                       int64_t *slot_mapping, void *stream);

/* Paged decode attention (2kiu.com section 2.3: walk the block table, mask the tail
 * block by the true length; section 3.3: prefix blocks are read per sequence):
 *   out[s][h] = sum_{t < L_s} softmax_t(scale * q[s][h] . K_t) V_t,  L_s = context_lens[s],
 * K_t/V_t read from block block_tables[s][t / block_size], offset t % block_size, KV head
 * h / (num_q_heads / num_kv_heads).  q, out: [num_seqs][num_q_heads][head_dim] model dtype;
 * block_tables: int32 [num_seqs][max_blocks_per_seq]; entries past ceil(L_s/block_size)
 * are never read.  L_s == 0 gives a zero row.  fp32 accumulation and softmax; the output
 * is rounded to the model dtype (nearest-even).  Runs a split-K pass over block-aligned chunks
 * of each sequence plus a merge; split boundaries depend only on L_s, so results do not depend
 * on block placement.  Any num_seqs: a batch larger than one launch takes (1024 sequences, or
 * fewer for the tensor-core kernel of grouped-query heads, whose shared memory holds fewer) runs
 * as consecutive launches of that many sequences on the stream, sharing one workspace sized for
 * a launch.  The workspace grows (cudaMalloc) on demand unless kv_cache_reserve covered the call. */
int paged_decode_attention(const void *q, pkv_cache_t cache, const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens, int num_seqs, int num_q_heads, float scale, void *out,
                           void *stream);

/* paged_decode_attention without any device-memory allocation.  The pages have no counterpart:
 * this entry point exists for callers that cannot let a library allocate, e.g. a serving engine
 * that hands nearly all device memory to its own allocator (its KV pool is sized to fill the GPU)
 * or that cannot afford the device-wide synchronisation cudaMalloc/cudaFree may cause.
 * Same arguments, results and errors as paged_decode_attention, but the split-K partials live in
 * one fixed 16 MiB array compiled into the library instead of the cache's workspace; nothing is
 * allocated, by CUDA or otherwise.  The array becomes resident on a device (and its device address
 * is looked up, one cudaGetSymbolAddress made with that device current) when kv_cache_create makes
 * a cache there, so create the cache before handing the rest of the device memory to another
 * allocator; it then stays until the process exits.  A cudaDeviceReset destroys every cache; the
 * next kv_cache_create on the device repeats the lookup.  The kernels' own code is loaded by CUDA on
 * their first launch (lazy module loading), which can allocate a little device memory once: make one
 * warm-up call (or run with CUDA_MODULE_LOADING=EAGER) before the memory is handed out.
 * A call whose partials for one launch do not fit (n x Hq x ceil(max_blocks_per_seq / split
 * blocks) x (D + 2) floats > 16 MiB, n = min(num_seqs, sequences per launch); with the default
 * 256-token splits, e.g., 32 sequences x 32 heads x 4096-token tables need 9 MB) returns PKV_EINVAL
 * with the sizes in pkv_last_error().  Every call shares the array: calls whose work can overlap
 * on the GPU (different streams, or different host threads) race on it and must be serialised by
 * the caller.  Nothing in the array has to start at zero; each call writes every partial before it
 * reads it. */
int paged_decode_attention_noalloc(const void *q, pkv_cache_t cache, const int32_t *block_tables,
                                   int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                   int num_q_heads, float scale, void *out, void *stream);

/* Cascade decode for a batch that shares a prefix (2kiu.com section 3.3: with a prefix cache many
 * requests share prefix blocks, and decode still reads them; section 6.4: decode-bound batches with
 * a high hit rate): same result as paged_decode_attention, but the first shared_prefix_len tokens,
 * which every table must name with the same blocks (those of table row 0), are read once per
 * (query head, prefix split) for the whole batch instead of once per sequence (splits sized so that
 * the prefix work fits one wave of resident CTAs).  Their attention runs on the tensor cores as a
 * matrix product of all the batch's queries with the prefix keys; the tokens past the prefix go
 * through the split-K decode, and the prefix kernel runs alongside that decode's last work units
 * (it reads nothing the decode writes); one merge combines both.  shared_prefix_len:
 * a multiple of block_size, at most max_blocks_per_seq * block_size, and at most every context
 * length (a shorter sequence sets PKV_DEVERR_LENGTH); 0 makes this paged_decode_attention.
 * fp16/bf16 and FP8 caches (E4M3 prefix codes are widened exactly to the model dtype in shared
 * memory, the per-head scales fold into the softmax scale and the split partials).  The prefix's
 * split partials are rounded like any split (fp32), so outputs agree with paged_decode_attention to
 * the decode tolerance, not bit for bit.  The tensor-core prefix phase takes two prefix splits of
 * one 128-sequence tile per item. */
int paged_decode_attention_cascade(const void *q, pkv_cache_t cache, const int32_t *block_tables,
                                   int max_blocks_per_seq, const int32_t *context_lens, int num_seqs, int num_q_heads,
                                   int shared_prefix_len, float scale, void *out, void *stream);

/* Packed causal prefill (discosf.com sections 3.1-3.3 and 4.2): sequences packed back to
 * back, sequence i owning rows [cu_seqlens[i], cu_seqlens[i+1]):
 *   out[cu_i + r][h] = sum_{c <= r} softmax_c(scale * q[cu_i + r][h] . k[cu_i + c][g]) v[cu_i + c][g]
 * with g = h / (num_q_heads / num_kv_heads); no attention across sequences.  The same call
 * writes every token's k/v into the cache at block_tables[i][r / block_size], offset
 * r % block_size (the bytes paged_kv_append would write).  q, out: [T][num_q_heads][head_dim];
 * k, v: [T][num_kv_heads][head_dim] (model dtype), T = total_tokens = cu_seqlens[num_seqs]
 * (passed from the host because the tensor maps of the loads need it); cu_seqlens: int32
 * [num_seqs + 1], non-decreasing, cu_seqlens[0] = 0; max_seqlen >= every length.  A sequence
 * whose bounds break these rules is skipped and sets PKV_DEVERR_CU_SEQLENS.  Q.K^T and P.V run on
 * the tensor cores (tcgen05, fp32 accumulation in tensor memory), two 128-row query tiles of one
 * (sequence, head) per work item sharing each 128-key K/V tile; P is rounded to the model dtype for
 * P.V (bf16: a hi + lo pair).  FP8 caches: the attention reads the packed k, v as given, and the
 * cache write is paged_kv_append's (E4M3 of fp32(x) / scale[head], the same bytes), issued as a
 * separate launch before it. */
int packed_prefill_attention(const void *q, const void *k, const void *v, const int32_t *cu_seqlens, int num_seqs,
                             int max_seqlen, int64_t total_tokens, const int32_t *block_tables,
                             int max_blocks_per_seq, pkv_cache_t cache, int num_q_heads, float scale, void *out,
                             void *stream);

/* Prefill of a prompt's tail over its cached prefix (2kiu.com section 4.3 steps 2-4: the blocks a
 * prefix-cache hit found are attached to the table, and only the tokens past the hit are prefilled;
 * section 3.3: the hit saves the prefill of the prefix, its blocks are still read).  Sequence i
 * already holds context_lens[i] tokens in its blocks; its n_i = cu_seqlens[i+1] - cu_seqlens[i]
 * new tokens (packed rows [cu_seqlens[i], cu_seqlens[i+1]) of q/k/v) sit at positions
 * context_lens[i] .. context_lens[i] + n_i - 1.  The call first writes every new token's k/v at
 * block_tables[i][p / block_size], offset p % block_size (p = its position), then computes
 *   out[cu_i + r][h] = sum_{c <= ctx_i + r} softmax_c(scale * q[cu_i + r][h] . K_c[g]) V_c[g]
 * with every key, cached or new, read from the pool through the table (g = h / group).  With all
 * context_lens 0 it computes what packed_prefill_attention computes.  context_lens: device int32
 * [num_seqs], each >= 0 with context + n_i <= max_blocks_per_seq * block_size (else the sequence
 * is skipped and PKV_DEVERR_LENGTH set); the table must name a block for every position below
 * context + n_i.  FP8 caches: the new tokens are written as paged_kv_append writes them, and every
 * key and value is read as its stored code times the head's scale (codes widened exactly to the
 * model dtype in shared memory).  Other arguments, shapes and errors as for
 * packed_prefill_attention. */
int paged_prefill_attention(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                            const int32_t *context_lens, int num_seqs, int max_seqlen, int64_t total_tokens,
                            const int32_t *block_tables, int max_blocks_per_seq, pkv_cache_t cache, int num_q_heads,
                            float scale, void *out, void *stream);

/* Block copy for copy-on-write (2kiu.com section 2.2: copy-on-write of prefix blocks shared by
 * beam search or parallel sampling; section 4.3 step 3: a shared block is never rewritten in
 * place, the diverging path gets its own copy): for i < num_pairs, physical block
 * dst_blocks[i] := physical block src_blocks[i], the whole block (K and V of every KV head, all
 * block_size slots).  src_blocks, dst_blocks: device int32 [num_pairs].  The destinations must
 * be distinct and none may also be a source in the same call (the copies run in parallel, so
 * overlapping pairs would race).  An id outside [0, num_blocks) skips its pair and sets
 * PKV_DEVERR_BLOCK_ID.  Exact byte copy. */
int paged_block_copy(pkv_cache_t cache, const int32_t *src_blocks, const int32_t *dst_blocks, int64_t num_pairs,
                     void *stream);

/* Swap out (2kiu.com section 2.2: on preemption a request's block contents go to CPU memory;
 * section 5.2): for i < num_ids, bytes [i*B, (i+1)*B) of dst := physical block block_ids[i],
 * B = the block size in bytes (kv_cache_view's num_bytes / num_blocks).  dst must be device
 * accessible: device memory, or page-locked host memory (cudaHostAlloc / cudaHostRegister; with
 * unified addressing its host pointer is also its device pointer), at least num_ids*B bytes,
 * 16-byte aligned.  block_ids: device int32 [num_ids].  Bad ids are skipped as above (their
 * bytes of dst are left as they were).  The copy kernel reads the pool and writes dst directly
 * (host memory over the host link, at the link's rate). */
int paged_block_swap_out(pkv_cache_t cache, const int32_t *block_ids, int64_t num_ids, void *dst, void *stream);

/* Swap in, the inverse: physical block block_ids[i] := bytes [i*B, (i+1)*B) of src (same rules for
 * src as for dst above; block_ids distinct).  Together with paged_block_swap_out this moves a
 * preempted request's blocks to CPU memory and back into whatever blocks the allocator hands out
 * on resumption; the block table is then rewritten by the caller. */
int paged_block_swap_in(pkv_cache_t cache, const int32_t *block_ids, int64_t num_ids, const void *src, void *stream);

/* ---------------------------------------------------------------- prefix cache (host work)
 * The functions below run on the host and take HOST pointers.  They implement the prefix cache
 * that sits on top of the paged pool (notes "vLLM：PagedAttention 与前缀缓存", sections on chained
 * hashing, lookup and reuse, reference counts and LRU, boundary conditions; 2kiu.com sections 3.2
 * and 4.3 steps 2-3).  Thread-safe per cache object. */

/* Chained block hashes: for every FULL block i of tokens[0 .. num_tokens) (num_tokens / block_size
 * of them; a partial tail block is not hashed),
 *   hash_i = SHA-256( hash_{i-1} (32 bytes) || tokens of block i as big-endian uint32 || extra )
 * with hash_{-1} = init (32 bytes) or 32 zero bytes when init is NULL.  extra (extra_bytes bytes,
 * may be NULL when 0) keys the semantic context: model and tokenizer version, adapter, salt.
 * hashes: [num_tokens / block_size][32] bytes, written; *num_hashes = their count. */
int pkv_block_hashes(const int32_t *tokens, int64_t num_tokens, int block_size, const void *extra, int64_t extra_bytes,
                     const uint8_t *init, uint8_t *hashes, int64_t *num_hashes);

typedef struct pkv_prefix_cache *pkv_prefix_cache_t; /* opaque */

/* A block manager over num_blocks physical block ids with a hash -> block map.  All blocks start
 * free and unhashed. */
int pkv_prefix_cache_create(int64_t num_blocks, pkv_prefix_cache_t *out);
int pkv_prefix_cache_destroy(pkv_prefix_cache_t pc);

/* Lookup: walk hashes[0 .. num_hashes) in order; each hash found in the map attaches its block
 * (blocks[i] = id, reference count + 1; a cached-free block leaves the LRU queue); the first hash
 * not found ends the walk.  *num_hit = number of blocks attached (the hit is *num_hit full blocks). */
int pkv_prefix_cache_match(pkv_prefix_cache_t pc, const uint8_t *hashes, int64_t num_hashes, int32_t *blocks,
                           int64_t *num_hit);

/* Take n blocks for new tokens (reference count 1): free unhashed blocks first, in the order they
 * became free, then cached-free blocks in LRU order (least recently released first), whose
 * mappings are dropped.  Fewer than n available: PKV_ENOMEM ("KV cache block pool exhausted") and
 * nothing is taken. */
int pkv_prefix_cache_allocate(pkv_prefix_cache_t pc, int64_t n, int32_t *blocks);

/* Publish full blocks after their prefill: map hashes[i] -> blocks[i].  A hash that already maps to
 * a block keeps its block.  Every block must be held by a request (EINVAL otherwise; nothing is
 * changed). */
int pkv_prefix_cache_insert(pkv_prefix_cache_t pc, const uint8_t *hashes, const int32_t *blocks, int64_t n);

/* A request lets go of its blocks: reference count - 1; at 0 a hashed block keeps its mapping and
 * joins the LRU queue (most recently released last), an unhashed block returns to the free list.
 * Releasing a block nobody holds is EINVAL (nothing is changed). */
int pkv_prefix_cache_release(pkv_prefix_cache_t pc, const int32_t *blocks, int64_t n);

/* out[0] = free unhashed blocks, out[1] = cached-free blocks (LRU queue), out[2] = blocks held by
 * requests, out[3] = mapped hashes. */
int pkv_prefix_cache_stats(pkv_prefix_cache_t pc, int64_t out[4]);

/* Profiling.  Between kv_cache_profile_start and kv_cache_profile_read the library records
 * CUDA events around each kernel it launches for this cache (decode split-K kernel, split
 * merge kernel, prefill kernel, append kernel, block copy kernel) on the launch stream.  kv_cache_profile_read synchronises
 * those events and returns the summed device time per kind (milliseconds) and launch
 * counts, then stops recording.  pkv_kernel_launches counts every kernel this library
 * launched in the process (all caches and free functions). */
typedef struct {
    int64_t decode_launches, prefill_launches, append_launches, merge_launches;
    double decode_ms, prefill_ms, append_ms, merge_ms;
    int64_t copy_launches; /* block copy / swap kernels */
    double copy_ms;
} pkv_profile_t;
#define PKV_PROFILE_DECODE 1u  /* the split-K decode kernel */
#define PKV_PROFILE_PREFILL 2u
#define PKV_PROFILE_APPEND 4u
#define PKV_PROFILE_MERGE 8u   /* the split merge kernel */
#define PKV_PROFILE_COPY 16u  /* block copy and swap */
#define PKV_PROFILE_ALL 31u
/* kinds: which kernels to bracket (events between two kernels stop their launches from overlapping,
 * so time only what you need). */
int kv_cache_profile_start(pkv_cache_t cache, unsigned kinds);
/* The same, bracketing only the 1st, (every+1)-th, (2 every+1)-th ... launch of each kind (every >= 1,
 * else PKV_EINVAL): the kernel times of a long run are sampled while the launches in between keep
 * their overlap.  kv_cache_profile_start(cache, kinds) is every = 1. */
int kv_cache_profile_start_sampled(pkv_cache_t cache, unsigned kinds, int every);
int kv_cache_profile_read(pkv_cache_t cache, pkv_profile_t *out);
int64_t pkv_kernel_launches(void);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H */
