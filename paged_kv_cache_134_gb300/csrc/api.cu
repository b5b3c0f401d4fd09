// C ABI of the library: handle management, host-side validation, launches, error
// reporting and profiling.  Every computation happens in the kernels of append.cu,
// decode*.cu, prefill.cu and blocks.cu.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>

#include "pkv_internal.h"

std::atomic<int64_t> g_pkv_launches{0};

namespace {
thread_local char g_msg[512] = "";

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int elem_bytes(pkv_dtype d) { return d == PKV_FP8_E4M3 ? 1 : 2; }

bool supported_head_dim(int d) { return d == 64 || d == 128; }
bool supported_block_size(int b) { return b == 8 || b == 16 || b == 32; }
bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

int check_device(const pkv_cache *c) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pkv_cuda_fail(e, "cudaGetDevice");
    if (dev != c->device) return pkv_fail(PKV_EINVAL, "cache lives on device %d but device %d is current", c->device, dev);
    return PKV_OK;
}

int ensure_workspace(pkv_cache *c, int64_t floats) {
    const int64_t bytes = floats * (int64_t)sizeof(float);
    if (bytes <= c->ws_bytes) return PKV_OK;
    if (c->ws) cudaFree(c->ws);
    c->ws = nullptr;
    c->ws_bytes = 0;
    cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&c->ws), (size_t)bytes);
    if (e != cudaSuccess) {
        c->ws = nullptr;
        cudaGetLastError();
        return pkv_fail(PKV_ENOMEM, "decode workspace of %lld bytes: %s", (long long)bytes, cudaGetErrorString(e));
    }
    c->ws_bytes = bytes;
    return PKV_OK;
}
} // namespace

int pkv_fail(int status, const char *fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return status;
}

int pkv_cuda_fail(cudaError_t e, const char *what) {
    return pkv_fail(PKV_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

cudaError_t launch_decode_chunked(pkv_cache *c, DecodeLaunch d, cudaStream_t st) {
    const int G = d.num_q_heads / c->num_kv_heads;
    const int per = decode_seqs_per_launch(c, G);
    const int total = d.num_seqs;
    const int64_t row_bytes = (int64_t)d.num_q_heads * c->head_dim * 2; // q and out rows, 16-bit model dtype
    const char *q0 = static_cast<const char *>(d.q);
    char *out0 = static_cast<char *>(d.out);
    const int32_t *tables0 = d.tables, *lens0 = d.lens;
    CascadePrefixLaunch p;
    if (d.prefix) p = *d.prefix;
    for (int s0 = 0; s0 < total; s0 += per) {
        const int n = total - s0 < per ? total - s0 : per;
        d.q = q0 + s0 * row_bytes;
        d.out = out0 + s0 * row_bytes;
        d.tables = tables0 ? tables0 + (int64_t)s0 * d.max_blocks : nullptr;
        d.lens = lens0 + s0;
        d.num_seqs = n;
        if (d.prefix) {
            // the launch's own rows: its queries, its tables (every one names the shared prefix), and the
            // (m, l) half of the workspace right after its n * Hq * max_splits partial rows
            p.q = d.q;
            p.tables = d.tables;
            p.num_seqs = n;
            p.ws_ml = p.ws_o + (int64_t)n * d.num_q_heads * d.max_splits * c->head_dim;
            cudaError_t e = launch_cascade_prefix(c, p, st, 1);
            if (e != cudaSuccess) return e;
            d.prefix = &p;
        }
        cudaError_t e = launch_decode(c, d, st);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

PkvTimer::PkvTimer(pkv_cache *c_, int kind_, cudaStream_t st_) : c(c_), kind(kind_), st(st_) {
    if (!c || !c->profiling || !(c->profile_kinds & (1u << kind))) return;
    std::lock_guard<std::mutex> lk(c->mu);
    // sampled profiling: the launches in between run without events, so that their overlap with
    // the neighbouring kernels (programmatic dependent launch) is left as it is
    if (c->profile_seen[kind]++ % c->profile_every != 0) return;
    for (cudaEvent_t *ev : {&a, &b}) {
        if (!c->event_pool.empty()) {
            *ev = c->event_pool.back();
            c->event_pool.pop_back();
        } else if (cudaEventCreate(ev) != cudaSuccess) {
            *ev = nullptr;
        }
    }
    if (a) cudaEventRecord(a, st);
}

PkvTimer::~PkvTimer() {
    if (!c || !c->profiling || !a || !b) return;
    cudaEventRecord(b, st);
    std::lock_guard<std::mutex> lk(c->mu);
    c->events.push_back({kind, a, b});
}

extern "C" {

const char *pkv_last_error(void) { return g_msg; }

int64_t pkv_kernel_launches(void) { return g_pkv_launches.load(); }

int kv_cache_create(int64_t num_blocks, int block_size, int num_kv_heads, int head_dim, pkv_dtype kv_dtype,
                    pkv_dtype model_dtype, pkv_cache_t *out) {
    if (!out) return pkv_fail(PKV_EINVAL, "out is NULL");
    if (num_blocks <= 0 || num_kv_heads <= 0) return pkv_fail(PKV_EINVAL, "num_blocks and num_kv_heads must be > 0");
    if (kv_dtype < PKV_F16 || kv_dtype > PKV_FP8_E4M3 || model_dtype < PKV_F16 || model_dtype > PKV_BF16)
        return pkv_fail(PKV_EINVAL, "bad dtype (kv %d, model %d)", (int)kv_dtype, (int)model_dtype);
    if (kv_dtype != PKV_FP8_E4M3 && kv_dtype != model_dtype)
        return pkv_fail(PKV_EINVAL, "a 16-bit cache must use its own dtype as model dtype");
    if (!supported_head_dim(head_dim)) return pkv_fail(PKV_EUNSUPPORTED, "head_dim %d not in {64, 128}", head_dim);
    if (!supported_block_size(block_size))
        return pkv_fail(PKV_EUNSUPPORTED, "block_size %d not in {8, 16, 32}", block_size);
    pkv_cache *c = new pkv_cache();
    cudaError_t e = cudaGetDevice(&c->device);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
    if (e != cudaSuccess) {
        delete c;
        return pkv_cuda_fail(e, "device query");
    }
    c->num_blocks = num_blocks;
    c->block_size = block_size;
    c->num_kv_heads = num_kv_heads;
    c->head_dim = head_dim;
    c->kv_dtype = kv_dtype;
    c->model_dtype = model_dtype;
    c->elem_bytes = elem_bytes(kv_dtype);
    c->tile_bytes = (int64_t)block_size * head_dim * c->elem_bytes;
    c->pool_bytes = num_blocks * 2 * num_kv_heads * c->tile_bytes;
    e = cudaMalloc(&c->pool, (size_t)c->pool_bytes);
    if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void **>(&c->err), 16);
    if (e == cudaSuccess && kv_dtype == PKV_FP8_E4M3) {
        e = cudaMalloc(reinterpret_cast<void **>(&c->k_scale), sizeof(float) * num_kv_heads);
        if (e == cudaSuccess) e = cudaMalloc(reinterpret_cast<void **>(&c->v_scale), sizeof(float) * num_kv_heads);
    }
    if (e == cudaSuccess) e = cudaMemset(c->pool, 0, (size_t)c->pool_bytes);
    if (e == cudaSuccess) e = cudaMemset(c->err, 0, 16);
    if (e == cudaSuccess) {
        // the no-alloc decode's fixed scratch is made resident on this device now, while the cache is
        // created, so that paged_decode_attention_noalloc never has to bring it in later
        if (int r = pkv_noalloc_scratch_prepare(c->device)) {
            kv_cache_destroy(c);
            return r;
        }
    }
    if (e == cudaSuccess && c->k_scale) {
        // default scale 1.0f (0x3F800000)
        float ones[256];
        for (float &x : ones) x = 1.0f;
        for (int h = 0; h < num_kv_heads && e == cudaSuccess; h += 256) {
            const int n = num_kv_heads - h < 256 ? num_kv_heads - h : 256;
            e = cudaMemcpy(c->k_scale + h, ones, n * sizeof(float), cudaMemcpyHostToDevice);
            if (e == cudaSuccess) e = cudaMemcpy(c->v_scale + h, ones, n * sizeof(float), cudaMemcpyHostToDevice);
        }
    }
    if (e != cudaSuccess) {
        const int st = (e == cudaErrorMemoryAllocation) ? PKV_ENOMEM : PKV_ECUDA;
        cudaGetLastError();
        kv_cache_destroy(c);
        return pkv_fail(st, "kv_cache_create (%lld bytes): %s", (long long)(num_blocks * 2 * num_kv_heads *
                                                                              (int64_t)block_size * head_dim *
                                                                              elem_bytes(kv_dtype)),
                        cudaGetErrorString(e));
    }
    *out = c;
    return PKV_OK;
}

int kv_cache_destroy(pkv_cache_t c) {
    if (!c) return PKV_OK;
    cudaDeviceSynchronize();
    if (c->pool) cudaFree(c->pool);
    if (c->err) cudaFree(c->err);
    if (c->k_scale) cudaFree(c->k_scale);
    if (c->v_scale) cudaFree(c->v_scale);
    if (c->ws) cudaFree(c->ws);
    if (c->plan) cudaFree(c->plan);
    for (auto &ev : c->events) {
        cudaEventDestroy(ev.a);
        cudaEventDestroy(ev.b);
    }
    for (auto ev : c->event_pool) cudaEventDestroy(ev);
    delete c;
    return PKV_OK;
}

int kv_cache_set_scales(pkv_cache_t c, const float *k_scale, const float *v_scale, void *stream) {
    PKV_RANGE("kv_cache_set_scales");
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (c->kv_dtype != PKV_FP8_E4M3) return pkv_fail(PKV_EINVAL, "scales apply to FP8 caches only");
    if (!k_scale || !v_scale) return pkv_fail(PKV_EINVAL, "scale pointer is NULL");
    if (int r = check_device(c)) return r;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t n = sizeof(float) * c->num_kv_heads;
    cudaError_t e = cudaMemcpyAsync(c->k_scale, k_scale, n, cudaMemcpyDeviceToDevice, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(c->v_scale, v_scale, n, cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return pkv_cuda_fail(e, "kv_cache_set_scales");
    return PKV_OK;
}

int kv_cache_view(pkv_cache_t c, void **base, int64_t strides_elems[5], int64_t *num_bytes) {
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    const int64_t tile = (int64_t)c->block_size * c->head_dim;
    if (base) *base = c->pool;
    if (strides_elems) {
        strides_elems[0] = 2 * c->num_kv_heads * tile;
        strides_elems[1] = c->num_kv_heads * tile;
        strides_elems[2] = tile;
        strides_elems[3] = c->head_dim;
        strides_elems[4] = 1;
    }
    if (num_bytes) *num_bytes = c->pool_bytes;
    return PKV_OK;
}

int kv_cache_reserve(pkv_cache_t c, int max_seqs, int max_q_heads, int max_blocks_per_seq) {
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (max_seqs < 0 || max_q_heads < 0 || max_blocks_per_seq < 0) return pkv_fail(PKV_EINVAL, "negative size");
    if (int r = check_device(c)) return r;
    const int bps = decode_split_blocks(c);
    const int max_splits = (max_blocks_per_seq + bps - 1) / bps;
    // consecutive launches of one call share the workspace: one launch's rows are enough
    int rows = max_seqs;
    if (max_q_heads > 0 && max_q_heads % c->num_kv_heads == 0 && supported_group(max_q_heads / c->num_kv_heads))
        rows = std::min(rows, decode_seqs_per_launch(c, max_q_heads / c->num_kv_heads));
    return ensure_workspace(c, decode_workspace_floats(c, rows, max_q_heads, max_splits));
}

int kv_cache_check_error(pkv_cache_t c, int *device_code) {
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return pkv_cuda_fail(e, "cudaDeviceSynchronize");
    unsigned int v = 0;
    e = cudaMemcpy(&v, c->err, sizeof v, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(c->err, 0, sizeof v);
    if (e != cudaSuccess) return pkv_cuda_fail(e, "reading the device error word");
    if (device_code) *device_code = static_cast<int>(v);
    if (v) return pkv_fail(PKV_EDEVICE, "device error bits 0x%x", v);
    return PKV_OK;
}

int paged_slot_mapping(const int32_t *block_tables, int num_rows, int max_blocks_per_seq, const int32_t *seq_ids,
                       const int32_t *positions, int64_t num_tokens, int block_size, int64_t *slot_mapping,
                       void *stream) {
    PKV_RANGE("paged_slot_mapping");
    if (num_tokens < 0 || num_rows < 0 || max_blocks_per_seq < 0) return pkv_fail(PKV_EINVAL, "negative size");
    if (block_size <= 0) return pkv_fail(PKV_EINVAL, "block_size must be > 0");
    if (num_tokens == 0) return PKV_OK;
    if (!seq_ids || !positions || !slot_mapping || (!block_tables && num_rows > 0 && max_blocks_per_seq > 0))
        return pkv_fail(PKV_EINVAL, "NULL pointer");
    cudaError_t e = launch_slot_mapping(block_tables, num_rows, max_blocks_per_seq, seq_ids, positions, num_tokens,
                                        block_size, slot_mapping, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pkv_cuda_fail(e, "slot mapping launch");
    return PKV_OK;
}

int paged_kv_append(pkv_cache_t c, const void *k, const void *v, const int64_t *slot_mapping, int64_t num_tokens,
                    void *stream) {
    PKV_RANGE("paged_kv_append");
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (num_tokens < 0) return pkv_fail(PKV_EINVAL, "num_tokens < 0");
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping) return pkv_fail(PKV_EINVAL, "NULL pointer");
    if (!aligned16(k) || !aligned16(v)) return pkv_fail(PKV_EINVAL, "k and v must be 16-byte aligned");
    if (int r = check_device(c)) return r;
    cudaError_t e = launch_append(c, k, v, slot_mapping, num_tokens, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pkv_cuda_fail(e, "append launch");
    return PKV_OK;
}

int paged_kv_append_at(pkv_cache_t c, const void *k, const void *v, const int32_t *block_tables, int num_rows,
                       int max_blocks_per_seq, const int32_t *seq_ids, const int32_t *positions, int64_t num_tokens,
                       int64_t *slot_mapping, void *stream) {
    PKV_RANGE("paged_kv_append_at");
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (num_tokens < 0 || num_rows < 0 || max_blocks_per_seq < 0) return pkv_fail(PKV_EINVAL, "negative size");
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !seq_ids || !positions || (!block_tables && num_rows > 0 && max_blocks_per_seq > 0))
        return pkv_fail(PKV_EINVAL, "NULL pointer");
    if (!aligned16(k) || !aligned16(v)) return pkv_fail(PKV_EINVAL, "k and v must be 16-byte aligned");
    if (int r = check_device(c)) return r;
    cudaError_t e = launch_append_at(c, k, v, block_tables, num_rows, max_blocks_per_seq, seq_ids, positions,
                                     num_tokens, slot_mapping, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pkv_cuda_fail(e, "append launch");
    return PKV_OK;
}

int paged_decode_attention(const void *q, pkv_cache_t c, const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens, int num_seqs, int num_q_heads, float scale, void *out,
                           void *stream) {
    PKV_RANGE("paged_decode_attention");
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (num_seqs < 0 || max_blocks_per_seq < 0) return pkv_fail(PKV_EINVAL, "negative size");
    if (num_seqs == 0) return PKV_OK;
    if (num_q_heads <= 0 || num_q_heads % c->num_kv_heads)
        return pkv_fail(PKV_EINVAL, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                        c->num_kv_heads);
    if (!supported_group(num_q_heads / c->num_kv_heads))
        return pkv_fail(PKV_EUNSUPPORTED, "num_q_heads / num_kv_heads = %d not in {1, 2, 4, 8}",
                        num_q_heads / c->num_kv_heads);
    if (!q || !out || !context_lens || (!block_tables && max_blocks_per_seq > 0))
        return pkv_fail(PKV_EINVAL, "NULL pointer");
    if (!aligned16(q) || !aligned16(out)) return pkv_fail(PKV_EINVAL, "q and out must be 16-byte aligned");
    if (!(scale == scale)) return pkv_fail(PKV_EINVAL, "scale is NaN");
    if (int r = check_device(c)) return r;
    // a batch larger than one launch takes runs in consecutive launches that share the workspace
    const int per_launch = std::min(num_seqs, decode_seqs_per_launch(c, num_q_heads / c->num_kv_heads));
    DecodeLaunch d;
    d.q = q;
    d.out = out;
    d.tables = block_tables;
    d.lens = context_lens;
    d.max_blocks = max_blocks_per_seq;
    d.num_seqs = num_seqs;
    d.num_q_heads = num_q_heads;
    d.scale = scale;
    d.split_blocks = decode_split_blocks(c);
    d.max_splits = (max_blocks_per_seq + d.split_blocks - 1) / d.split_blocks;
    const int64_t ws = decode_workspace_floats(c, per_launch, num_q_heads, d.max_splits);
    if (int r = ensure_workspace(c, ws)) return r;
    d.ws_o = ws ? c->ws : nullptr;
    d.ws_ml = nullptr;
    cudaError_t e = launch_decode_chunked(c, d, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pkv_cuda_fail(e, "decode launch");
    return PKV_OK;
}

static int prefill_entry(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                         const int32_t *context_lens, int num_seqs, int max_seqlen, int64_t total_tokens,
                         const int32_t *block_tables, int max_blocks_per_seq, pkv_cache_t c, int num_q_heads,
                         float scale, void *out, void *stream) {
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (num_seqs < 0 || max_seqlen < 0 || max_blocks_per_seq < 0 || total_tokens < 0)
        return pkv_fail(PKV_EINVAL, "negative size");
    if (total_tokens > 0x7FFFFFFF) return pkv_fail(PKV_EUNSUPPORTED, "more than 2^31 - 1 packed tokens");
    if (num_seqs == 0 || max_seqlen == 0 || total_tokens == 0) return PKV_OK;
    if (num_q_heads <= 0 || num_q_heads % c->num_kv_heads)
        return pkv_fail(PKV_EINVAL, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                        c->num_kv_heads);
    if (!supported_group(num_q_heads / c->num_kv_heads))
        return pkv_fail(PKV_EUNSUPPORTED, "num_q_heads / num_kv_heads = %d not in {1, 2, 4, 8}",
                        num_q_heads / c->num_kv_heads);
    if (!q || !k || !v || !out || !cu_seqlens || !block_tables) return pkv_fail(PKV_EINVAL, "NULL pointer");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
        return pkv_fail(PKV_EINVAL, "q, k, v and out must be 16-byte aligned");
    if (int r = check_device(c)) return r;
    PrefillLaunch p;
    p.q = q;
    p.k = k;
    p.v = v;
    p.out = out;
    p.cu = cu_seqlens;
    p.ctx = context_lens;
    p.tables = block_tables;
    p.num_seqs = num_seqs;
    p.max_seqlen = max_seqlen;
    p.total_tokens = total_tokens;
    p.max_blocks = max_blocks_per_seq;
    p.num_q_heads = num_q_heads;
    p.scale = scale;
    cudaError_t e = launch_prefill(c, p, static_cast<cudaStream_t>(stream));
    if (e == cudaErrorNotSupported) return pkv_fail(PKV_EUNSUPPORTED, "prefill shape not supported");
    if (e != cudaSuccess) return pkv_cuda_fail(e, "prefill launch");
    return PKV_OK;
}

int paged_decode_attention_cascade(const void *q, pkv_cache_t c, const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *context_lens, int num_seqs, int num_q_heads, int shared_prefix_len,
                                   float scale, void *out, void *stream) {
    PKV_RANGE("paged_decode_attention_cascade");
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (shared_prefix_len < 0 || shared_prefix_len % c->block_size)
        return pkv_fail(PKV_EINVAL, "shared_prefix_len %d is not a non-negative multiple of block_size %d",
                        shared_prefix_len, c->block_size);
    if (shared_prefix_len == 0)
        return paged_decode_attention(q, c, block_tables, max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                                      scale, out, stream);
    if (num_seqs < 0 || max_blocks_per_seq < 0) return pkv_fail(PKV_EINVAL, "negative size");
    if (num_seqs == 0) return PKV_OK;
    if ((int64_t)shared_prefix_len > (int64_t)max_blocks_per_seq * c->block_size)
        return pkv_fail(PKV_EINVAL, "shared prefix longer than the tables");
    if (num_q_heads <= 0 || num_q_heads % c->num_kv_heads)
        return pkv_fail(PKV_EINVAL, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                        c->num_kv_heads);
    if (!supported_group(num_q_heads / c->num_kv_heads))
        return pkv_fail(PKV_EUNSUPPORTED, "num_q_heads / num_kv_heads = %d not in {1, 2, 4, 8}",
                        num_q_heads / c->num_kv_heads);
    if (!q || !out || !context_lens || !block_tables) return pkv_fail(PKV_EINVAL, "NULL pointer");
    if (!aligned16(q) || !aligned16(out)) return pkv_fail(PKV_EINVAL, "q and out must be 16-byte aligned");
    if (!(scale == scale)) return pkv_fail(PKV_EINVAL, "scale is NaN");
    if (int r = check_device(c)) return r;
    // a batch larger than one launch takes runs in consecutive launches (each reads the prefix once)
    const int per_launch = std::min(num_seqs, decode_seqs_per_launch(c, num_q_heads / c->num_kv_heads));
    const int split_tokens = cascade_split_tokens(c, per_launch, num_q_heads, shared_prefix_len);
    const int nps = (shared_prefix_len + split_tokens - 1) / split_tokens;
    const int pb = shared_prefix_len / c->block_size;
    DecodeLaunch d;
    d.q = q;
    d.out = out;
    d.tables = block_tables;
    d.lens = context_lens;
    d.max_blocks = max_blocks_per_seq;
    d.num_seqs = num_seqs;
    d.num_q_heads = num_q_heads;
    d.scale = scale;
    d.split_blocks = cascade_suffix_split_blocks(c);
    d.max_splits = nps + (max_blocks_per_seq - pb + d.split_blocks - 1) / d.split_blocks;
    d.start_block = pb;
    d.slot0 = nps;
    const int64_t rows = (int64_t)per_launch * num_q_heads * d.max_splits;
    if (int r = ensure_workspace(c, rows * (c->head_dim + 2))) return r;
    d.ws_o = c->ws;
    d.ws_ml = nullptr;
    CascadePrefixLaunch p;
    p.q = q;
    p.tables = block_tables;
    p.max_blocks = max_blocks_per_seq;
    p.num_seqs = num_seqs;
    p.num_q_heads = num_q_heads;
    p.prefix_tokens = shared_prefix_len;
    p.split_tokens = split_tokens;
    p.max_splits = d.max_splits;
    p.scale = scale;
    p.ws_o = c->ws;
    p.ws_ml = c->ws + rows * c->head_dim;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // launches, per run of sequences: the prefix phase's plan, the suffix decode, the prefix kernel,
    // the merge
    d.prefix = &p;
    cudaError_t e = launch_decode_chunked(c, d, st);
    if (e == cudaErrorNotSupported) return pkv_fail(PKV_EUNSUPPORTED, "cascade shape not supported");
    if (e != cudaSuccess) return pkv_cuda_fail(e, "cascade decode launch");
    return PKV_OK;
}

int packed_prefill_attention(const void *q, const void *k, const void *v, const int32_t *cu_seqlens, int num_seqs,
                             int max_seqlen, int64_t total_tokens, const int32_t *block_tables,
                             int max_blocks_per_seq, pkv_cache_t c, int num_q_heads, float scale, void *out,
                             void *stream) {
    PKV_RANGE("packed_prefill_attention");
    return prefill_entry(q, k, v, cu_seqlens, nullptr, num_seqs, max_seqlen, total_tokens, block_tables,
                         max_blocks_per_seq, c, num_q_heads, scale, out, stream);
}

int paged_prefill_attention(const void *q, const void *k, const void *v, const int32_t *cu_seqlens,
                            const int32_t *context_lens, int num_seqs, int max_seqlen, int64_t total_tokens,
                            const int32_t *block_tables, int max_blocks_per_seq, pkv_cache_t c, int num_q_heads,
                            float scale, void *out, void *stream) {
    PKV_RANGE("paged_prefill_attention");
    if (!context_lens && num_seqs > 0) return pkv_fail(PKV_EINVAL, "NULL pointer");
    return prefill_entry(q, k, v, cu_seqlens, context_lens, num_seqs, max_seqlen, total_tokens, block_tables,
                         max_blocks_per_seq, c, num_q_heads, scale, out, stream);
}

int paged_block_copy(pkv_cache_t c, const int32_t *src_blocks, const int32_t *dst_blocks, int64_t num_pairs,
                     void *stream) {
    PKV_RANGE("paged_block_copy");
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (num_pairs < 0) return pkv_fail(PKV_EINVAL, "num_pairs < 0");
    if (num_pairs == 0) return PKV_OK;
    if (!src_blocks || !dst_blocks) return pkv_fail(PKV_EINVAL, "NULL pointer");
    if (int r = check_device(c)) return r;
    cudaError_t e = launch_copy_blocks(c, c->pool, src_blocks, c->num_blocks, c->pool, dst_blocks, c->num_blocks,
                                       num_pairs, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pkv_cuda_fail(e, "block copy launch");
    return PKV_OK;
}

int paged_block_swap_out(pkv_cache_t c, const int32_t *block_ids, int64_t num_ids, void *dst, void *stream) {
    PKV_RANGE("paged_block_swap_out");
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (num_ids < 0) return pkv_fail(PKV_EINVAL, "num_ids < 0");
    if (num_ids == 0) return PKV_OK;
    if (!block_ids || !dst) return pkv_fail(PKV_EINVAL, "NULL pointer");
    if (!aligned16(dst)) return pkv_fail(PKV_EINVAL, "dst must be 16-byte aligned");
    if (int r = check_device(c)) return r;
    cudaError_t e = launch_copy_blocks(c, c->pool, block_ids, c->num_blocks, dst, nullptr, num_ids, num_ids,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pkv_cuda_fail(e, "swap-out launch");
    return PKV_OK;
}

int paged_block_swap_in(pkv_cache_t c, const int32_t *block_ids, int64_t num_ids, const void *src, void *stream) {
    PKV_RANGE("paged_block_swap_in");
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (num_ids < 0) return pkv_fail(PKV_EINVAL, "num_ids < 0");
    if (num_ids == 0) return PKV_OK;
    if (!block_ids || !src) return pkv_fail(PKV_EINVAL, "NULL pointer");
    if (!aligned16(src)) return pkv_fail(PKV_EINVAL, "src must be 16-byte aligned");
    if (int r = check_device(c)) return r;
    cudaError_t e = launch_copy_blocks(c, src, nullptr, num_ids, c->pool, block_ids, c->num_blocks, num_ids,
                                       static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pkv_cuda_fail(e, "swap-in launch");
    return PKV_OK;
}

int kv_cache_profile_start(pkv_cache_t c, unsigned kinds) { return kv_cache_profile_start_sampled(c, kinds, 1); }

int kv_cache_profile_start_sampled(pkv_cache_t c, unsigned kinds, int every) {
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (every < 1) return pkv_fail(PKV_EINVAL, "every must be >= 1, got %d", every);
    // PKV_PROFILE_* bits map onto (1 << PKV_KIND_*)
    c->profile_kinds = ((kinds & PKV_PROFILE_DECODE) ? 1u << PKV_KIND_DECODE : 0u) |
                       ((kinds & PKV_PROFILE_PREFILL) ? 1u << PKV_KIND_PREFILL : 0u) |
                       ((kinds & PKV_PROFILE_APPEND) ? 1u << PKV_KIND_APPEND : 0u) |
                       ((kinds & PKV_PROFILE_MERGE) ? 1u << PKV_KIND_MERGE : 0u) |
                       ((kinds & PKV_PROFILE_COPY) ? 1u << PKV_KIND_COPY : 0u);
    std::lock_guard<std::mutex> lk(c->mu);
    for (auto &ev : c->events) {
        c->event_pool.push_back(ev.a);
        c->event_pool.push_back(ev.b);
    }
    c->events.clear();
    c->profile_every = every;
    for (int64_t &n : c->profile_seen) n = 0;
    c->profiling = true;
    return PKV_OK;
}

int kv_cache_profile_read(pkv_cache_t c, pkv_profile_t *out) {
    if (!c || !out) return pkv_fail(PKV_EINVAL, "NULL argument");
    std::lock_guard<std::mutex> lk(c->mu);
    c->profiling = false;
    std::memset(out, 0, sizeof *out);
    for (auto &ev : c->events) {
        cudaError_t e = cudaEventSynchronize(ev.b);
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, ev.a, ev.b);
        if (e != cudaSuccess) return pkv_cuda_fail(e, "profile events");
        if (ev.kind == PKV_KIND_DECODE) {
            out->decode_launches++;
            out->decode_ms += ms;
        } else if (ev.kind == PKV_KIND_PREFILL) {
            out->prefill_launches++;
            out->prefill_ms += ms;
        } else if (ev.kind == PKV_KIND_APPEND) {
            out->append_launches++;
            out->append_ms += ms;
        } else if (ev.kind == PKV_KIND_COPY) {
            out->copy_launches++;
            out->copy_ms += ms;
        } else {
            out->merge_launches++;
            out->merge_ms += ms;
        }
        c->event_pool.push_back(ev.a);
        c->event_pool.push_back(ev.b);
    }
    c->events.clear();
    return PKV_OK;
}

} // extern "C"
