// paged_decode_attention_noalloc: the paged decode without any device-memory allocation.
//
// paged_decode_attention keeps its split-K partials in a workspace owned by the cache and grows
// it with cudaMalloc when a call needs more.  Some callers cannot allow that: a serving engine
// that has handed nearly all device memory to its own allocator (the KV pool is sized to fill
// the GPU) must not see a library allocate behind its back; cudaMalloc and cudaFree may also
// synchronise the whole device, which stalls every other stream such a caller is running.  This
// entry point takes its scratch from one file-scope __device__ array of fixed size instead, and
// calls no allocating routine (no cudaMalloc, no cudaFree, nothing from torch).
//
// The array's name in host code is only a host-side stand-in, not a device address, so the host
// looks up the real address with cudaGetSymbolAddress, once per device, with that device current,
// on the first call made on that device, and passes it to the kernel.
#include <mutex>

#include "pkv_internal.h"

// 16 MiB of fp32 partials, held by every GPU that loads the library until the process exits.
constexpr int64_t kScratchFloats = int64_t(4) << 20;
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

namespace {

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
float *g_scratch_ptr[kMaxDevices] = {};

int scratch_for_device(int dev, float **out) {
    if (dev < 0 || dev >= kMaxDevices) return pkv_fail(PKV_EUNSUPPORTED, "device index %d out of range", dev);
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return pkv_cuda_fail(e, "cudaGetSymbolAddress of the decode scratch array");
        g_scratch_ptr[dev] = static_cast<float *>(p);
    }
    *out = g_scratch_ptr[dev];
    return PKV_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

} // namespace

extern "C" int paged_decode_attention_noalloc(const void *q, pkv_cache_t c, const int32_t *block_tables,
                                              int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                              int num_q_heads, float scale, void *out, void *stream) {
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (num_seqs < 0 || max_blocks_per_seq < 0) return pkv_fail(PKV_EINVAL, "negative size");
    if (num_seqs == 0) return PKV_OK;
    if (num_seqs > 1024) return pkv_fail(PKV_EUNSUPPORTED, "num_seqs %d > 1024 per call", num_seqs);
    if (num_q_heads <= 0 || num_q_heads % c->num_kv_heads)
        return pkv_fail(PKV_EINVAL, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                        c->num_kv_heads);
    const int group = num_q_heads / c->num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8)
        return pkv_fail(PKV_EUNSUPPORTED, "num_q_heads / num_kv_heads = %d not in {1, 2, 4, 8}", group);
    if (!q || !out || !context_lens || (!block_tables && max_blocks_per_seq > 0))
        return pkv_fail(PKV_EINVAL, "NULL pointer");
    if (!aligned16(q) || !aligned16(out)) return pkv_fail(PKV_EINVAL, "q and out must be 16-byte aligned");
    if (!(scale == scale)) return pkv_fail(PKV_EINVAL, "scale is NaN");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pkv_cuda_fail(e, "cudaGetDevice");
    if (dev != c->device) return pkv_fail(PKV_EINVAL, "cache lives on device %d but device %d is current", c->device, dev);

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
    d.ws_ml = nullptr;
    const int64_t need = decode_workspace_floats(c, num_seqs, num_q_heads, d.max_splits);
    if (need > kScratchFloats)
        return pkv_fail(PKV_EINVAL,
                        "no-alloc decode needs %lld bytes of scratch for %d sequences x %d query heads x %d splits; "
                        "its fixed scratch holds %lld bytes (use fewer sequences per call or paged_decode_attention)",
                        (long long)(need * 4), num_seqs, num_q_heads, d.max_splits, (long long)(kScratchFloats * 4));
    d.ws_o = nullptr;
    if (need > 0) {
        float *p = nullptr;
        if (int r = scratch_for_device(dev, &p)) return r;
        d.ws_o = p;
    }
    e = launch_decode(c, d, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pkv_cuda_fail(e, "decode launch");
    return PKV_OK;
}
