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
// and passes it to the kernel.  With CUDA's lazy module loading the array only becomes resident on
// a device when something first refers to it there, and that first reference allocates it; so the
// lookup is made by kv_cache_create (every call here needs a cache, created on the same device),
// before the caller's own allocator takes the rest of the device memory.
#include <mutex>

#include "pkv_internal.h"

// 16 MiB of fp32 partials, held by every device on which a cache was created until the process exits.
constexpr int64_t kScratchFloats = int64_t(4) << 20;
static __device__ __align__(256) float g_decode_scratch[kScratchFloats];

namespace {

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
float *g_scratch_ptr[kMaxDevices] = {};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

} // namespace

// Called by kv_cache_create with `device` current.  The lookup is repeated on every cache creation:
// after a cudaDeviceReset the module is loaded again and the array may sit elsewhere, and a reset also
// destroys every cache, so the next cache created on the device refreshes the address before any
// no-alloc call can use it.
int pkv_noalloc_scratch_prepare(int device) {
    if (device < 0 || device >= kMaxDevices) return pkv_fail(PKV_EUNSUPPORTED, "device index %d out of range", device);
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_decode_scratch);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return pkv_fail(e == cudaErrorMemoryAllocation ? PKV_ENOMEM : PKV_ECUDA,
                        "making the no-alloc decode scratch (%lld bytes) resident: %s",
                        (long long)(kScratchFloats * 4), cudaGetErrorString(e));
    }
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    g_scratch_ptr[device] = static_cast<float *>(p);
    return PKV_OK;
}

extern "C" int paged_decode_attention_noalloc(const void *q, pkv_cache_t c, const int32_t *block_tables,
                                              int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                              int num_q_heads, float scale, void *out, void *stream) {
    PKV_RANGE("paged_decode_attention_noalloc");
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (num_seqs < 0 || max_blocks_per_seq < 0) return pkv_fail(PKV_EINVAL, "negative size");
    if (num_seqs == 0) return PKV_OK;
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
    // a batch larger than one launch takes runs in consecutive launches that share the scratch
    const int per_launch = num_seqs < decode_seqs_per_launch(c, group) ? num_seqs : decode_seqs_per_launch(c, group);
    const int64_t need = decode_workspace_floats(c, per_launch, num_q_heads, d.max_splits);
    if (need > kScratchFloats)
        return pkv_fail(PKV_EINVAL,
                        "no-alloc decode needs %lld bytes of scratch for %d sequences x %d query heads x %d splits; "
                        "its fixed scratch holds %lld bytes (use fewer sequences per call or paged_decode_attention)",
                        (long long)(need * 4), per_launch, num_q_heads, d.max_splits, (long long)(kScratchFloats * 4));
    d.ws_o = nullptr;
    if (need > 0) {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        d.ws_o = dev < kMaxDevices ? g_scratch_ptr[dev] : nullptr;
    }
    if (need > 0 && !d.ws_o)
        return pkv_fail(PKV_EINVAL, "no-alloc decode scratch is not resident on device %d (create a cache there first)",
                        dev);
    e = launch_decode_chunked(c, d, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pkv_cuda_fail(e, "decode launch");
    return PKV_OK;
}
