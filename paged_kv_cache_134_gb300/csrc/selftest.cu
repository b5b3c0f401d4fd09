// Self-test of the bounded mbarrier wait that every kernel of the library uses.
//
// The pages ask that the cache degrade rather than crash when something goes wrong ("Paged KV Cache
// 与 Packed Sequence", discosf.com, section 5.1; "PagedAttention 与前缀缓存", 2kiu.com, section 6.1 on
// an exhausted block pool).  On the GPU that means no wait may hang: every wait on an mbarrier gives
// up after a time limit and reports PKV_DEVERR_TIMEOUT in the cache's error word.  This kernel makes
// exactly that happen on purpose, safely: one CTA initialises an mbarrier that nothing ever arrives
// on, waits for its first phase with the same wait routines the kernels use (the spinning form and
// the suspend-hint form), gives up after the given limit and reports.  No copy is in flight, nothing
// traps, and the CUDA context stays usable.
#include "device_common.cuh"
#include "pkv_internal.h"

namespace {

__global__ void __launch_bounds__(64) wait_timeout_kernel(unsigned int *err, uint64_t limit_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbarrier_init();
    }
    __syncthreads();
    // warp 0 spins with mbar_wait_for, warp 1 sleeps in the barrier with mbar_wait_sleep; neither
    // phase can complete, so both must give up after limit_ns
    const bool done = threadIdx.x < 32 ? mbar_wait_for(&bar, 0, limit_ns) : mbar_wait_sleep(&bar, 0, limit_ns);
    if (!done && (threadIdx.x & 31) == 0) set_error(err, PKV_DEVERR_TIMEOUT);
}

} // namespace

extern "C" int kv_cache_selftest_wait_timeout(pkv_cache_t c, uint64_t limit_ns, void *stream) {
    PKV_RANGE("kv_cache_selftest_wait_timeout");
    if (!c) return pkv_fail(PKV_EINVAL, "cache is NULL");
    if (limit_ns == 0 || limit_ns > 1000000000ull)
        return pkv_fail(PKV_EINVAL, "limit_ns %llu not in [1, 1e9]", (unsigned long long)limit_ns);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return pkv_cuda_fail(e, "cudaGetDevice");
    if (dev != c->device) return pkv_fail(PKV_EINVAL, "cache lives on device %d but device %d is current", c->device, dev);
    wait_timeout_kernel<<<1, 64, 0, static_cast<cudaStream_t>(stream)>>>(c->err, limit_ns);
    e = cudaGetLastError();
    if (e != cudaSuccess) return pkv_cuda_fail(e, "self-test launch");
    g_pkv_launches++;
    return PKV_OK;
}
