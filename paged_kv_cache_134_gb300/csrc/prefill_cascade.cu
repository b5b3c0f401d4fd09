// Instantiations of the tensor-core attention (prefill_impl.cuh) for the cascade decode's prefix phase (16-bit and E4M3 caches).
#include "prefill_impl.cuh"

namespace pkv_prefill {
PKV_ATTN_INSTANTIATE(MODE_CASCADE, false)
PKV_ATTN_INSTANTIATE(MODE_CASCADE, true)
} // namespace pkv_prefill
