// Instantiations of the tensor-core attention (prefill_impl.cuh) for the prefill over a cached prefix (keys read from the pool through the block table; 16-bit and E4M3 caches).
#include "prefill_impl.cuh"

namespace pkv_prefill {
PKV_ATTN_INSTANTIATE(MODE_PAGED, false)
PKV_ATTN_INSTANTIATE(MODE_PAGED, true)
} // namespace pkv_prefill
