// Instantiations of the tensor-core attention (prefill_impl.cuh) for the packed prefill (keys from the packed k, v; fused paged K/V write).
#include "prefill_impl.cuh"

namespace pkv_prefill {
PKV_ATTN_INSTANTIATE(MODE_PACKED, false)
} // namespace pkv_prefill
