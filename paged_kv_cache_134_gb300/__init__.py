"""GB300-native paged KV cache: paged append, paged decode attention and packed causal
prefill, hand-written CUDA for sm_103a behind the C ABI declared in include/pagedkv.h.

``binding`` marshals torch tensors into that ABI (no computation in Python);
``workloads`` generates the seeded synthetic inputs; ``build`` compiles the library.
"""
from .binding import (KVCache, PagedKVError, PrefixCache, block_hashes, kernel_launches, lib,  # noqa: F401
                      packed_prefill_attention,
                      paged_block_copy, paged_block_swap_in, paged_block_swap_out, paged_decode_attention,
                      paged_decode_attention_cascade,
                      paged_decode_attention_noalloc, paged_kv_append, paged_kv_append_at, paged_prefill_attention,
                      paged_slot_mapping)

__all__ = ["KVCache", "PagedKVError", "PrefixCache", "block_hashes", "kernel_launches", "lib", "packed_prefill_attention", "paged_block_copy",
           "paged_block_swap_in", "paged_block_swap_out", "paged_decode_attention", "paged_decode_attention_cascade", "paged_decode_attention_noalloc",
           "paged_kv_append", "paged_kv_append_at", "paged_prefill_attention", "paged_slot_mapping"]
