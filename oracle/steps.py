"""Whole hot-path passes composed from the oracle's functions (TEST INFRASTRUCTURE ONLY).

A decode step, as the pages order it (discosf.com "Paged KV Cache 与 Packed
Sequence", section 4.3; 2kiu.com "PagedAttention 与前缀缓存", section 4.1):
slot indexing for every token -> write the cached context and the new token's
K/V at their slots -> attention of each sequence over its L+1 tokens.

A prefill step (discosf.com sections 3.3 and 4.2): block-diagonal causal
attention over the packed sequences, plus the write of every token's K/V into
block_table[i][r / bs] at offset r % bs.

A prefill on a cached prefix (2kiu.com section 4.3 steps 2-4): the cached
tokens are written first (once for a shared prefix), then the tail tokens'
K/V at positions context + r, then attention of the tail rows over every key
of their sequence, read through the table.
"""
from __future__ import annotations

import numpy as np

from . import contiguous_strides, kv_append, new_pool, packed_prefill, paged_decode, prefill_ctx, slot_mapping

_NAN = {"f16": 0x7E00, "bf16": 0x7FC0, "fp8": 0x7F}


def decode_step(w, strides=None, pool_elems=None, with_psum=False):
    """Returns dict(fill_slots, new_slots, pool, out[, psum]) for a DecodeWorkload."""
    st = contiguous_strides(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim) if strides is None \
        else np.asarray(strides, np.int64)
    n_elems = pool_elems if pool_elems is not None else w.num_blocks * 2 * w.num_kv_heads * w.block_size * w.head_dim
    pool = new_pool(n_elems, w.kv_dtype, _NAN[w.kv_dtype])
    fill_slots = slot_mapping(w.fill_tables, w.fill_seq_ids, w.fill_positions, w.block_size)
    new_slots = slot_mapping(w.block_tables, np.arange(w.num_seqs, dtype=np.int32), w.context_lens, w.block_size)
    bad = kv_append(pool, st, w.kv_dtype, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim,
                    w.fill_k, w.fill_v, w.model_dtype, fill_slots, w.k_scale, w.v_scale)
    bad += kv_append(pool, st, w.kv_dtype, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim,
                     w.new_k, w.new_v, w.model_dtype, new_slots, w.k_scale, w.v_scale)
    assert bad == 0, "workload produced slots outside the pool"
    res = paged_decode(w.q, w.model_dtype, pool, st, w.kv_dtype, w.num_blocks, w.block_tables,
                       w.context_lens + 1, w.num_kv_heads, w.block_size, float(w.scale),
                       w.k_scale, w.v_scale, with_psum=with_psum)
    out = dict(fill_slots=fill_slots, new_slots=new_slots, pool=pool)
    if with_psum:
        out["out"], out["psum"] = res
    else:
        out["out"] = res
    return out


def prefill_step(w, strides=None, pool_elems=None):
    """Returns dict(slots, pool, out) for a PrefillWorkload (cache starts NaN-filled)."""
    st = contiguous_strides(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim) if strides is None \
        else np.asarray(strides, np.int64)
    n_elems = pool_elems if pool_elems is not None else w.num_blocks * 2 * w.num_kv_heads * w.block_size * w.head_dim
    pool = new_pool(n_elems, w.kv_dtype, _NAN[w.kv_dtype])
    seq_ids = np.repeat(np.arange(len(w.lengths), dtype=np.int32), w.lengths)
    positions = np.concatenate([np.arange(n, dtype=np.int32) for n in w.lengths]) if len(w.lengths) else \
        np.zeros(0, np.int32)
    slots = slot_mapping(w.block_tables, seq_ids, positions, w.block_size)
    bad = kv_append(pool, st, w.kv_dtype, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.k, w.v, w.dtype,
                    slots, w.k_scale, w.v_scale)
    assert bad == 0
    out = packed_prefill(w.q, w.k, w.v, w.dtype, w.cu_seqlens, float(w.scale))
    return dict(slots=slots, pool=pool, out=out)


def context_prefill_step(w, strides=None, pool_elems=None):
    """Returns dict(fill_slots, new_slots, pool, out) for a ContextPrefillWorkload."""
    st = contiguous_strides(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim) if strides is None \
        else np.asarray(strides, np.int64)
    n_elems = pool_elems if pool_elems is not None else w.num_blocks * 2 * w.num_kv_heads * w.block_size * w.head_dim
    pool = new_pool(n_elems, w.kv_dtype, _NAN[w.kv_dtype])
    fill_slots = slot_mapping(w.block_tables, w.fill_seq_ids, w.fill_positions, w.block_size)
    bad = kv_append(pool, st, w.kv_dtype, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.fill_k, w.fill_v,
                    w.dtype, fill_slots, w.k_scale, w.v_scale)
    seq_ids = np.repeat(np.arange(w.num_seqs, dtype=np.int32), w.new_lens)
    positions = np.concatenate([c + np.arange(n, dtype=np.int32) for c, n in zip(w.context_lens, w.new_lens)]) \
        if w.total_tokens else np.zeros(0, np.int32)
    new_slots = slot_mapping(w.block_tables, seq_ids, positions, w.block_size)
    bad += kv_append(pool, st, w.kv_dtype, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.k, w.v, w.dtype,
                     new_slots, w.k_scale, w.v_scale)
    assert bad == 0, "workload produced slots outside the pool"
    out = prefill_ctx(w.q, w.dtype, pool, st, w.kv_dtype, w.num_blocks, w.block_tables, w.cu_seqlens, w.context_lens,
                      w.num_kv_heads, w.block_size, float(w.scale), w.k_scale, w.v_scale)
    return dict(fill_slots=fill_slots, new_slots=new_slots, pool=pool, out=out)
