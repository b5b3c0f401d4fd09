"""Hot-path passes composed from the library's calls (all work runs in the CUDA kernels).

A decode step, in the order the pages give it ("Paged KV Cache 与 Packed Sequence",
discosf.com, section 4.3; "PagedAttention 与前缀缓存", 2kiu.com, section 4.1): slot indexing
of the new tokens -> paged append of their K/V -> paged decode attention.  A prefill step:
packed causal prefill, which also writes every token's K/V into its blocks (discosf.com
sections 3.3 and 4.2).  Helpers move the seeded host workloads to the device.
"""
import numpy as np
import torch

import paged_kv_cache_134_gb300 as P
from paged_kv_cache_134_gb300 import workloads as W

TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def dev(a: np.ndarray, dtype=None) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        t = torch.from_numpy(a.view(np.int16)).cuda()
        return t.view(dtype) if dtype is not None else t
    return torch.from_numpy(a).cuda()


def new_cache(w_like, num_blocks, block_size, hkv, d, kv_dtype, model_dtype, k_scale=None, v_scale=None):
    cache = P.KVCache(num_blocks, block_size, hkv, d, kv_dtype, model_dtype)
    if kv_dtype == "fp8":
        cache.set_scales(dev(k_scale), dev(v_scale))
    bits = W.NAN_BITS[kv_dtype]
    pool = cache.pool_elems()
    pool.fill_(bits if kv_dtype == "fp8" else int(np.array([bits], np.uint16).view(np.int16)[0]))
    return cache


def pool_numpy(cache) -> np.ndarray:
    p = cache.pool_elems().cpu().numpy()
    return p if cache.kv_dtype == "fp8" else p.view(np.uint16)


def fill_cache(cache, w):
    """Write every cached context token of a DecodeWorkload; returns the slots used."""
    md = TORCH_DT[w.model_dtype]
    slots = P.paged_slot_mapping(dev(w.fill_tables), dev(w.fill_seq_ids), dev(w.fill_positions), w.block_size)
    if len(w.fill_seq_ids):
        P.paged_kv_append(cache, dev(w.fill_k, md), dev(w.fill_v, md), slots)
    return slots


class DecodeInputs:
    """Device-resident inputs of one decode step."""

    def __init__(self, w):
        md = TORCH_DT[w.model_dtype]
        self.tables = dev(w.block_tables)
        self.seq_ids = dev(np.arange(w.num_seqs, dtype=np.int32))
        self.positions = dev(w.context_lens.astype(np.int32))
        self.lens = dev(w.decode_lens)
        self.q = dev(w.q, md)
        self.new_k = dev(w.new_k, md)
        self.new_v = dev(w.new_v, md)
        self.out = torch.empty_like(self.q)
        self.slots = torch.empty(w.num_seqs, dtype=torch.int64, device="cuda")
        self.scale = float(w.scale)
        self.block_size = w.block_size


def decode_step(cache, x: DecodeInputs, fused: bool = True, cascade_prefix: int = 0):
    """One decode step: slot indexing -> append of the new token -> paged decode attention.

    ``fused`` computes the slots inside the append launch (paged_kv_append_at); otherwise slot
    indexing and append are two launches.  Both write the same slots and the same bytes.
    ``cascade_prefix`` > 0: the tables share their first that many tokens, and the attention runs
    as a cascade decode (the shared prefix read once for the batch)."""
    if fused:
        P.paged_kv_append_at(cache, x.new_k, x.new_v, x.tables, x.seq_ids, x.positions, x.slots)
    else:
        P.paged_slot_mapping(x.tables, x.seq_ids, x.positions, x.block_size, out=x.slots)
        P.paged_kv_append(cache, x.new_k, x.new_v, x.slots)
    if cascade_prefix:
        P.paged_decode_attention_cascade(x.q, cache, x.tables, x.lens, cascade_prefix, x.scale, out=x.out)
    else:
        P.paged_decode_attention(x.q, cache, x.tables, x.lens, x.scale, out=x.out)
    return x.out


def run_decode(w, keep_cache=False, fused=True, cascade_prefix=0):
    cache = new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype, w.model_dtype,
                      w.k_scale, w.v_scale)
    fill_slots = fill_cache(cache, w)
    x = DecodeInputs(w)
    out = decode_step(cache, x, fused=fused, cascade_prefix=cascade_prefix)
    torch.cuda.synchronize()
    res = dict(fill_slots=fill_slots.cpu().numpy(), new_slots=x.slots.cpu().numpy(),
               out=out.float().cpu().double().numpy(), err=cache.check_error(),
               strides=cache.view()[1], pool=pool_numpy(cache))
    if keep_cache:
        res["cache"], res["inputs"] = cache, x
    else:
        cache.close()
    return res


def run_prefill(w, keep_cache=False):
    md = TORCH_DT[w.dtype]
    cache = new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype, w.dtype, w.k_scale,
                      w.v_scale)
    q, k, v = dev(w.q, md), dev(w.k, md), dev(w.v, md)
    out = P.packed_prefill_attention(q, k, v, dev(w.cu_seqlens), w.max_seqlen, dev(w.block_tables), cache,
                                     float(w.scale))
    torch.cuda.synchronize()
    res = dict(out=out.float().cpu().double().numpy(), err=cache.check_error(), strides=cache.view()[1],
               pool=pool_numpy(cache))
    if keep_cache:
        res["cache"] = cache
    else:
        cache.close()
    return res



class ContextPrefillInputs:
    """Device-resident inputs of a prefill over cached prefixes."""

    def __init__(self, w):
        md = TORCH_DT[w.dtype]
        self.q, self.k, self.v = dev(w.q, md), dev(w.k, md), dev(w.v, md)
        self.cu = dev(w.cu_seqlens)
        self.ctx = dev(w.context_lens.astype(np.int32))
        self.tables = dev(w.block_tables)
        self.out = torch.empty_like(self.q)
        self.max_seqlen = w.max_seqlen
        self.scale = float(w.scale)


def fill_context(cache, w):
    """Write the cached tokens of a ContextPrefillWorkload (the shared prefix once)."""
    md = TORCH_DT[w.dtype]
    if len(w.fill_seq_ids):
        slots = P.paged_slot_mapping(dev(w.block_tables), dev(w.fill_seq_ids), dev(w.fill_positions), w.block_size)
        P.paged_kv_append(cache, dev(w.fill_k, md), dev(w.fill_v, md), slots)


def context_prefill_step(cache, x: ContextPrefillInputs):
    return P.paged_prefill_attention(x.q, x.k, x.v, x.cu, x.ctx, x.max_seqlen, x.tables, cache, x.scale, out=x.out)


def run_context_prefill(w, keep_cache=False):
    cache = new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype, w.dtype, w.k_scale,
                      w.v_scale)
    fill_context(cache, w)
    x = ContextPrefillInputs(w)
    out = context_prefill_step(cache, x)
    torch.cuda.synchronize()
    res = dict(out=out.float().cpu().double().numpy(), err=cache.check_error(), strides=cache.view()[1],
               pool=pool_numpy(cache))
    if keep_cache:
        res["cache"], res["inputs"] = cache, x
    else:
        cache.close()
    return res
