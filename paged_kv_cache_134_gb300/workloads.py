"""Seeded synthetic inputs for the paged KV cache hot path.

This module produces data and host-side block bookkeeping only: random Q/K/V
values, sequence lengths, a free-list block allocator with reference counts,
per-sequence block tables, and the (sequence id, position) of every token
that has to be written into the cache.  It holds none of the method's
arithmetic: no slot computation, no cache writes, no attention.  Both the
CUDA path and the CPU oracle consume what it returns and each derives slots,
cache contents and attention outputs on its own.

Workload shapes follow the five synthetic configurations that the paged
decode, packed prefill, prefix sharing and stress sweep are measured on:

* ``tiny``      4 sequences, lengths {1,15,16,37}, 8/8 heads, D=64, bs=16, fp16,
                a 64-block pool handed out from a shuffled free list.
* ``decode7b``  LLaMA-2-7B layer shape: 32 sequences, 32/32 heads, D=128,
                bs=16, fp16, lengths U{1..4096}, pool = 110% of blocks needed.
* ``prefill``   packed causal prefill of 8 sequences with lengths
                128,200,512,1024,2048,256,64,1024 (5256 tokens), 32 heads,
                D=128, bs=16, fp16, blocks from a seeded permutation.
* ``prefix13b`` 13B layer shape: 64 sequences, 40/40 heads, D=128, bs=32,
                a 4096-token prefix (128 blocks) shared by every table
                (ref count 64) plus a private suffix U{1..512}.
* ``prefix_hit_prefill``  16 requests behind one cached 1500-token system prompt (its 93 whole
                blocks shared by every table), each prefilling the prompt's last 12 tokens
                plus a tail of U{100..300} tokens; 32/32 heads, D=128, bs=16, fp16.
* ``stress``    256 sequences, log-normal lengths (median 500, cap 8192),
                32 query / 8 KV heads, D=128, bs in {8,16,32}, KV bf16 or
                FP8-E4M3 with a per-KV-head fp32 scale, block ids drawn from
                a free list fragmented by 3 rounds of allocate/free churn.

The free list follows the manager sketched in "PagedAttention 与前缀缓存"
(2kiu.com, section 2.2): ``allocate`` takes ids from the front and raises
"KV cache block pool exhausted" when short, ``free`` returns them to the
tail, and a per-block reference count records sharing (section 4.3, step 3).
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np
import torch

# dtype names used throughout (the C ABI uses the same order)
F16, BF16, FP8 = "f16", "bf16", "fp8"
DTYPE_CODE = {F16: 0, BF16: 1, FP8: 2}
ELEM_BYTES = {F16: 2, BF16: 2, FP8: 1}
# quiet-NaN bit patterns used to poison every cache slot that no token owns
NAN_BITS = {F16: 0x7E00, BF16: 0x7FC0, FP8: 0x7F}


class PoolExhausted(RuntimeError):
    pass


class BlockAllocator:
    """Host free list of physical block ids with reference counts."""

    def __init__(self, num_blocks: int, rng: np.random.Generator):
        self.num_blocks = int(num_blocks)
        self.free_list: List[int] = [int(b) for b in rng.permutation(self.num_blocks)]
        self.ref_count = np.zeros(self.num_blocks, dtype=np.int32)

    def allocate(self, n: int) -> List[int]:
        if n > len(self.free_list):
            raise PoolExhausted("KV cache block pool exhausted")
        blocks = self.free_list[:n]
        del self.free_list[:n]
        for b in blocks:
            self.ref_count[b] = 1
        return blocks

    def share(self, blocks: List[int]) -> None:
        for b in blocks:
            if self.ref_count[b] <= 0:
                raise ValueError(f"block {b} is not allocated")
            self.ref_count[b] += 1

    def free(self, blocks: List[int]) -> None:
        for b in blocks:
            if self.ref_count[b] <= 0:
                raise ValueError(f"double free of block {b}")
            self.ref_count[b] -= 1
            if self.ref_count[b] == 0:
                self.free_list.append(b)

    @property
    def num_free(self) -> int:
        return len(self.free_list)


def blocks_for(num_tokens: int, block_size: int) -> int:
    """Number of fixed-size blocks that hold ``num_tokens`` tokens."""
    return -(-int(num_tokens) // int(block_size))


def _to_bits(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round float32 values to fp16/bf16 (round-to-nearest-even) and return raw uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    if dtype == F16:
        return t.to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    if dtype == BF16:
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    raise ValueError(dtype)


def bits_to_float(bits: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of raw fp16/bf16 bits to float64 (for brute-force references)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    if dtype == F16:
        return t.view(torch.float16).to(torch.float64).numpy()
    if dtype == BF16:
        return t.view(torch.bfloat16).to(torch.float64).numpy()
    raise ValueError(dtype)


def normal_bits(rng: np.random.Generator, shape, dtype: str, chunk_rows: int = 4096) -> np.ndarray:
    """N(0,1) samples rounded to ``dtype``; generated in row chunks to bound host memory."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    if shape[0] == 0:
        return out
    row = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    flat = out.reshape(shape[0], row)
    for r0 in range(0, shape[0], chunk_rows):
        r1 = min(shape[0], r0 + chunk_rows)
        flat[r0:r1] = _to_bits(rng.standard_normal((r1 - r0, row), dtype=np.float32), dtype)
    return out


@dataclasses.dataclass
class DecodeWorkload:
    """One decode step: append one token per sequence, then attend over L+1 tokens."""

    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    kv_dtype: str
    model_dtype: str
    scale: np.float32
    context_lens: np.ndarray        # int32 [S]   tokens already cached (before the step)
    block_tables: np.ndarray        # int32 [S, max_blocks] covering L+1 tokens, -1 padded
    fill_tables: np.ndarray         # int32 [R, max_blocks] tables used to write the cached tokens
    fill_seq_ids: np.ndarray        # int32 [N]   row of fill_tables for each cached token
    fill_positions: np.ndarray      # int32 [N]   logical position of each cached token
    fill_k: np.ndarray              # uint16 [N, Hkv, D] model-dtype bits
    fill_v: np.ndarray
    q: np.ndarray                   # uint16 [S, Hq, D]
    new_k: np.ndarray               # uint16 [S, Hkv, D]
    new_v: np.ndarray
    k_scale: Optional[np.ndarray]   # float32 [Hkv] (FP8 cache only)
    v_scale: Optional[np.ndarray]
    ref_count: np.ndarray           # int32 [NB]
    seq_fill_row: np.ndarray        # int32 [S] fill row holding each sequence's own tokens
    shared_prefix_len: int = 0      # tokens at the head of every table stored once (row 0)

    @property
    def seq_ids(self) -> np.ndarray:
        return np.arange(self.num_seqs, dtype=np.int32)

    @property
    def positions(self) -> np.ndarray:
        return self.context_lens.astype(np.int32)

    @property
    def decode_lens(self) -> np.ndarray:
        return (self.context_lens + 1).astype(np.int32)

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    def kv_read_bytes(self) -> int:
        """Algorithmic K+V bytes one decode pass reads: sum(L+1) * Hkv * D * elt * 2."""
        return int(self.decode_lens.sum()) * self.num_kv_heads * self.head_dim * ELEM_BYTES[self.kv_dtype] * 2


@dataclasses.dataclass
class PrefillWorkload:
    name: str
    lengths: np.ndarray             # int32 [num_seqs]
    cu_seqlens: np.ndarray          # int32 [num_seqs + 1]
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: str
    scale: np.float32
    q: np.ndarray                   # uint16 [T, Hq, D]
    k: np.ndarray                   # uint16 [T, Hkv, D]
    v: np.ndarray
    block_tables: np.ndarray        # int32 [num_seqs, max_blocks], -1 padded
    kv_dtype: Optional[str] = None  # cache dtype (None: the model dtype)
    k_scale: Optional[np.ndarray] = None  # float32 [Hkv] (FP8 cache only)
    v_scale: Optional[np.ndarray] = None

    def __post_init__(self):
        if self.kv_dtype is None:
            self.kv_dtype = self.dtype

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_seqlen(self) -> int:
        return int(self.lengths.max()) if len(self.lengths) else 0

    def causal_pairs(self) -> int:
        return int(sum(int(n) * (int(n) + 1) // 2 for n in self.lengths))

    def flops(self) -> int:
        """Causal attention flops: 2 contractions * 2 flop/MAC * D per (query, key) pair per head."""
        return 4 * self.head_dim * self.num_q_heads * self.causal_pairs()


@dataclasses.dataclass
class ContextPrefillWorkload:
    """Prefill of each prompt's tail over the prefix its blocks already hold."""

    name: str
    context_lens: np.ndarray        # int32 [S] tokens already cached (a multiple of bs when shared)
    new_lens: np.ndarray            # int32 [S] tail tokens to prefill
    cu_seqlens: np.ndarray          # int32 [S + 1] over the tail tokens
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: str
    scale: np.float32
    block_tables: np.ndarray        # int32 [S, max_blocks] covering context + tail, -1 padded
    fill_seq_ids: np.ndarray        # int32 [N] table row used to write each cached token
    fill_positions: np.ndarray      # int32 [N]
    fill_k: np.ndarray              # uint16 [N, Hkv, D]
    fill_v: np.ndarray
    q: np.ndarray                   # uint16 [T, Hq, D] tail tokens, packed
    k: np.ndarray                   # uint16 [T, Hkv, D]
    v: np.ndarray
    ref_count: np.ndarray           # int32 [NB]
    shared_prefix_len: int = 0      # tokens at the head of every table, stored once
    kv_dtype: Optional[str] = None  # cache dtype (None: the model dtype)
    k_scale: Optional[np.ndarray] = None  # float32 [Hkv] (FP8 cache only)
    v_scale: Optional[np.ndarray] = None

    def __post_init__(self):
        if self.kv_dtype is None:
            self.kv_dtype = self.dtype

    @property
    def num_seqs(self) -> int:
        return len(self.new_lens)

    @property
    def total_tokens(self) -> int:
        return int(self.cu_seqlens[-1])

    @property
    def max_seqlen(self) -> int:
        return int(self.new_lens.max()) if len(self.new_lens) else 0

    def causal_pairs(self) -> int:
        """(query, key) pairs: tail row r of sequence i sees context_i + r + 1 keys."""
        return int(sum(int(n) * int(c) + int(n) * (int(n) + 1) // 2 for c, n in zip(self.context_lens, self.new_lens)))

    def flops(self) -> int:
        return 4 * self.head_dim * self.num_q_heads * self.causal_pairs()


def context_prefill(seed: int = 1006, context_lens=(0, 16, 37, 200), new_lens=(5, 130, 64, 1), shared_prefix: int = 0,
                    heads: int = 4, kv_heads: Optional[int] = None, d: int = 128, bs: int = 16, dtype: str = F16,
                    pool_factor: float = 1.25, kv_dtype: Optional[str] = None) -> ContextPrefillWorkload:
    """Sequences holding context_lens[i] cached tokens get new_lens[i] tail tokens.  With shared_prefix
    > 0 (a multiple of bs) the first shared_prefix tokens of every sequence live once, in blocks every
    table points at (the prefix-cache hit, 2kiu.com section 4.3 step 3); the rest is private."""
    rng = np.random.default_rng(seed)
    prng = np.random.default_rng(seed + 0x9E37)
    ctx = np.asarray(context_lens, dtype=np.int32)
    nl = np.asarray(new_lens, dtype=np.int32)
    S = len(nl)
    hkv = heads if kv_heads is None else kv_heads
    assert shared_prefix % bs == 0 and all(int(c) >= shared_prefix for c in ctx)
    nshared = shared_prefix // bs
    need = nshared + int(sum(blocks_for(int(c) + int(n), bs) - nshared for c, n in zip(ctx, nl)))
    nb = max(1, int(math.ceil(pool_factor * need)))
    alloc = BlockAllocator(nb, prng)
    shared = alloc.allocate(nshared) if nshared else []
    tables = []
    for c, n in zip(ctx, nl):
        if shared:
            alloc.share(shared)
            # the allocator counted the creator's reference already; every table adds one
        tables.append(list(shared) + alloc.allocate(blocks_for(int(c) + int(n), bs) - nshared))
    bt = _tables_array(tables)
    # cached tokens: the shared prefix once (through table 0), every private context token once
    fill_ids, fill_pos = [], []
    if S and shared_prefix:
        fill_ids.append(np.zeros(shared_prefix, np.int32))
        fill_pos.append(np.arange(shared_prefix, dtype=np.int32))
    for i, c in enumerate(ctx):
        fill_ids.append(np.full(int(c) - shared_prefix, i, np.int32))
        fill_pos.append(np.arange(shared_prefix, int(c), dtype=np.int32))
    fill_ids = np.concatenate(fill_ids) if fill_ids else np.zeros(0, np.int32)
    fill_pos = np.concatenate(fill_pos) if fill_pos else np.zeros(0, np.int32)
    N, T = len(fill_ids), int(nl.sum())
    cu = np.zeros(S + 1, dtype=np.int32)
    cu[1:] = np.cumsum(nl)
    fill_k, fill_v = normal_bits(rng, (N, hkv, d), dtype), normal_bits(rng, (N, hkv, d), dtype)
    q, k, v = normal_bits(rng, (T, heads, d), dtype), normal_bits(rng, (T, hkv, d), dtype), \
        normal_bits(rng, (T, hkv, d), dtype)
    ks = vs = None
    if kv_dtype == FP8:
        ks, vs = _fp8_scales(fill_k, k, dtype), _fp8_scales(fill_v, v, dtype)
    return ContextPrefillWorkload(
        name=f"context_prefill_T{T}", context_lens=ctx, new_lens=nl, cu_seqlens=cu, num_q_heads=heads,
        num_kv_heads=hkv, head_dim=d, block_size=bs, num_blocks=nb, dtype=dtype,
        scale=np.float32(1.0 / math.sqrt(d)), block_tables=bt, fill_seq_ids=fill_ids, fill_positions=fill_pos,
        fill_k=fill_k, fill_v=fill_v, q=q, k=k, v=v, ref_count=alloc.ref_count.copy(), shared_prefix_len=shared_prefix,
        kv_dtype=kv_dtype or dtype, k_scale=ks, v_scale=vs)


def prefix_hit_prefill(seed: int = 1006, num_seqs: int = 16, prompt: int = 1500, tail=(100, 300), heads: int = 32,
                       d: int = 128, bs: int = 16, dtype: str = F16,
                       kv_dtype: Optional[str] = None) -> ContextPrefillWorkload:
    """A 1500-token system prompt cached once (its whole blocks: 1488 tokens), then per request the
    prompt's remaining 12 tokens plus a tail of U{100..300} tokens to prefill (the scenario of
    2kiu.com section 3.3: only the tail after the prefix hit is prefilled)."""
    rng = np.random.default_rng(seed ^ 0x5EED)
    hit = (prompt // bs) * bs
    nl = (prompt - hit) + rng.integers(tail[0], tail[1] + 1, size=num_seqs)
    return context_prefill(seed=seed, context_lens=[hit] * num_seqs, new_lens=nl, shared_prefix=hit, heads=heads,
                           d=d, bs=bs, dtype=dtype, pool_factor=1.1, kv_dtype=kv_dtype)


def _tables_array(tables: List[List[int]], max_blocks: Optional[int] = None) -> np.ndarray:
    mb = max_blocks if max_blocks is not None else max(1, max((len(t) for t in tables), default=1))
    arr = np.full((len(tables), mb), -1, dtype=np.int32)
    for i, t in enumerate(tables):
        arr[i, : len(t)] = t
    return arr


def _fp8_scales(fill: np.ndarray, new: np.ndarray, dtype: str) -> np.ndarray:
    """Per-KV-head scale = max(amax of that head's values, 1e-6) / 448 in fp32."""
    amax = np.maximum(np.abs(bits_to_float(fill, dtype)).max(axis=(0, 2)) if len(fill) else 0.0,
                      np.abs(bits_to_float(new, dtype)).max(axis=(0, 2)))
    return (np.maximum(amax, 1e-6) / 448.0).astype(np.float32)


def _decode_from_lens(name, lens, *, hq, hkv, d, bs, kv_dtype, model_dtype, seed,
                      pool_factor=1.1, num_blocks=None, churn_rounds=0, len_sampler=None,
                      placement_seed=None) -> DecodeWorkload:
    # values and block placement draw from separate streams, so a different pool size or
    # placement seed moves the same logical data to different physical blocks
    rng = np.random.default_rng(seed)
    prng = np.random.default_rng(seed + 0x9E37 if placement_seed is None else placement_seed)
    lens = np.asarray(lens, dtype=np.int32)
    S = len(lens)
    need = int(sum(blocks_for(L + 1, bs) for L in lens))
    nb = int(num_blocks) if num_blocks is not None else int(math.ceil(pool_factor * need))
    alloc = BlockAllocator(nb, prng)
    if churn_rounds:
        _churn(alloc, prng, bs, churn_rounds, len_sampler)
    tables = [alloc.allocate(blocks_for(L + 1, bs)) for L in lens]
    bt = _tables_array(tables)
    n = int(lens.sum())
    fill_ids = np.repeat(np.arange(S, dtype=np.int32), lens)
    fill_pos = np.concatenate([np.arange(L, dtype=np.int32) for L in lens]) if n else np.zeros(0, np.int32)
    fill_k = normal_bits(rng, (n, hkv, d), model_dtype)
    fill_v = normal_bits(rng, (n, hkv, d), model_dtype)
    q = normal_bits(rng, (S, hq, d), model_dtype)
    new_k = normal_bits(rng, (S, hkv, d), model_dtype)
    new_v = normal_bits(rng, (S, hkv, d), model_dtype)
    ks = vs = None
    if kv_dtype == FP8:
        ks = _fp8_scales(fill_k, new_k, model_dtype)
        vs = _fp8_scales(fill_v, new_v, model_dtype)
    return DecodeWorkload(
        name=name, num_seqs=S, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
        num_blocks=nb, kv_dtype=kv_dtype, model_dtype=model_dtype,
        scale=np.float32(1.0 / math.sqrt(d)), context_lens=lens, block_tables=bt,
        fill_tables=bt, fill_seq_ids=fill_ids, fill_positions=fill_pos, fill_k=fill_k, fill_v=fill_v,
        q=q, new_k=new_k, new_v=new_v, k_scale=ks, v_scale=vs, ref_count=alloc.ref_count.copy(),
        seq_fill_row=np.arange(S, dtype=np.int32))


def _lognormal_lens(rng, n, median=500.0, sigma=1.0, cap=8192):
    x = np.exp(rng.normal(math.log(median), sigma, size=n))
    return np.clip(np.rint(x), 1, cap).astype(np.int32)


def _churn(alloc: BlockAllocator, rng, bs, rounds, len_sampler):
    """Fragment the free list: fill >=90% of the pool with dummy sequences, free half, repeat."""
    live: List[List[int]] = []
    for _ in range(rounds):
        while alloc.num_blocks - alloc.num_free < 0.9 * alloc.num_blocks:
            nblk = blocks_for(int(len_sampler(rng, 1)[0]), bs)
            if nblk > alloc.num_free:
                break
            live.append(alloc.allocate(nblk))
        order = rng.permutation(len(live))
        keep = []
        for i, j in enumerate(order):
            if i < len(order) // 2:
                alloc.free(live[j])
            else:
                keep.append(live[j])
        live = keep
    for j in rng.permutation(len(live)):
        alloc.free(live[j])


# ----------------------------------------------------------------------------------------------
# the five configurations (seed = 1000 + config number)

def tiny(seed: int = 1001) -> DecodeWorkload:
    return _decode_from_lens("tiny", [1, 15, 16, 37], hq=8, hkv=8, d=64, bs=16,
                             kv_dtype=F16, model_dtype=F16, seed=seed, num_blocks=64)


def decode7b(seed: int = 1002, num_seqs: int = 32, max_len: int = 4096) -> DecodeWorkload:
    rng = np.random.default_rng(seed ^ 0x5EED)
    lens = rng.integers(1, max_len + 1, size=num_seqs, dtype=np.int64).astype(np.int32)
    return _decode_from_lens(f"decode7b_S{num_seqs}", lens, hq=32, hkv=32, d=128, bs=16,
                             kv_dtype=F16, model_dtype=F16, seed=seed)


PACKED_LENGTHS = (128, 200, 512, 1024, 2048, 256, 64, 1024)


def prefill(seed: int = 1003, lengths=PACKED_LENGTHS, heads: int = 32, kv_heads: Optional[int] = None,
            d: int = 128, bs: int = 16, dtype: str = F16, pool_factor: float = 1.1,
            kv_dtype: Optional[str] = None) -> PrefillWorkload:
    rng = np.random.default_rng(seed)
    lengths = np.asarray(lengths, dtype=np.int32)
    hkv = heads if kv_heads is None else kv_heads
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lengths)
    need = int(sum(blocks_for(n, bs) for n in lengths))
    nb = max(1, int(math.ceil(pool_factor * need)))
    alloc = BlockAllocator(nb, rng)
    tables = [alloc.allocate(blocks_for(n, bs)) for n in lengths]
    T = int(cu[-1])
    q, k, v = normal_bits(rng, (T, heads, d), dtype), normal_bits(rng, (T, hkv, d), dtype), \
        normal_bits(rng, (T, hkv, d), dtype)
    ks = vs = None
    if kv_dtype == FP8:
        empty = np.zeros((0, hkv, d), np.uint16)
        ks, vs = _fp8_scales(empty, k, dtype), _fp8_scales(empty, v, dtype)
    return PrefillWorkload(
        name=f"prefill_T{T}", lengths=lengths, cu_seqlens=cu, num_q_heads=heads, num_kv_heads=hkv,
        head_dim=d, block_size=bs, num_blocks=nb, dtype=dtype, scale=np.float32(1.0 / math.sqrt(d)),
        q=q, k=k, v=v, block_tables=_tables_array(tables), kv_dtype=kv_dtype or dtype, k_scale=ks, v_scale=vs)


def prefix13b(seed: int = 1004, num_seqs: int = 64, prefix_tokens: int = 4096, max_suffix: int = 512,
              heads: int = 40, d: int = 128, bs: int = 32, private_prefix: bool = False,
              kv_heads: Optional[int] = None, dtype: str = F16, kv_dtype: Optional[str] = None) -> DecodeWorkload:
    """Shared-prefix decode.  ``private_prefix`` gives every sequence its own copy of the prefix
    blocks (same values, different physical blocks) for the shared-vs-private equality check."""
    rng = np.random.default_rng(seed)
    suffix = rng.integers(1, max_suffix + 1, size=num_seqs, dtype=np.int64).astype(np.int32)
    lens = (prefix_tokens + suffix).astype(np.int32)
    assert prefix_tokens % bs == 0
    pblk = prefix_tokens // bs
    need = pblk * (num_seqs if private_prefix else 1) + sum(blocks_for(s + 1, bs) for s in suffix)
    nb = int(math.ceil(1.1 * need))
    alloc = BlockAllocator(nb, np.random.default_rng(seed + 77))
    hkv = heads if kv_heads is None else kv_heads
    pk = normal_bits(rng, (prefix_tokens, hkv, d), dtype)
    pv = normal_bits(rng, (prefix_tokens, hkv, d), dtype)
    sk = [normal_bits(rng, (int(s), hkv, d), dtype) for s in suffix]
    sv = [normal_bits(rng, (int(s), hkv, d), dtype) for s in suffix]
    q = normal_bits(rng, (num_seqs, heads, d), dtype)
    new_k = normal_bits(rng, (num_seqs, hkv, d), dtype)
    new_v = normal_bits(rng, (num_seqs, hkv, d), dtype)
    tables = []
    fill_tables = []
    ids, pos, fk, fv = [], [], [], []
    if not private_prefix:
        shared = alloc.allocate(pblk)
        fill_tables.append(list(shared))
        ids.append(np.zeros(prefix_tokens, np.int32)); pos.append(np.arange(prefix_tokens, dtype=np.int32))
        fk.append(pk); fv.append(pv)
    for s in range(num_seqs):
        if private_prefix:
            pre = alloc.allocate(pblk)
        else:
            pre = list(shared)
            alloc.share(shared)
        own = alloc.allocate(blocks_for(int(lens[s]) + 1, bs) - pblk)
        tables.append(pre + own)
        fill_tables.append(pre + own)
        row = len(fill_tables) - 1
        if private_prefix:
            ids.append(np.full(prefix_tokens, row, np.int32)); pos.append(np.arange(prefix_tokens, dtype=np.int32))
            fk.append(pk); fv.append(pv)
        ids.append(np.full(int(suffix[s]), row, np.int32))
        pos.append(np.arange(prefix_tokens, int(lens[s]), dtype=np.int32))
        fk.append(sk[s]); fv.append(sv[s])
    if not private_prefix:
        # the creating sequence's reference is dropped once the prefill that wrote it is done
        alloc.free(shared)
    mb = max(len(t) for t in fill_tables)
    fill_k, fill_v = np.concatenate(fk), np.concatenate(fv)
    ks = vs = None
    if kv_dtype == FP8:
        ks, vs = _fp8_scales(fill_k, new_k, dtype), _fp8_scales(fill_v, new_v, dtype)
    return DecodeWorkload(
        name="prefix13b" + ("_private" if private_prefix else ""), num_seqs=num_seqs, num_q_heads=heads,
        num_kv_heads=hkv, head_dim=d, block_size=bs, num_blocks=nb, kv_dtype=kv_dtype or dtype, model_dtype=dtype,
        scale=np.float32(1.0 / math.sqrt(d)), context_lens=lens, block_tables=_tables_array(tables, mb),
        fill_tables=_tables_array(fill_tables, mb), fill_seq_ids=np.concatenate(ids),
        fill_positions=np.concatenate(pos), fill_k=fill_k, fill_v=fill_v,
        q=q, new_k=new_k, new_v=new_v, k_scale=ks, v_scale=vs, ref_count=alloc.ref_count.copy(),
        seq_fill_row=np.arange(num_seqs, dtype=np.int32) + (0 if private_prefix else 1),
        shared_prefix_len=0 if private_prefix else prefix_tokens)


def stress(bs: int = 16, kv_dtype: str = BF16, seed: int = 1005, num_seqs: int = 256) -> DecodeWorkload:
    rng = np.random.default_rng(seed)
    lens = _lognormal_lens(rng, num_seqs)
    need = int(sum(blocks_for(L + 1, bs) for L in lens))
    return _decode_from_lens(f"stress_bs{bs}_{kv_dtype}", lens, hq=32, hkv=8, d=128, bs=bs,
                             kv_dtype=kv_dtype, model_dtype=BF16, seed=seed + 1,
                             num_blocks=int(math.ceil(1.5 * need)), churn_rounds=3,
                             len_sampler=lambda r, n: _lognormal_lens(r, n))


def small_decode(name, lens, *, hq, hkv, d, bs, kv_dtype=F16, model_dtype=None, seed=7,
                 num_blocks=None, pool_factor=1.5, placement_seed=None) -> DecodeWorkload:
    """Arbitrary small decode case for edge-case tests."""
    md = model_dtype or (kv_dtype if kv_dtype != FP8 else BF16)
    return _decode_from_lens(name, lens, hq=hq, hkv=hkv, d=d, bs=bs, kv_dtype=kv_dtype,
                             model_dtype=md, seed=seed, num_blocks=num_blocks, pool_factor=pool_factor,
                             placement_seed=placement_seed)


def logical_kv(w: DecodeWorkload, s: int):
    """Per-sequence logical K/V bits [L+1, Hkv, D] in position order (cached tokens + the new one).

    Used only by brute-force references that never look at block tables."""
    rows = [w.seq_fill_row[s]]
    if w.shared_prefix_len:
        rows = [0, w.seq_fill_row[s]]
    sel = np.isin(w.fill_seq_ids, rows)
    pos = w.fill_positions[sel]
    order = np.argsort(pos, kind="stable")
    k = np.concatenate([w.fill_k[sel][order], w.new_k[s:s + 1]])
    v = np.concatenate([w.fill_v[sel][order], w.new_v[s:s + 1]])
    assert len(k) == int(w.context_lens[s]) + 1
    return k, v


def kv_bytes_per_token(layers: int, kv_heads: int, head_dim: int, elem_bytes: int) -> int:
    """KV bytes one token costs: 2 (K and V) x layers x KV heads x head_dim x bytes per element
    (2kiu.com "PagedAttention 与前缀缓存", section 1.1)."""
    return 2 * int(layers) * int(kv_heads) * int(head_dim) * int(elem_bytes)


def pool_capacity_blocks(budget_bytes: int, block_size: int, bytes_per_token: int) -> int:
    """Whole blocks that fit a KV budget (discosf.com "Paged KV Cache 与 Packed Sequence", section 4.1)."""
    return int(budget_bytes) // (int(block_size) * int(bytes_per_token))
