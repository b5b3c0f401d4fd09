"""Pins of the oracle's prefill-on-a-cached-prefix and whole-block copy functions (no GPU needed).

Prefill over a cached prefix (2kiu.com "PagedAttention 与前缀缓存", section 4.3 steps 2-4) is pinned
to things other than itself:
* textbook causal attention (numpy) on each sequence's contiguous logical K/V, with the query rows
  offset by the cached length, computed from the generator's token arrays and never from tables;
* a zero-length context reduces it to the packed prefill, and every tail row to a paged decode of
  the sequence cut after that row (both pinned in test_oracle.py);
* cutting a tail into two chunks changes nothing; a prefix stored once for every table equals
  private copies.

Block copy and swap (2kiu.com sections 2.2, 4.3 step 3 and 5.2) are pinned by their consequences:
decode through a table that points at copied (or swapped-out-and-back) blocks gives the bitwise
same output, a write into a copy leaves the original untouched (copy-on-write), everything that is
not a destination keeps its bytes, and the swap buffer holds each token's K/V where the documented
block layout puts it.
"""
import numpy as np
import pytest

import oracle
from oracle import steps
from paged_kv_cache_134_gb300 import workloads as W


# ------------------------------------------------------------------------------ prefill on a cached prefix

def logical_tokens(w, i):
    """Sequence i's K/V bits in position order: cached tokens (from the fill lists), then the tail."""
    n_ctx = int(w.context_lens[i])
    k = np.zeros((n_ctx, w.num_kv_heads, w.head_dim), np.uint16)
    v = np.zeros_like(k)
    for j, (s, p) in enumerate(zip(w.fill_seq_ids, w.fill_positions)):
        if s == i or (p < w.shared_prefix_len and s == 0):
            k[p], v[p] = w.fill_k[j], w.fill_v[j]
    a, b = w.cu_seqlens[i], w.cu_seqlens[i + 1]
    return np.concatenate([k, w.k[a:b]]), np.concatenate([v, w.v[a:b]])


def brute_context_prefill(w):
    T, hq, d = w.q.shape
    G = hq // w.num_kv_heads
    q = W.bits_to_float(w.q, w.dtype)
    out = np.zeros((T, hq, d))
    for i in range(w.num_seqs):
        kb, vb = logical_tokens(w, i)
        K, V = W.bits_to_float(kb, w.dtype), W.bits_to_float(vb, w.dtype)
        c0 = int(w.context_lens[i])
        for r in range(int(w.new_lens[i])):
            row = w.cu_seqlens[i] + r
            for h in range(hq):
                x = float(w.scale) * (K[: c0 + r + 1, h // G, :] @ q[row, h])
                p = np.exp(x - x.max())
                p /= p.sum()
                out[row, h] = p @ V[: c0 + r + 1, h // G, :]
    return out


CTX_CASES = [
    dict(context_lens=(0, 16, 37, 200), new_lens=(5, 130, 64, 1), heads=4, kv_heads=4, d=64, bs=16),
    dict(context_lens=(7, 64, 1), new_lens=(3, 70, 129), heads=4, kv_heads=1, d=64, bs=8),
    dict(context_lens=(32, 32, 32), new_lens=(1, 40, 9), shared_prefix=32, heads=2, kv_heads=2, d=64, bs=32),
    dict(context_lens=(48, 50), new_lens=(20, 3), shared_prefix=48, heads=4, kv_heads=2, d=128, bs=16, dtype="bf16"),
]


@pytest.mark.parametrize("case", CTX_CASES, ids=lambda c: f"G{c['heads'] // c['kv_heads']}_d{c['d']}_bs{c['bs']}"
                                                         f"_sh{c.get('shared_prefix', 0)}")
def test_context_prefill_matches_contiguous_brute_force(case):
    w = W.context_prefill(seed=61, **case)
    r = steps.context_prefill_step(w)
    assert np.allclose(r["out"], brute_context_prefill(w), rtol=0, atol=1e-12)


def test_context_prefill_zero_context_is_the_packed_prefill():
    w = W.context_prefill(seed=62, context_lens=(0, 0, 0), new_lens=(1, 65, 200), heads=4, kv_heads=2, d=64)
    r = steps.context_prefill_step(w)
    ref = oracle.packed_prefill(w.q, w.k, w.v, w.dtype, w.cu_seqlens, float(w.scale))
    assert np.allclose(r["out"], ref, rtol=0, atol=1e-12)


def test_context_prefill_rows_are_decodes_of_the_cut_sequence():
    w = W.context_prefill(seed=63, context_lens=(19, 40), new_lens=(6, 33), heads=4, kv_heads=2, d=64, bs=8)
    r = steps.context_prefill_step(w)
    st = oracle.contiguous_strides(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    for i in range(w.num_seqs):
        for rr in range(int(w.new_lens[i])):
            row = w.cu_seqlens[i] + rr
            lens = np.array([w.context_lens[i] + rr + 1], np.int32)
            dec = oracle.paged_decode(w.q[row:row + 1], w.dtype, r["pool"], st, w.dtype, w.num_blocks,
                                      w.block_tables[i:i + 1], lens, w.num_kv_heads, w.block_size, float(w.scale))
            assert np.allclose(dec[0], r["out"][row], rtol=0, atol=1e-12)


def test_context_prefill_chunks_equal_the_whole_tail():
    w = W.context_prefill(seed=64, context_lens=(23,), new_lens=(150,), heads=2, kv_heads=2, d=64, bs=16)
    r = steps.context_prefill_step(w)
    st = oracle.contiguous_strides(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    n1 = 61   # the first chunk is prefilled (the pool holds every token); prefill the rest as a second chunk
    out2 = oracle.prefill_ctx(w.q[n1:], w.dtype, r["pool"], st, w.dtype, w.num_blocks, w.block_tables,
                              np.array([0, 150 - n1], np.int32), np.array([23 + n1], np.int32), w.num_kv_heads,
                              w.block_size, float(w.scale))
    assert np.array_equal(out2, r["out"][n1:])


def test_context_prefill_shared_prefix_equals_private_copies():
    kw = dict(seed=65, context_lens=(32, 32, 45), new_lens=(10, 70, 3), heads=2, kv_heads=2, d=64, bs=16)
    shared = W.context_prefill(shared_prefix=32, **kw)
    private = W.context_prefill(shared_prefix=0, **kw)
    rs = steps.context_prefill_step(shared)
    assert np.array_equal(shared.block_tables[:, :2], np.repeat(shared.block_tables[:1, :2], 3, axis=0))
    assert shared.ref_count[shared.block_tables[0, 0]] == 4
    # rebuild the private workload's cached values from the shared one so that only placement differs
    pfill_k, pfill_v = [], []
    for s, p in zip(private.fill_seq_ids, private.fill_positions):
        k, v = logical_tokens(shared, int(s))
        pfill_k.append(k[p])
        pfill_v.append(v[p])
    private.fill_k = np.stack(pfill_k)
    private.fill_v = np.stack(pfill_v)
    private.q, private.k, private.v = shared.q, shared.k, shared.v
    rp = steps.context_prefill_step(private)
    assert np.array_equal(rs["out"], rp["out"])


def test_prefix_hit_prefill_config_shape():
    w = W.prefix_hit_prefill()
    assert w.num_seqs == 16 and int(w.context_lens[0]) == 1488 and w.shared_prefix_len == 1488
    assert np.all((w.new_lens >= 112) & (w.new_lens <= 312))
    assert np.all(w.block_tables[:, :93] == w.block_tables[0, :93])
    assert w.ref_count[w.block_tables[0, 0]] == 17


# ------------------------------------------------------------------------------ block copy and swap

def _decode(w, pool, tables, lens):
    st = oracle.contiguous_strides(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    return oracle.paged_decode(w.q, w.model_dtype, pool, st, w.kv_dtype, w.num_blocks, tables, lens,
                               w.num_kv_heads, w.block_size, float(w.scale), w.k_scale, w.v_scale)


def _free_blocks(w, n):
    used = set(int(b) for b in w.block_tables.ravel() if b >= 0)
    free = [b for b in range(w.num_blocks) if b not in used]
    assert len(free) >= n
    return np.array(free[:n], np.int32)


@pytest.mark.parametrize("kv_dtype", ["f16", "fp8"])
def test_block_copy_is_copy_on_write(kv_dtype):
    w = W.small_decode("cow", [37, 20], hq=4, hkv=2, d=64, bs=16, kv_dtype=kv_dtype, seed=71, pool_factor=3.0)
    r = steps.decode_step(w)
    pool = r["pool"]
    st = oracle.contiguous_strides(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    lens = w.decode_lens
    before = pool.copy()
    src = w.block_tables[0, :3].astype(np.int32)
    dst = _free_blocks(w, 3)
    assert oracle.block_copy(pool, st, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, src, dst) == 0
    # only the destinations changed
    per = pool.size // w.num_blocks
    changed = np.nonzero((pool != before).reshape(w.num_blocks, per).any(axis=1))[0]
    assert set(changed.tolist()) <= set(dst.tolist())
    # the forked table reads the copies and sees the same attention output
    forked = w.block_tables.copy()
    forked[0, :3] = dst
    assert np.array_equal(_decode(w, pool, forked, lens), _decode(w, pool, w.block_tables, lens))
    # a new token written through the fork lands in the copy only
    slot = oracle.slot_mapping(forked, np.array([0], np.int32), np.array([lens[0]], np.int32), w.block_size)
    k = np.full((1, w.num_kv_heads, w.head_dim), 0x3C00, np.uint16)   # 1.0
    oracle.kv_append(pool, st, kv_dtype, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, k, k,
                     w.model_dtype, slot, w.k_scale, w.v_scale)
    lens2 = lens.copy()
    lens2[0] += 1
    assert np.array_equal(_decode(w, pool, w.block_tables, lens), _decode(w, before, w.block_tables, lens))
    assert not np.array_equal(_decode(w, pool, forked, lens2)[0], _decode(w, pool, forked, lens)[0])


def test_block_copy_skips_and_counts_bad_ids():
    pool = np.arange(4 * 2 * 1 * 8 * 8, dtype=np.uint16)
    st = oracle.contiguous_strides(4, 1, 8, 8)
    before = pool.copy()
    bad = oracle.block_copy(pool, st, 4, 8, 1, 8, np.array([0, 5, -1, 2], np.int32), np.array([1, 2, 3, 4], np.int32))
    assert bad == 3
    p, b = pool.reshape(4, -1), before.reshape(4, -1)
    assert np.array_equal(p[1], b[0]) and np.array_equal(p[0], b[0])
    assert np.array_equal(p[2:], b[2:])


def test_swap_out_layout_and_round_trip_into_other_blocks():
    w = W.small_decode("swap", [40, 9], hq=4, hkv=2, d=64, bs=16, seed=72, pool_factor=3.0)
    r = steps.decode_step(w)
    pool = r["pool"]
    st = oracle.contiguous_strides(w.num_blocks, w.num_kv_heads, w.block_size, w.head_dim)
    nblk = int(np.sum(w.block_tables[0] >= 0))
    ids = w.block_tables[0, :nblk].astype(np.int32)
    buf, bad = oracle.block_swap_out(pool, st, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, ids)
    assert bad == 0
    # each token's K and V sit where the documented block layout [K|V][head][slot][dim] puts them
    kl, vl = W.logical_kv(w, 0)
    b5 = buf.reshape(nblk, 2, w.num_kv_heads, w.block_size, w.head_dim)
    for t in range(len(kl)):
        assert np.array_equal(b5[t // w.block_size, 0, :, t % w.block_size], kl[t])
        assert np.array_equal(b5[t // w.block_size, 1, :, t % w.block_size], vl[t])
    ref = _decode(w, pool, w.block_tables, w.decode_lens)
    # preemption frees the blocks (poison them), resumption swaps in elsewhere and remaps the table
    pool5 = pool.reshape(w.num_blocks, -1)
    pool5[ids] = 0x7E00
    new_ids = _free_blocks(w, nblk)
    assert oracle.block_swap_in(pool, st, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, new_ids, buf) == 0
    tables = w.block_tables.copy()
    tables[0, :nblk] = new_ids
    assert np.array_equal(_decode(w, pool, tables, w.decode_lens), ref)
