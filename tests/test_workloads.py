"""Host-side logic of the synthetic workloads: free list, ref counts, tables, config shapes."""
import json
import math
import os

import numpy as np
import pytest

from paged_kv_cache_134_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_allocator_front_pop_tail_free_and_exhaustion():
    a = W.BlockAllocator(8, np.random.default_rng(0))
    order = list(a.free_list)
    got = a.allocate(3)
    assert got == order[:3] and a.num_free == 5
    assert all(a.ref_count[b] == 1 for b in got)
    a.free([got[1]])
    assert a.free_list[-1] == got[1] and a.ref_count[got[1]] == 0
    with pytest.raises(W.PoolExhausted, match="KV cache block pool exhausted"):
        a.allocate(7)
    with pytest.raises(ValueError):
        a.free([got[1]])


def test_allocator_shared_block_freed_only_at_zero():
    a = W.BlockAllocator(4, np.random.default_rng(1))
    b = a.allocate(1)
    a.share(b)
    a.share(b)
    a.free(b)
    assert b[0] not in a.free_list and a.ref_count[b[0]] == 2
    a.free(b)
    a.free(b)
    assert a.free_list[-1] == b[0]


def test_kv_bytes_golden():
    g = json.load(open(os.path.join(GOLD, "kv_bytes.json")))
    for c in g["cases"]:
        assert W.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], c["elem_bytes"]) == c["bytes_per_token"]
    per_tok = W.kv_bytes_per_token(32, 32, 128, 2)
    assert 4096 * per_tok == g["tokens_4096_7b_bytes"]
    assert 16 * per_tok == g["block_16_all_layers_7b_bytes"]
    # 60 GB pool / 8 MB blocks = 7680 blocks (2kiu.com section 5.2); 20 GB -> 2560 (discosf.com section 4.1)
    assert W.pool_capacity_blocks(60 * 2**30, 16, per_tok) == 7680
    assert W.pool_capacity_blocks(20 * 2**30, 16, per_tok) == 2560


def _check_tables(w):
    used = w.block_tables[w.block_tables >= 0]
    assert used.max() < w.num_blocks
    for s in range(w.num_seqs):
        nb = W.blocks_for(int(w.context_lens[s]) + 1, w.block_size)
        row = w.block_tables[s]
        assert np.all(row[:nb] >= 0) and np.all(row[nb:] == -1)


def test_tiny_config():
    w = W.tiny()
    assert w.context_lens.tolist() == [1, 15, 16, 37]
    assert (w.num_blocks, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size) == (64, 8, 8, 64, 16)
    assert w.scale == np.float32(0.125)
    _check_tables(w)
    # length 16 fills its first block, so the appended token opens a second one
    assert W.blocks_for(17, 16) == 2 and w.block_tables[2, 1] >= 0
    assert len(set(w.block_tables[w.block_tables >= 0].tolist())) == int((w.block_tables >= 0).sum())
    assert w.fill_k.shape == (1 + 15 + 16 + 37, 8, 64)


def test_decode7b_shape_logic_small():
    w = W.decode7b(num_seqs=3, max_len=40)
    need = sum(W.blocks_for(int(L) + 1, 16) for L in w.context_lens)
    assert w.num_blocks == math.ceil(1.1 * need)
    assert (w.num_q_heads, w.num_kv_heads, w.head_dim) == (32, 32, 128)
    _check_tables(w)
    assert w.kv_read_bytes() == int((w.context_lens + 1).sum()) * 32 * 128 * 2 * 2


def test_decode7b_full_lengths():
    # lengths only (values of the full workload are 1 GB; generated on the GPU machine)
    rng = np.random.default_rng(1002 ^ 0x5EED)
    lens = rng.integers(1, 4097, size=32, dtype=np.int64)
    assert lens.min() >= 1 and lens.max() <= 4096


def test_prefill_config():
    w = W.prefill(heads=1, d=64)   # full lengths, small head count
    assert w.total_tokens == 5256 and w.max_seqlen == 2048
    assert w.num_blocks == math.ceil(1.1 * 329) == 362
    assert w.block_tables.shape == (8, 128)
    assert (w.block_tables[1] >= 0).sum() == 13
    assert w.causal_pairs() == sum(n * (n + 1) // 2 for n in W.PACKED_LENGTHS) == 3342436


def test_prefix13b_refcount_and_sharing():
    w = W.prefix13b(heads=1, d=64)
    assert w.num_seqs == 64 and w.block_size == 32
    prefix = w.block_tables[:, :128]
    assert np.all(prefix == prefix[0:1])
    assert np.all(w.ref_count[prefix[0]] == 64)
    own = w.block_tables[:, 128:]
    own = own[own >= 0]
    assert len(set(own.tolist())) == len(own) and not set(own.tolist()) & set(prefix[0].tolist())
    assert np.all((w.context_lens >= 4097) & (w.context_lens <= 4096 + 512))


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_stress_churned_free_list(bs):
    w = W.stress(bs=bs, num_seqs=40)
    _check_tables(w)
    assert w.num_kv_heads == 8 and w.num_q_heads == 32
    assert w.context_lens.max() <= 8192 and w.context_lens.min() >= 1
    used = w.block_tables[w.block_tables >= 0]
    assert len(set(used.tolist())) == len(used)
    # churn leaves the ids far from the untouched permutation order: not one long run of the initial list
    fresh = W.BlockAllocator(w.num_blocks, np.random.default_rng(0)).free_list
    assert used.tolist() != fresh[:len(used)]


def test_stress_lengths_lognormal():
    lens = W._lognormal_lens(np.random.default_rng(5), 20000)
    assert 450 < np.median(lens) < 550 and lens.max() <= 8192


def test_fp8_scales_cover_amax():
    w = W.stress(bs=16, kv_dtype="fp8", num_seqs=6)
    k = np.abs(W.bits_to_float(np.concatenate([w.fill_k, w.new_k]), "bf16")).max(axis=(0, 2))
    assert np.all(k / w.k_scale <= 448.0 * (1 + 1e-6))
