"""Prefix cache: the oracle pinned to the notes' boundary conditions, and the library's host code
(chained SHA-256 hashes, hash -> block map, reference counts, LRU retention) checked against the
oracle.  No GPU needed: these calls run on the host.

Pins of the oracle ("vLLM：PagedAttention 与前缀缓存" notes, boundary conditions and lookup/reuse;
2kiu.com "PagedAttention 与前缀缓存", sections 2.2, 3.2, 4.3):
* only full blocks are hashed: a 100-token prefix in 16-token blocks caches 96 tokens (6 blocks);
* a changed token changes its block's hash and every later one, never an earlier one;
* equal block contents at another position, or after another prefix, hash differently (the chain);
* an extra key (model / tokenizer version) separates otherwise equal prompts;
* lookup stops at the first miss (partial hit); released blocks keep their mapping until evicted,
  least recently released first; an empty pool raises "KV cache block pool exhausted".
"""
import os
import random

import numpy as np
import pytest

from oracle.prefix_cache import PrefixCacheModel, chained_hashes


# ------------------------------------------------------------------------------ oracle pins

def test_only_full_blocks_are_hashed():
    assert len(chained_hashes(list(range(100)), 16)) == 6
    assert len(chained_hashes(list(range(96)), 16)) == 6
    assert len(chained_hashes(list(range(15)), 16)) == 0


def test_a_changed_token_changes_its_block_and_every_later_hash():
    rng = np.random.default_rng(1)
    toks = [int(t) for t in rng.integers(0, 32000, 160)]
    base = chained_hashes(toks, 16)
    for pos in (0, 15, 16, 77, 159):
        t2 = list(toks)
        t2[pos] ^= 1
        h2 = chained_hashes(t2, 16)
        blk = pos // 16
        assert h2[:blk] == base[:blk]
        assert all(a != b for a, b in zip(h2[blk:], base[blk:]))


def test_hash_depends_on_the_prefix_not_only_the_block():
    a = list(range(16))
    b = list(range(100, 116))
    assert chained_hashes(a + b, 16)[1] != chained_hashes(b, 16)[0]
    assert chained_hashes(a + a, 16)[0] != chained_hashes(a + a, 16)[1]
    assert chained_hashes(a, 16, init=bytes([7] * 32)) != chained_hashes(a, 16)


def test_extra_key_separates_semantic_contexts():
    toks = list(range(48))
    assert chained_hashes(toks, 16, extra=b"llama-2-7b-fp16-v1") != chained_hashes(toks, 16, extra=b"other")
    assert chained_hashes(toks, 16, extra=b"x") == chained_hashes(toks, 16, extra=b"x")


def test_model_partial_hit_reuse_and_lru_eviction():
    pc = PrefixCacheModel(6)
    sys_prompt = list(range(32))
    a = chained_hashes(sys_prompt + list(range(500, 516)), 16)     # 3 full blocks
    blocks_a = pc.allocate(3)
    pc.insert(a, blocks_a)
    pc.release(blocks_a)                                             # mapping kept, blocks cached-free
    assert pc.stats() == dict(free=3, cached_free=3, in_use=0, hashed=3)
    b = chained_hashes(sys_prompt + list(range(900, 916)), 16)      # same first 2 blocks
    hit = pc.match(b)
    assert hit == blocks_a[:2]                                       # partial hit, stops at block 2
    assert pc.ref[blocks_a[0]] == 1 and pc.stats()["cached_free"] == 1
    pc.release(hit)
    # the pool fills up: free blocks first, then the least recently released cached block
    got = pc.allocate(4)
    assert set(got[:3]) == {3, 4, 5} and got[3] == blocks_a[2]     # a's 3rd block was released first
    assert pc.match(a) == blocks_a[:2]                               # its mapping is gone, the others stay
    with pytest.raises(MemoryError, match="KV cache block pool exhausted"):
        pc.allocate(1)


def test_model_rejects_releasing_more_than_held():
    pc = PrefixCacheModel(4)
    b = pc.allocate(1)
    with pytest.raises(ValueError):
        pc.release([b[0], b[0]])
    pc.release(b)


# ------------------------------------------------------------------------------ library vs oracle

@pytest.fixture(scope="module")
def P():
    from paged_kv_cache_134_gb300 import build
    try:
        build.nvcc()
    except RuntimeError:
        pytest.skip("nvcc not available")
    build.build()
    import paged_kv_cache_134_gb300 as pkg
    return pkg


@pytest.mark.parametrize("bs,n,extra,init", [(16, 100, b"", None), (8, 64, b"llama-2-7b-fp16-v1", None),
                                             (32, 1000, b"salt", bytes(range(32))), (16, 15, b"", None)])
def test_library_block_hashes_match_oracle(P, bs, n, extra, init):
    rng = np.random.default_rng(n)
    toks = rng.integers(0, 2 ** 31 - 1, n).astype(np.int32)
    got = P.block_hashes(toks, bs, extra=extra, init=init)
    ref = chained_hashes([int(t) for t in toks], bs, extra=extra, init=init)
    assert [bytes(r) for r in got] == ref


def test_library_prefix_cache_matches_oracle_on_random_traffic(P):
    rng = random.Random(5)
    nb, bs = 48, 4
    lib, ref = P.PrefixCache(nb), PrefixCacheModel(nb)
    prompts = [[rng.randrange(50) for _ in range(rng.randrange(4, 40))] for _ in range(12)]
    live = []
    for step in range(400):
        op = rng.random()
        if op < 0.5:
            toks = list(rng.choice(prompts))
            if rng.random() < 0.3:
                toks += [rng.randrange(50) for _ in range(rng.randrange(1, 9))]
            hs = chained_hashes(toks, bs)
            assert [bytes(h) for h in P.block_hashes(np.array(toks, np.int32), bs)] == hs
            hit_l = [int(b) for b in lib.match(np.frombuffer(b"".join(hs), np.uint8))] if hs else []
            hit_r = ref.match(hs)
            assert hit_l == hit_r, step
            need = -(-len(toks) // bs) - len(hit_r)
            try:
                new_r = ref.allocate(need)
            except MemoryError:
                with pytest.raises(Exception, match="exhausted"):
                    lib.allocate(need)
                if hit_r:
                    lib.release(np.array(hit_r, np.int32))
                    ref.release(hit_r)
                continue
            new_l = [int(b) for b in lib.allocate(need)]
            assert new_l == new_r, step
            blocks = hit_r + new_r
            full = len(hs)
            if full > len(hit_r):
                pub = slice(len(hit_r), full)
                lib.insert(np.frombuffer(b"".join(hs[pub]), np.uint8), np.array(blocks[pub], np.int32))
                ref.insert(hs[pub], blocks[pub])
            live.append(blocks)
        elif live:
            blocks = live.pop(rng.randrange(len(live)))
            lib.release(np.array(blocks, np.int32))
            ref.release(blocks)
        assert lib.stats() == ref.stats(), step
    lib.close()


def test_library_rejects_bad_release_and_exhaustion(P):
    pc = P.PrefixCache(2)
    b = pc.allocate(2)
    with pytest.raises(P.PagedKVError, match="exhausted"):
        pc.allocate(1)
    with pytest.raises(P.PagedKVError):
        pc.release(np.array([b[0], b[0]], np.int32))
    assert pc.stats() == dict(free=0, cached_free=0, in_use=2, hashed=0)
    pc.release(b)
    assert pc.stats()["free"] == 2
    pc.close()
