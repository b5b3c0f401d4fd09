"""GPU parity of the prefill over a cached prefix and of the whole-block copy / swap kernels.

Prefill over a cached prefix (2kiu.com "PagedAttention 与前缀缓存", section 4.3 steps 2-4): outputs
within |gpu - ref| <= 2e-3 + 1e-2 |ref| of the oracle; the pool (cached tokens, the appended tail,
every untouched NaN slot) bit-exact.  Block copy and swap (sections 2.2, 4.3, 5.2): bit-exact
against the oracle, with device and page-locked host swap buffers, and bad block ids reported
without a fault.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import steps
import paged_kv_cache_134_gb300 as P
from paged_kv_cache_134_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from gpu_path import OUT_DT, assert_close, dev, run_decode  # noqa: E402
from paged_kv_cache_134_gb300.runner import run_context_prefill, run_prefill  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


# ------------------------------------------------------------------------------ prefill over a cached prefix

def check_context_prefill(w, tag, atol=ATOL):
    g = run_context_prefill(w)
    r = steps.context_prefill_step(w, strides=g["strides"], pool_elems=g["pool"].size)
    assert g["err"] == 0, f"device error bits {g['err']}"
    assert np.array_equal(g["pool"], r["pool"]), f"pool differs at {int(np.sum(g['pool'] != r['pool']))} elements"
    mx, rel = assert_close(g["out"], r["out"], atol, RTOL, tag, out_dtype=OUT_DT(w))
    print(f"{tag}: max abs {mx:.2e} max rel {rel:.2e}")
    return g


CTX_CASES = [
    # contexts and tails around block (16) and tile (64 keys, 128 queries) edges
    dict(context_lens=(0, 16, 37, 200), new_lens=(5, 130, 64, 1), heads=4, kv_heads=4, d=128, bs=16),
    dict(context_lens=(63, 64, 65, 127), new_lens=(1, 128, 129, 64), heads=2, kv_heads=2, d=128, bs=16),
    dict(context_lens=(1, 300), new_lens=(255, 17), heads=8, kv_heads=2, d=128, bs=16),
    dict(context_lens=(7, 64, 1), new_lens=(3, 70, 129), heads=4, kv_heads=1, d=64, bs=8),
    dict(context_lens=(32, 32, 32), new_lens=(1, 40, 9), shared_prefix=32, heads=2, kv_heads=2, d=128, bs=32),
    dict(context_lens=(48, 50, 100), new_lens=(20, 3, 190), shared_prefix=48, heads=4, kv_heads=2, d=128, bs=16,
         dtype="bf16"),
    dict(context_lens=(500,), new_lens=(300,), heads=2, kv_heads=2, d=64, bs=32, dtype="bf16"),
]


@pytest.mark.parametrize("case", CTX_CASES, ids=lambda c: f"G{c['heads'] // c['kv_heads']}_d{c['d']}_bs{c['bs']}"
                                                         f"_{c.get('dtype', 'f16')}_{c['context_lens'][0]}")
def test_context_prefill_small_cases(case):
    check_context_prefill(W.context_prefill(seed=81, **case), "ctx")


def test_prefix_hit_prefill_config():
    w = W.prefix_hit_prefill()
    check_context_prefill(w, "prefix_hit")


# FP8 cache: the tails are appended as E4M3 codes, and every key and value, cached or new, is read as
# its code times the head's scale; the oracle reads the same stored codes (gate 5e-2 abs)
FP8_CTX_CASES = [
    dict(context_lens=(0, 16, 37, 200), new_lens=(5, 130, 64, 1), heads=4, kv_heads=4, d=128, bs=16),
    dict(context_lens=(1, 300), new_lens=(255, 17), heads=8, kv_heads=2, d=128, bs=8, dtype="bf16"),
    dict(context_lens=(63, 500), new_lens=(1, 200), heads=2, kv_heads=1, d=64, bs=32),
]


@pytest.mark.parametrize("case", FP8_CTX_CASES, ids=lambda c: f"G{c['heads'] // c['kv_heads']}_d{c['d']}_bs{c['bs']}")
def test_fp8_cache_context_prefill(case):
    check_context_prefill(W.context_prefill(seed=47, kv_dtype="fp8", **case), "fp8 ctx", atol=5e-2)


@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_fp8_cache_prefix_hit_prefill_config(dtype):
    check_context_prefill(W.prefix_hit_prefill(kv_dtype="fp8", dtype=dtype), f"fp8 prefix_hit {dtype}", atol=5e-2)


def test_zero_context_matches_the_packed_prefill_kernel():
    w = W.context_prefill(seed=82, context_lens=(0, 0, 0), new_lens=(1, 200, 129), heads=4, kv_heads=2, d=128)
    g = run_context_prefill(w)
    pw = W.PrefillWorkload(name="same", lengths=w.new_lens, cu_seqlens=w.cu_seqlens, num_q_heads=4, num_kv_heads=2,
                           head_dim=128, block_size=16, num_blocks=w.num_blocks, dtype="f16", scale=w.scale, q=w.q,
                           k=w.k, v=w.v, block_tables=w.block_tables)
    gp = run_prefill(pw)
    assert g["err"] == 0 and gp["err"] == 0
    assert np.array_equal(g["pool"], gp["pool"])
    assert np.allclose(g["out"], gp["out"], rtol=0, atol=1e-3)


def test_context_beyond_the_table_is_reported_not_faulted():
    w = W.context_prefill(seed=83, context_lens=(16, 20), new_lens=(10, 10), heads=2, kv_heads=2, d=128, bs=16)
    cache = P.KVCache(w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, "f16")
    q, k, v = dev(w.q, torch.float16), dev(w.k, torch.float16), dev(w.v, torch.float16)
    bad_ctx = torch.tensor([16, 10 ** 6], dtype=torch.int32, device="cuda")
    P.paged_prefill_attention(q, k, v, dev(w.cu_seqlens), bad_ctx, w.max_seqlen, dev(w.block_tables), cache,
                              float(w.scale))
    err = cache.check_error()
    cache.close()
    assert err & 4   # PKV_DEVERR_LENGTH


# ------------------------------------------------------------------------------ block copy and swap

def _setup(kv_dtype="f16", bs=16):
    w = W.small_decode("blk", [37, 20, 64, 5], hq=4, hkv=2, d=128, bs=bs, kv_dtype=kv_dtype, seed=84,
                       pool_factor=3.0)
    g = run_decode(w, keep_cache=True)
    assert g["err"] == 0
    used = set(int(b) for b in w.block_tables.ravel() if b >= 0)
    free = np.array([b for b in range(w.num_blocks) if b not in used], np.int32)
    return w, g, free


@pytest.mark.parametrize("kv_dtype,bs", [("f16", 16), ("bf16", 8), ("fp8", 32)])
def test_block_copy_matches_oracle_and_reports_bad_ids(kv_dtype, bs):
    w, g, free = _setup(kv_dtype, bs)
    cache = g["cache"]
    used = w.block_tables[w.block_tables >= 0]
    n = min(len(used), len(free))
    src = np.concatenate([used[:n], [w.num_blocks + 3]]).astype(np.int32)
    dst = np.concatenate([free[:n], [free[0]]]).astype(np.int32)
    pool = g["pool"].copy()
    bad = oracle.block_copy(pool, g["strides"], w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, src, dst)
    P.paged_block_copy(cache, dev(src), dev(dst))
    err = cache.check_error()
    got = cache.pool_elems().cpu().numpy()
    got = got if kv_dtype == "fp8" else got.view(np.uint16)
    cache.close()
    assert bad == 1 and err & 1
    assert np.array_equal(got, pool)


@pytest.mark.parametrize("where", ["device", "pinned_host"])
def test_swap_out_and_in_match_oracle(where):
    w, g, free = _setup()
    cache = g["cache"]
    ids = w.block_tables[0][w.block_tables[0] >= 0].astype(np.int32)
    buf_ref, bad = oracle.block_swap_out(g["pool"], g["strides"], w.num_blocks, w.block_size, w.num_kv_heads,
                                         w.head_dim, ids)
    assert bad == 0
    nbytes = len(ids) * cache.block_bytes
    buf = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if where == "device" else \
        torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    P.paged_block_swap_out(cache, dev(ids), buf)
    torch.cuda.synchronize()
    assert np.array_equal(buf.cpu().numpy().view(np.uint16), buf_ref)
    # resume into other blocks: the pool equals the oracle's after the same swap-in
    new_ids = free[: len(ids)]
    pool = g["pool"].copy()
    oracle.block_swap_in(pool, g["strides"], w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, new_ids,
                         buf_ref)
    P.paged_block_swap_in(cache, dev(new_ids), buf)
    assert cache.check_error() == 0
    got = cache.pool_elems().cpu().numpy().view(np.uint16)
    assert np.array_equal(got, pool)
    # decode through the remapped table gives the bitwise same output
    x = g["inputs"]
    tables = w.block_tables.copy()
    tables[0, : len(ids)] = new_ids
    out2 = P.paged_decode_attention(x.q, cache, dev(tables), x.lens, float(w.scale))
    torch.cuda.synchronize()
    assert np.array_equal(out2.float().cpu().numpy(), g["out"].astype(np.float32))
    cache.close()


def test_large_swap_with_host_memory_keeps_bad_pairs():
    """A swap of 300 blocks of 256 KB (75 MB) to page-locked host memory and back into other blocks
    of a fresh cache is bit-exact; a bad block id leaves its host bytes as they were and sets the
    error bit (2kiu.com section 5.2: swap-out on preemption, swap-in on resumption)."""
    nb = 640
    cache = P.KVCache(nb, 16, 32, 128, "f16")
    B = cache.block_bytes
    gen = torch.Generator().manual_seed(612)
    raw, _ = cache.view()                             # the pool's bytes
    raw.copy_(torch.randint(0, 256, raw.shape, generator=gen, dtype=torch.uint8))
    torch.cuda.synchronize()
    before = raw.reshape(nb, B).cpu().clone()
    perm = torch.randperm(nb, generator=gen)
    ids = perm[:300].to(torch.int32).clone()
    ids[7] = nb + 5                                   # bad id: pair 7 skipped
    host = torch.full((300 * B,), 0xAB, dtype=torch.uint8).pin_memory()
    P.paged_block_swap_out(cache, ids.cuda(), host)
    torch.cuda.synchronize()
    assert cache.check_error() & 1, "block-id error bit not set"
    got = host.reshape(300, B)
    for i in range(300):
        if i == 7:
            assert bool((got[i] == 0xAB).all()), "a skipped pair's host bytes changed"
        else:
            assert torch.equal(got[i], before[int(ids[i])]), f"block {i}"
    cache.close()
    # swap back into other blocks of a fresh cache: every good pair lands bit-exact
    cache = P.KVCache(nb, 16, 32, 128, "f16")
    new_ids = perm[300:600].to(torch.int32).clone()
    P.paged_block_swap_in(cache, new_ids.cuda(), host)
    torch.cuda.synchronize()
    assert cache.check_error() == 0
    after = cache.view()[0].reshape(nb, B).cpu()
    for i in range(300):
        assert torch.equal(after[int(new_ids[i])], got[i]), f"block {i}"
    cache.close()


def test_copy_on_write_decode_is_bitwise_equal():
    w, g, free = _setup()
    cache, x = g["cache"], g["inputs"]
    nblk = int(np.sum(w.block_tables[2] >= 0))
    src = w.block_tables[2, :nblk].astype(np.int32)
    dst = free[:nblk]
    P.paged_block_copy(cache, dev(src), dev(dst))
    forked = w.block_tables.copy()
    forked[2, :nblk] = dst
    out2 = P.paged_decode_attention(x.q, cache, dev(forked), x.lens, float(w.scale))
    torch.cuda.synchronize()
    assert cache.check_error() == 0
    assert np.array_equal(out2.float().cpu().numpy(), g["out"].astype(np.float32))
    cache.close()
