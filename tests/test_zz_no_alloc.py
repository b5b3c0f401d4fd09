"""paged_decode_attention_noalloc: the decode for callers that must not allocate device memory.

Such callers (a serving engine whose own allocator owns nearly all of the GPU's memory, or code
that cannot afford the device-wide synchronisation of cudaMalloc/cudaFree) get the same decode
with the split-K partials kept in a fixed scratch array inside the library, made resident when the
cache is created.  Through the C ABI this file checks that:
  * after one warm-up call (the first launch of a kernel may load its code), a no-alloc call on a
    fresh cache leaves the device's free memory exactly as it was;
  * two calls in a row (different batches, so the second runs on the first one's leftover scratch
    contents) give bit for bit the output of paged_decode_attention, which runs the same kernels
    with the same split plan, and both match the oracle within the decode tolerance;
  * a call too large for the scratch is refused.
It is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

from oracle import steps
from paged_kv_cache_134_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import paged_kv_cache_134_gb300 as P  # noqa: E402
from gpu_path import DecodeInputs, assert_close, fill_cache, new_cache  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def _prepared(w):
    cache = new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype, w.model_dtype,
                      w.k_scale, w.v_scale)
    fill_cache(cache, w)
    x = DecodeInputs(w)
    P.paged_kv_append_at(cache, x.new_k, x.new_v, x.tables, x.seq_ids, x.positions, x.slots)
    return cache, x


def test_noalloc_allocates_nothing_and_matches_the_decode_bitwise_on_two_calls_in_a_row():
    batches = [W.decode7b(),  # 32 sequences up to 4097 tokens: most rows have several splits
               W.small_decode("second", [3000, 17, 0, 900, 2500, 64], hq=8, hkv=2, d=128, bs=16, seed=61)]
    for i, w in enumerate(batches):
        cache, x = _prepared(w)
        got = torch.full_like(x.q, float("nan"))
        warm = torch.empty_like(x.q)
        # warm-up: the first launch of a kernel may load its code onto the device
        P.paged_decode_attention_noalloc(x.q, cache, x.tables, x.lens, x.scale, warm)
        torch.cuda.synchronize()
        free0, _ = torch.cuda.mem_get_info()
        P.paged_decode_attention_noalloc(x.q, cache, x.tables, x.lens, x.scale, got)
        torch.cuda.synchronize()
        free1, _ = torch.cuda.mem_get_info()
        assert free1 == free0, f"batch {i}: device free memory moved by {free0 - free1} bytes"
        assert cache.check_error() == 0
        assert torch.equal(got, warm), f"batch {i}: two no-alloc calls differ"
        # only now the allocating decode (it may grow the cache's workspace): same kernels, same splits
        ref = P.paged_decode_attention(x.q, cache, x.tables, x.lens, x.scale)
        torch.cuda.synchronize()
        assert cache.check_error() == 0
        assert torch.equal(got, ref), f"batch {i}: no-alloc output differs from paged_decode_attention"
        r = steps.decode_step(w, strides=cache.view()[1], pool_elems=int(cache.pool_elems().numel()))
        assert_close(got.float().cpu().numpy(), r["out"], ATOL, RTOL, f"no-alloc {w.name}", out_dtype=w.model_dtype)
        cache.close()


def test_noalloc_refuses_a_batch_beyond_its_scratch():
    w = W.small_decode("big", [10, 20], hq=32, hkv=32, d=128, bs=16, seed=62)
    cache, x = _prepared(w)
    # 1024 sequences x 32 heads with 16384-token tables would need far more than the fixed scratch
    q = torch.zeros(1024, 32, 128, dtype=torch.float16, device="cuda")
    tables = torch.zeros(1024, 1024, dtype=torch.int32, device="cuda")
    lens = torch.ones(1024, dtype=torch.int32, device="cuda")
    with pytest.raises(P.PagedKVError, match="scratch"):
        P.paged_decode_attention_noalloc(q, cache, tables, lens, 0.1, torch.empty_like(q))
    cache.close()
