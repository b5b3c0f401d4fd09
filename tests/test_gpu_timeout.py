"""The kernels' bounded waits give up, report and leave the cache usable.

Every mbarrier wait in the library is bounded: after a time limit it stops, or-s PKV_DEVERR_TIMEOUT
into the cache's error word and lets the kernel wind down, so that a failure degrades instead of
hanging the GPU ("Paged KV Cache 与 Packed Sequence", discosf.com, section 5.1; "PagedAttention 与前缀
缓存", 2kiu.com, section 6.1).  kv_cache_selftest_wait_timeout runs the same wait routines (spinning
and suspend-hint forms) on an mbarrier nothing ever arrives on, with a short limit; nothing else is
touched and nothing traps.  The test checks the reported bit, that the error word is cleared by the
read, and that a decode on the same cache right after it matches the oracle.
"""
import time

import numpy as np
import pytest
import torch

from oracle import steps
from paged_kv_cache_134_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

import paged_kv_cache_134_gb300 as P  # noqa: E402
from gpu_path import DecodeInputs, assert_close, decode_step, fill_cache, new_cache  # noqa: E402

TIMEOUT_BIT = 16


@pytest.mark.parametrize("limit_ns", [1_000_000, 20_000_000])
def test_bounded_wait_gives_up_reports_and_the_cache_stays_usable(limit_ns):
    w = W.small_decode("after_timeout", [700, 33, 0, 1500], hq=8, hkv=8, d=128, bs=16, seed=81)
    cache = new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype, w.model_dtype)
    try:
        fill_cache(cache, w)
        torch.cuda.synchronize()
        assert cache.check_error() == 0
        t0 = time.perf_counter()
        cache.selftest_wait_timeout(limit_ns)
        code = cache.check_error()
        waited = time.perf_counter() - t0
        assert code == TIMEOUT_BIT, f"device error bits {code}"
        assert waited >= limit_ns * 1e-9, "the wait gave up before its limit"
        assert waited < limit_ns * 1e-9 + 2.0, "the wait ran far past its limit"
        assert cache.check_error() == 0, "reading the error word clears it"
        x = DecodeInputs(w)
        out = decode_step(cache, x)
        torch.cuda.synchronize()
        assert cache.check_error() == 0
        r = steps.decode_step(w, strides=cache.view()[1], pool_elems=int(cache.pool_elems().numel()))
        assert_close(out.float().cpu().double().numpy(), r["out"], 2e-3, 1e-2, "decode after a timeout",
                     out_dtype=w.model_dtype)
    finally:
        cache.close()


def test_selftest_rejects_a_limit_outside_its_range():
    cache = P.KVCache(4, 16, 1, 64, "f16")
    try:
        for bad in (0, 2_000_000_000):
            with pytest.raises(P.PagedKVError, match="limit_ns"):
                cache.selftest_wait_timeout(bad)
    finally:
        cache.close()
