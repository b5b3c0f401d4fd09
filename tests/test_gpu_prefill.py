"""GPU parity of the tcgen05 packed causal prefill (and its fused paged K/V write) against the oracle.

Outputs: |gpu - ref| <= 2e-3 + 1e-2 |ref| per element.  Cache contents: bit-exact, every byte of
the pool (untouched slots keep their NaN fill).
"""
import numpy as np
import pytest
import torch

from oracle import steps
from paged_kv_cache_134_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from gpu_path import OUT_DT, assert_close, run_prefill  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def check_prefill(w, tag):
    g = run_prefill(w)
    r = steps.prefill_step(w, strides=g["strides"], pool_elems=g["pool"].size)
    assert g["err"] == 0, f"device error bits {g['err']}"
    assert np.array_equal(g["pool"], r["pool"]), f"pool differs at {int(np.sum(g['pool'] != r['pool']))} elements"
    mx, rel = assert_close(g["out"], r["out"], ATOL, RTOL, tag, out_dtype=OUT_DT(w))
    print(f"{tag}: max abs {mx:.2e} max rel {rel:.2e}")
    return g


SMALL = [
    dict(lengths=(1,), heads=1, kv_heads=1, d=128),
    dict(lengths=(5, 64, 65, 127, 128, 129), heads=2, kv_heads=2, d=128),
    dict(lengths=(200, 3, 300), heads=4, kv_heads=1, d=128),
    dict(lengths=(33, 257, 64, 1), heads=4, kv_heads=2, d=64),
    dict(lengths=(130, 17, 500), heads=2, kv_heads=2, d=128, dtype="bf16"),
    dict(lengths=(70, 190), heads=8, kv_heads=1, d=64, dtype="bf16", bs=8),
    dict(lengths=(96, 40, 300), heads=2, kv_heads=2, d=128, bs=32),
]


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "_".join(f"{k}{v}" for k, v in c.items()).replace(" ", ""))
def test_small_cases(case):
    check_prefill(W.prefill(seed=51, **case), "small")


# lengths around 128- and 256-row boundaries, odd tile counts, up to 32 blocks of bs 8 per 256 rows
BOUNDARY_CASES = [
    dict(lengths=(256, 257, 383, 384, 385), heads=2, kv_heads=2, d=128, bs=8),
    dict(lengths=(640, 1000, 1), heads=4, kv_heads=1, d=64, bs=16),
    dict(lengths=(129, 255, 511), heads=8, kv_heads=2, d=128, bs=32),
]


@pytest.mark.parametrize("case", BOUNDARY_CASES, ids=lambda c: "_".join(f"{k}{v}" for k, v in c.items()).replace(" ", ""))
def test_tile_boundary_cases(case):
    check_prefill(W.prefill(seed=53, **case), "boundaries")


def test_packed_config_5256_tokens():
    w = W.prefill()
    assert w.total_tokens == 5256
    check_prefill(w, "prefill5256")


def test_first_row_is_v0_exactly():
    w = W.prefill(lengths=(40, 1, 129, 300), heads=4, kv_heads=2, d=128, seed=52)
    g = run_prefill(w)
    v = W.bits_to_float(w.v, "f16")
    for i in range(4):
        a = w.cu_seqlens[i]
        for h in range(4):
            assert np.array_equal(g["out"][a, h], v[a, h // 2])


def test_sequences_do_not_see_each_other_bitwise():
    w = W.prefill(lengths=(150, 77, 260), heads=2, d=128, seed=53)
    base = run_prefill(w)["out"]
    cu = w.cu_seqlens
    w.k[cu[1]:cu[2]] ^= 0x0400
    w.v[cu[1]:cu[2]] ^= 0x0400
    out = run_prefill(w)["out"]
    for i in (0, 2):
        assert np.array_equal(out[cu[i]:cu[i + 1]], base[cu[i]:cu[i + 1]])
    assert not np.array_equal(out[cu[1]:cu[2]], base[cu[1]:cu[2]])


def test_deterministic():
    w = W.prefill(lengths=(1000, 24), heads=4, d=128, seed=54)
    assert np.array_equal(run_prefill(w)["out"], run_prefill(w)["out"])


def test_bad_cu_seqlens_reported_not_fatal():
    w = W.prefill(lengths=(40, 50), heads=2, d=64, seed=55)
    import paged_kv_cache_134_gb300 as P
    from gpu_path import TORCH_DT, dev, new_cache
    cache = new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, "f16", "f16")
    md = TORCH_DT["f16"]
    cu = w.cu_seqlens.copy()
    out = P.packed_prefill_attention(dev(w.q, md), dev(w.k, md), dev(w.v, md), dev(cu), 45, dev(w.block_tables),
                                     cache, float(w.scale))
    assert cache.check_error() & 8   # the 50-token sequence exceeds max_seqlen 45
    assert np.all(np.isfinite(out[:40].float().cpu().numpy()))
    cache.close()


# FP8 cache (E4M3 with per-head scales): the attention reads the packed k, v as given (the 16-bit
# tolerance applies), and the cache holds what the append writes (bit-exact against the oracle's
# append): config 3's lengths, a bf16 model with grouped heads and bs 8, and D = 64 with bs 32
FP8_CASES = [
    dict(lengths=(128, 200, 512, 1024, 2048, 256, 64, 1024), heads=8, kv_heads=8, d=128, bs=16),
    dict(lengths=(130, 17, 500), heads=4, kv_heads=2, d=128, dtype="bf16", bs=8),
    dict(lengths=(33, 257, 64, 1), heads=4, kv_heads=2, d=64, bs=32),
]


@pytest.mark.parametrize("case", FP8_CASES, ids=lambda c: "_".join(f"{k}{v}" for k, v in c.items()).replace(" ", ""))
def test_fp8_cache_packed_prefill(case):
    check_prefill(W.prefill(seed=57, kv_dtype="fp8", **case), "fp8 cache packed")
