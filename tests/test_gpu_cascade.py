"""GPU parity of the cascade decode (shared prefix read once for the batch) against the oracle's paged
decode, which computes the same attention sequence by sequence (2kiu.com "PagedAttention 与前缀缓存",
sections 2.3 and 3.3).  Outputs within |gpu - ref| <= 2e-3 + 1e-2 |ref|; the appended token's bytes
and the whole pool bit-exact; a sequence shorter than the claimed prefix is reported, not faulted.
"""
import numpy as np
import pytest
import torch

from oracle import steps
import paged_kv_cache_134_gb300 as P
from paged_kv_cache_134_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from gpu_path import OUT_DT, DecodeInputs, assert_close, decode_step, fill_cache, new_cache, run_decode  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def check_cascade(w, tag):
    g = run_decode(w, cascade_prefix=w.shared_prefix_len)
    r = steps.decode_step(w, strides=g["strides"], pool_elems=g["pool"].size)
    assert g["err"] == 0, f"device error bits {g['err']}"
    assert np.array_equal(g["new_slots"], r["new_slots"]) and np.array_equal(g["pool"], r["pool"])
    atol = 5e-2 if w.kv_dtype == "fp8" else ATOL   # FP8: the oracle reads the same stored codes
    mx, rel = assert_close(g["out"], r["out"], atol, RTOL, tag, out_dtype=OUT_DT(w))
    print(f"{tag}: max abs {mx:.2e} max rel {rel:.2e}")
    return g


CASES = [
    # prefix not a multiple of the 64-key tile; grouped-query heads; bf16
    dict(num_seqs=5, prefix_tokens=96, max_suffix=40, heads=8, kv_heads=2, d=64, bs=16, dtype="bf16"),
    # more than 128 sequences (two query-row tiles), four 256-key prefix splits
    dict(num_seqs=130, prefix_tokens=1024, max_suffix=300, heads=2, d=128, bs=32),
    # five prefix splits (the last one partial), G = 4 (tensor-core suffix decode), bs 8
    dict(num_seqs=9, prefix_tokens=1120, max_suffix=700, heads=8, kv_heads=2, d=128, bs=8, dtype="bf16"),
    # suffixes shorter than a block and longer than a split
    dict(num_seqs=16, prefix_tokens=256, max_suffix=2000, heads=4, d=128, bs=16),
    # more sequences than one launch takes (1024): two runs of launches, each reading the prefix once
    dict(num_seqs=1100, prefix_tokens=256, max_suffix=60, heads=2, d=128, bs=16),
    # the same with G = 4 (tensor-core suffix decode, whose launches take fewer sequences)
    dict(num_seqs=1100, prefix_tokens=192, max_suffix=60, heads=8, kv_heads=2, d=128, bs=16, dtype="bf16"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"S{c['num_seqs']}_P{c['prefix_tokens']}_bs{c['bs']}")
def test_cascade_small_cases(case):
    check_cascade(W.prefix13b(seed=91, **case), "cascade")


# FP8 cache: prefix codes widened exactly in shared memory, scales folded into the softmax and the
# partials; the 13B-shape batch, grouped heads with a bf16 model and bs 8, D = 64
FP8_CASES = [
    dict(num_seqs=64, prefix_tokens=4096, max_suffix=512, heads=40, d=128, bs=32),
    dict(num_seqs=9, prefix_tokens=1120, max_suffix=700, heads=8, kv_heads=2, d=128, bs=8, dtype="bf16"),
    dict(num_seqs=5, prefix_tokens=96, max_suffix=40, heads=8, kv_heads=2, d=64, bs=16),
]


@pytest.mark.parametrize("case", FP8_CASES, ids=lambda c: f"S{c['num_seqs']}_P{c['prefix_tokens']}_bs{c['bs']}")
def test_cascade_fp8_cache(case):
    check_cascade(W.prefix13b(seed=95, kv_dtype="fp8", **case), "cascade fp8")


def test_cascade_prefix13b_config():
    w = W.prefix13b()
    g = check_cascade(w, "prefix13b")
    plain = run_decode(w)
    assert plain["err"] == 0
    assert np.allclose(g["out"], plain["out"], rtol=1e-2, atol=2e-3)


def test_cascade_rejects_a_sequence_shorter_than_the_prefix():
    w = W.prefix13b(seed=92, num_seqs=4, prefix_tokens=128, max_suffix=20, heads=2, d=128, bs=16)
    g = run_decode(w, keep_cache=True)
    cache, x = g["cache"], g["inputs"]
    short = x.lens.clone()
    short[2] = 100   # below the 128 shared tokens
    P.paged_decode_attention_cascade(x.q, cache, x.tables, short, 128, float(w.scale))
    err = cache.check_error()
    cache.close()
    assert err & 4   # PKV_DEVERR_LENGTH


@pytest.mark.parametrize("kv_heads", [40, 10], ids=["mha", "gqa4"])
def test_back_to_back_cascade_steps_agree(kv_heads):
    # The prefix phase and the suffix decode overlap inside each call, and consecutive calls follow
    # each other on one stream with no host synchronisation in between; 24 such steps must all give
    # the first step's output bit for bit, and that output must match the oracle.
    w = W.prefix13b(seed=93, num_seqs=64, prefix_tokens=2048, max_suffix=400, heads=40, kv_heads=kv_heads,
                    d=128, bs=32)
    cache = new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype, w.model_dtype)
    try:
        fill_cache(cache, w)
        x = DecodeInputs(w)
        outs = []
        for _ in range(24):
            decode_step(cache, x, cascade_prefix=w.shared_prefix_len)
            outs.append(x.out.clone())
        torch.cuda.synchronize()
        assert cache.check_error() == 0
        first = outs[0]
        for i, o in enumerate(outs[1:], 1):
            assert torch.equal(o, first), f"step {i} differs from step 0"
        r = steps.decode_step(w, strides=cache.view()[1], pool_elems=int(cache.pool_elems().numel()))
        assert_close(first.float().cpu().double().numpy(), r["out"], ATOL, RTOL, "back-to-back cascade",
                     out_dtype=OUT_DT(w))
    finally:
        cache.close()
