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

from gpu_path import assert_close, run_decode  # noqa: E402

ATOL, RTOL = 2e-3, 1e-2


def check_cascade(w, tag):
    g = run_decode(w, cascade_prefix=w.shared_prefix_len)
    r = steps.decode_step(w, strides=g["strides"], pool_elems=g["pool"].size)
    assert g["err"] == 0, f"device error bits {g['err']}"
    assert np.array_equal(g["new_slots"], r["new_slots"]) and np.array_equal(g["pool"], r["pool"])
    mx, rel = assert_close(g["out"], r["out"], ATOL, RTOL, tag)
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
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"S{c['num_seqs']}_P{c['prefix_tokens']}_bs{c['bs']}")
def test_cascade_small_cases(case):
    check_cascade(W.prefix13b(seed=91, **case), "cascade")


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
