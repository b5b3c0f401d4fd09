"""GPU parity of the tensor-core decode for grouped-query heads (head_dim 128, G = 2, 4 or 8 query
heads per KV head), including the FP8 E4M3 cache, whose codes are widened to fp16 in shared memory
and whose per-head scales fold into the score scale and the output ("PagedAttention 与前缀缓存",
2kiu.com, section 2.3 for the attention; the FP8 cache layout as the oracle's append stores it).

Outputs are compared element by element with the oracle: |gpu - ref| <= atol + rtol |ref|,
atol = 2e-3 (5e-2 for FP8, whose reference runs on the stored codes), rtol = 1e-2.  The same
workloads through the CUDA-core kernel (PAGEDKV_DECODE_TC=0) must meet the same bound.
"""
import os

import numpy as np
import pytest
import torch

from oracle import steps
from paged_kv_cache_134_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA device", allow_module_level=True)

from gpu_path import OUT_DT, assert_close, run_decode  # noqa: E402

ATOL = {"f16": 2e-3, "bf16": 2e-3, "fp8": 5e-2}
RTOL = 1e-2

# token counts around the 128-token MMA step and the split (512 tokens for 16-bit caches, 1024 for
# E4M3 ones)
LENS = [0, 1, 127, 128, 129, 511, 512, 513, 1023, 1025, 2000, 37]


def check(w, tag):
    g = run_decode(w)
    r = steps.decode_step(w, strides=g["strides"], pool_elems=g["pool"].size)
    assert g["err"] == 0, f"{tag}: device error bits {g['err']}"
    assert np.array_equal(g["pool"], r["pool"]), f"{tag}: pool bytes differ"
    mx, rel = assert_close(g["out"], r["out"], ATOL[w.kv_dtype], RTOL, tag, out_dtype=w.model_dtype)
    print(f"{tag}: max abs {mx:.2e} max rel {rel:.2e}")
    return g


FP8_CASES = [
    dict(G=2, model="f16", bs=16),
    dict(G=4, model="bf16", bs=8),
    dict(G=8, model="bf16", bs=32),
    dict(G=8, model="f16", bs=8),
    dict(G=4, model="f16", bs=32),
]


@pytest.mark.parametrize("c", FP8_CASES, ids=lambda c: f"G{c['G']}_{c['model']}_bs{c['bs']}")
def test_fp8_grouped_heads(c):
    hkv = 2
    w = W.small_decode("fp8tc", LENS, hq=hkv * c["G"], hkv=hkv, d=128, bs=c["bs"], kv_dtype="fp8",
                       model_dtype=c["model"], seed=500 + c["G"] + c["bs"])
    check(w, f"fp8 G{c['G']} {c['model']} bs{c['bs']}")


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
def test_tensor_core_and_cuda_core_paths_agree(kv, monkeypatch):
    w = W.small_decode("agree", [3000, 64, 700, 1], hq=16, hkv=4, d=128, bs=16, kv_dtype=kv, seed=510)
    tc = check(w, f"{kv} tensor cores")
    monkeypatch.setenv("PAGEDKV_DECODE_TC", "0")
    cc = check(w, f"{kv} CUDA cores")
    assert os.environ["PAGEDKV_DECODE_TC"] == "0"
    assert_close(tc["out"], cc["out"], ATOL[kv], RTOL, "paths", out_dtype=OUT_DT(w))


@pytest.mark.parametrize("kv", ["fp8", "bf16"])
def test_invalid_block_id_on_the_tensor_core_path(kv):
    lens = [300, 300, 130]
    w = W.small_decode("badtc", lens, hq=8, hkv=2, d=128, bs=16, kv_dtype=kv, seed=520)
    w.block_tables = w.block_tables.copy()
    w.block_tables[1, 3] = w.num_blocks + 7   # sequence 1 only; its new token lands in a later block
    g = run_decode(w)
    assert g["err"] & 1, "block-id error bit not set"
    r = steps.decode_step(W.small_decode("badtc", lens, hq=8, hkv=2, d=128, bs=16, kv_dtype=kv, seed=520),
                          strides=g["strides"], pool_elems=g["pool"].size)
    for s in (0, 2):
        assert_close(g["out"][s], r["out"][s], ATOL[kv], RTOL, f"unaffected sequence {s}", out_dtype=OUT_DT(w))
