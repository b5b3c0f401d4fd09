"""GPU parity of slot indexing, paged append and paged decode attention against the oracle.

Slot indexing and append are compared bit for bit (every slot, every byte of the pool);
attention outputs element by element with |gpu - ref| <= atol + rtol * |ref|, atol = 2e-3
(5e-2 for the FP8 cache), rtol = 1e-2.  The FP8 reference is the oracle run on the stored
codes (its own append), so the gate checks the kernel, not the quantisation error.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import steps
from paged_kv_cache_134_gb300 import workloads as W

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU too; every test here needs the device
    pytest.skip("needs a CUDA device", allow_module_level=True)

from gpu_path import OUT_DT, assert_close, run_decode  # noqa: E402

ATOL = {"f16": 2e-3, "bf16": 2e-3, "fp8": 5e-2}
RTOL = 1e-2


def check_decode(w, tag):
    g = run_decode(w)
    n_elems = g["pool"].size
    r = steps.decode_step(w, strides=g["strides"], pool_elems=n_elems)
    assert g["err"] == 0, f"device error bits {g['err']}"
    assert np.array_equal(g["fill_slots"], r["fill_slots"]), "fill slots differ"
    assert np.array_equal(g["new_slots"], r["new_slots"]), "new-token slots differ"
    assert np.array_equal(g["pool"], r["pool"]), f"pool bytes differ at {int(np.sum(g['pool'] != r['pool']))} elements"
    mx, rel = assert_close(g["out"], r["out"], ATOL[w.kv_dtype], RTOL, tag, out_dtype=w.model_dtype)
    print(f"{tag}: max abs {mx:.2e} max rel {rel:.2e}")
    return g, r


def test_tiny_config():
    check_decode(W.tiny(), "tiny")


def test_decode7b_config():
    check_decode(W.decode7b(), "decode7b")


def test_prefix13b_config_and_shared_equals_private():
    shared = W.prefix13b()
    g, _ = check_decode(shared, "prefix13b")
    private = W.prefix13b(private_prefix=True)
    gp = run_decode(private)
    assert gp["err"] == 0
    assert np.array_equal(g["out"], gp["out"]), "shared-prefix output differs from private copies"


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("bs", [8, 16, 32])
def test_stress_config(bs, kv):
    check_decode(W.stress(bs=bs, kv_dtype=kv), f"stress_bs{bs}_{kv}")


EDGE = [
    dict(lens=[0, 1, 15, 16, 17], hq=4, hkv=4, d=128, bs=16, kv_dtype="f16"),
    dict(lens=[0, 1, 7, 8, 9, 100], hq=8, hkv=2, d=64, bs=8, kv_dtype="bf16"),
    dict(lens=[31, 32, 33, 511, 512, 513], hq=8, hkv=1, d=128, bs=32, kv_dtype="f16"),
    dict(lens=[3, 250, 1000], hq=16, hkv=2, d=128, bs=16, kv_dtype="fp8", model_dtype="f16"),
    dict(lens=[5, 77, 300], hq=16, hkv=4, d=64, bs=32, kv_dtype="fp8", model_dtype="bf16"),
    dict(lens=[1000, 2, 4095, 0], hq=2, hkv=1, d=64, bs=16, kv_dtype="bf16"),
]


@pytest.mark.parametrize("case", EDGE, ids=lambda c: f"{c['kv_dtype']}_G{c['hq'] // c['hkv']}_d{c['d']}_bs{c['bs']}")
def test_edge_cases(case):
    case = dict(case)
    check_decode(W.small_decode("edge", case.pop("lens"), seed=41, **case), "edge")


# A block whose K plus V tiles exceed a stage of the CUDA-core kernel goes in parts of consecutive
# tokens (16 at fp16 and D=128 with the default 8 KB stage, 8 with a 4 KB one, the whole block with
# a 64 KB one); parts wholly past a sequence's end are not loaded.  Lengths around the parts' and
# the blocks' ends, one head per KV head and four (grouped heads kept off the tensor cores).
PARTS_LENS = [1, 7, 8, 9, 15, 16, 17, 24, 31, 32, 33, 48, 49, 257, 300, 513]


@pytest.mark.parametrize("stage_bytes", [None, "4096", "65536"])
@pytest.mark.parametrize("hq,kv", [(4, "f16"), (16, "bf16")], ids=["G1_f16", "G4_bf16"])
def test_blocks_in_stage_parts(stage_bytes, hq, kv, monkeypatch):
    if stage_bytes:
        monkeypatch.setenv("PAGEDKV_DECODE_STAGE_BYTES", stage_bytes)
    monkeypatch.setenv("PAGEDKV_DECODE_TC", "0")
    w = W.small_decode("parts", PARTS_LENS, hq=hq, hkv=4, d=128, bs=32, kv_dtype=kv, seed=48)
    check_decode(w, f"parts {stage_bytes} {kv}")


def test_single_token_returns_v0_bit_exact():
    w = W.small_decode("one", [0, 0, 0, 0], hq=8, hkv=2, d=128, bs=16, kv_dtype="bf16", seed=42)
    g = run_decode(w)
    v = W.bits_to_float(w.new_v, "bf16")
    for s in range(4):
        for h in range(8):
            assert np.array_equal(g["out"][s, h], v[s, h // 4])


def test_placement_invariance_is_bitwise():
    a = W.small_decode("p", [100, 513, 2000, 7], hq=8, hkv=8, d=128, bs=16, seed=43)
    b = W.small_decode("p", [100, 513, 2000, 7], hq=8, hkv=8, d=128, bs=16, seed=43, num_blocks=a.num_blocks * 2,
                       placement_seed=99)
    assert not np.array_equal(a.block_tables, b.block_tables)
    assert np.array_equal(run_decode(a)["out"], run_decode(b)["out"])


def test_run_to_run_determinism():
    w = W.small_decode("det", [4000, 3000, 17, 999], hq=8, hkv=2, d=128, bs=16, seed=44)
    assert np.array_equal(run_decode(w)["out"], run_decode(w)["out"])


def test_sampled_profiling_brackets_every_nth_launch():
    # 23 decode steps with every = 5: launches 1, 6, 11, 16, 21 are timed (the others run without events)
    import paged_kv_cache_134_gb300 as P
    from paged_kv_cache_134_gb300 import runner as G
    w = W.small_decode("prof", [300, 40, 1], hq=4, hkv=4, d=128, bs=16, seed=46)
    cache = G.new_cache(w, w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim, w.kv_dtype, w.model_dtype)
    try:
        G.fill_cache(cache, w)
        x = G.DecodeInputs(w)
        cache.profile_start(kinds=("decode", "append"), every=5)
        for _ in range(23):
            G.decode_step(cache, x)
        prof = cache.profile_read()
        assert prof["decode_launches"] == 5 and prof["append_launches"] == 5, prof
        assert prof["merge_launches"] == 0 and prof["decode_ms"] > 0.0
        with pytest.raises(P.PagedKVError):
            cache.profile_start(kinds=("decode",), every=0)
    finally:
        cache.close()


def test_invalid_block_id_is_reported_not_fatal():
    w = W.small_decode("bad", [40, 40], hq=2, hkv=2, d=64, bs=16, seed=45)
    w.block_tables = w.block_tables.copy()
    w.block_tables[1, 1] = w.num_blocks + 5   # out of the pool; the append of seq 1's new token still lands
    g = run_decode(w)
    assert g["err"] & 1, "block-id error bit not set"
    r = steps.decode_step(W.small_decode("bad", [40, 40], hq=2, hkv=2, d=64, bs=16, seed=45),
                          strides=g["strides"], pool_elems=g["pool"].size)
    assert_close(g["out"][0], r["out"][0], 2e-3, RTOL, "unaffected sequence", out_dtype=OUT_DT(w))


def test_append_out_of_pool_slot_is_reported_and_skipped():
    import paged_kv_cache_134_gb300 as P
    from gpu_path import new_cache, pool_numpy
    cache = new_cache(None, 4, 16, 1, 64, "f16", "f16")
    before = pool_numpy(cache)
    k = torch.randn(2, 1, 64, dtype=torch.float16, device="cuda")
    slots = torch.tensor([4 * 16, -1], dtype=torch.int64, device="cuda")
    P.paged_kv_append(cache, k, k, slots)
    assert cache.check_error() & 2
    assert np.array_equal(pool_numpy(cache), before)
    cache.close()


@pytest.mark.parametrize("src", ["f16", "bf16"])
@pytest.mark.parametrize("scale", [1.0, 0.125, 3.0])
def test_fp8_append_exhaustive_encode(src, scale):
    """Every 16-bit source pattern through the FP8 append, against the oracle's E4M3 encoder."""
    import paged_kv_cache_134_gb300 as P
    from gpu_path import dev, new_cache, pool_numpy, TORCH_DT
    d, bs = 64, 16
    n_tok = 65536 // d
    bits = np.arange(65536, dtype=np.uint16).reshape(n_tok, 1, d)
    cache = new_cache(None, n_tok // bs, bs, 1, d, "fp8", src, np.array([scale], np.float32),
                      np.array([scale], np.float32))
    slots = np.arange(n_tok, dtype=np.int64)
    P.paged_kv_append(cache, dev(bits, TORCH_DT[src]), dev(bits, TORCH_DT[src]), dev(slots))
    assert cache.check_error() == 0
    got = pool_numpy(cache).reshape(n_tok // bs, 2, 1, bs, d)
    ref = oracle.new_pool(got.size, "fp8", 0x7F)
    oracle.kv_append(ref, oracle.contiguous_strides(n_tok // bs, 1, bs, d), "fp8", n_tok // bs, bs, 1, d, bits, bits,
                     src, slots, np.array([scale], np.float32), np.array([scale], np.float32))
    assert np.array_equal(got.ravel(), ref), int(np.sum(got.ravel() != ref))
    cache.close()


def test_slot_mapping_matches_oracle_including_invalid():
    import paged_kv_cache_134_gb300 as P
    from gpu_path import dev
    rng = np.random.default_rng(46)
    for bs in (8, 16, 32):
        tables = rng.integers(-1, 5000, size=(37, 50)).astype(np.int32)
        seq = rng.integers(-2, 40, size=10000).astype(np.int32)
        pos = rng.integers(-5, 50 * bs + 20, size=10000).astype(np.int32)
        got = P.paged_slot_mapping(dev(tables), dev(seq), dev(pos), bs).cpu().numpy()
        assert np.array_equal(got, oracle.slot_mapping(tables, seq, pos, bs))


def test_fused_append_matches_slot_mapping_plus_append():
    w = W.small_decode("fuse", [0, 15, 16, 33, 500], hq=8, hkv=2, d=128, bs=16, seed=47)
    a = run_decode(w, fused=True)
    b = run_decode(w, fused=False)
    assert a["err"] == 0 and b["err"] == 0
    assert np.array_equal(a["new_slots"], b["new_slots"])
    assert np.array_equal(a["pool"], b["pool"])
    assert np.array_equal(a["out"], b["out"])


@pytest.mark.parametrize("hq,hkv,kv", [(8, 8, "f16"), (8, 2, "bf16"), (8, 2, "fp8")], ids=["mha_f16", "gqa4_bf16",
                                                                                      "gqa4_fp8"])
def test_more_sequences_than_one_launch(hq, hkv, kv):
    # 1500 sequences: more than one decode launch takes (1024, fewer for the tensor-core kernel of
    # grouped-query heads), so the call runs as consecutive launches sharing one workspace
    lens = np.random.default_rng(71).integers(0, 700, 1500)
    w = W.small_decode(f"many_{kv}", lens, hq=hq, hkv=hkv, d=128, bs=16, kv_dtype=kv, seed=72)
    check_decode(w, f"1500 sequences {kv} G={hq // hkv}")
