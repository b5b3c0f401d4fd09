"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each pin is chosen so that a plausible slip in the oracle (a dropped scale, a
wrong head mapping, an off-by-one tail, a swapped block/offset, a transposed
operand, a wrong rounding rule) fails at least one test:

* worked examples printed on the pages (tests/golden/*.json, each cited);
* library routines for the scalar formats (numpy float16, torch bfloat16 and
  torch float8_e4m3fn), plus brute-force nearest-value search over all codes;
* textbook contiguous attention (numpy matmul + softmax) on tiny inputs,
  computed from the logical per-sequence K/V and never from block tables;
* closed forms (one key returns V[0] exactly; equal keys return the mean of V)
  and invariants (softmax weights sum to 1, placement of physical blocks does
  not matter, shared prefix blocks equal private copies, NaN in unowned slots
  never reaches the output, packed sequences do not see each other).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import steps
from paged_kv_cache_134_gb300 import workloads as W

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------------------ scalar formats

def test_f16_decode_matches_numpy_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.f16_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_decode_matches_torch_all_patterns():
    bits = np.arange(65536, dtype=np.uint16)
    ours = oracle.bf16_to_double(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decode_matches_torch_and_ocp_table():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_to_double(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    g = gold("e4m3_ocp.json")
    for code, val in g["decode"]:
        v = oracle.e4m3_to_double(np.array([int(code, 16)], np.uint8))[0]
        assert v == val and math.copysign(1, v) == math.copysign(1, val), code
    for code in g["nan_codes"]:
        assert np.isnan(oracle.e4m3_to_double(np.array([int(code, 16)], np.uint8))[0])
    assert np.nanmax(ours) == 448.0 and np.nanmin(ours) == -448.0


def test_e4m3_encode_golden():
    for x, code in gold("e4m3_ocp.json")["encode"]:
        assert oracle.e4m3_encode(np.array([x], np.float32))[0] == int(code, 16), x


def _all_fp16_values():
    v = np.arange(65536, dtype=np.uint16).view(np.float16).astype(np.float32)
    return v[np.isfinite(v)]


def test_e4m3_encode_matches_torch_inside_range():
    # torch rounds to nearest-even like the OCP rule; it differs only where it overflows to NaN (>= 464)
    x = _all_fp16_values()
    x = np.concatenate([x, np.random.default_rng(0).standard_normal(20000).astype(np.float32) * 37])
    x = x[np.abs(x) < 464]
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_brute_force_nearest_even():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = oracle.e4m3_to_double(codes)
    x = _all_fp16_values()
    x = x[np.abs(x) <= 448]
    ours = oracle.e4m3_encode(x)
    dist = np.abs(x.astype(np.float64)[:, None] - vals[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    # ties go to the even code (mantissa LSB 0)
    for i in range(len(x)):
        cs = codes[cand[i]]
        if len(cs) > 1:   # +0 and -0 tie for tiny inputs: the sign of x decides
            cs = cs[(cs >> 7) == (1 if np.signbit(x[i]) else 0)]
        if len(cs) > 1:
            cs = cs[(cs & 1) == 0]
        assert len(cs) == 1 and cs[0] == ours[i], (x[i], cs, ours[i])


def test_e4m3_encode_saturates_and_nan():
    big = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, np.inf], np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)
    assert np.all(oracle.e4m3_encode(-big) == 0xFE)
    assert oracle.e4m3_encode(np.array([np.nan], np.float32))[0] == 0x7F


# ------------------------------------------------------------------------------ slot indexing

def test_slot_golden_2kiu_block_table():
    g = gold("block_table_2kiu.json")
    bs = g["block_size"]
    tables = np.array([g["table"]], np.int32)
    pos = np.arange(g["expect_positions_per_table"], dtype=np.int32)
    slots = oracle.slot_mapping(tables, np.zeros_like(pos), pos, bs)
    for p, blk in g["expect_block_of_position"]:
        assert slots[p] // bs == blk and slots[p] % bs == p % bs
    assert np.array_equal(slots // bs, np.repeat(g["table"], bs))


def test_slot_golden_discosf_block_table():
    g = gold("block_table_discosf.json")
    bs = g["block_size"]
    tables = np.full((g["seq"] + 1, len(g["row"])), -1, np.int32)
    tables[g["seq"]] = g["row"]
    for t, blk, off in g["expect"]:
        s = oracle.slot_mapping(tables, np.array([g["seq"]], np.int32), np.array([t], np.int32), bs)[0]
        assert (s // bs, s % bs) == (blk, off)
        assert s == blk * bs + off


def test_slot_partial_tail_block_discosf():
    g = gold("partial_block_discosf.json")
    bs = g["block_size"]
    assert W.blocks_for(g["length"], bs) == g["blocks"]
    tables = np.array([[5, 9]], np.int32)
    pos = np.arange(g["length"], dtype=np.int32)
    slots = oracle.slot_mapping(tables, np.zeros_like(pos), pos, bs)
    assert int(np.sum(slots // bs == 9)) == g["valid_in_last_block"]


def test_slot_brute_force_and_invalid():
    rng = np.random.default_rng(3)
    for bs in (8, 16, 32):
        tables = rng.integers(0, 1000, size=(5, 7)).astype(np.int32)
        tables[2, 4:] = -1
        seq = rng.integers(-1, 6, size=300).astype(np.int32)
        pos = rng.integers(-3, 7 * bs + 5, size=300).astype(np.int32)
        got = oracle.slot_mapping(tables, seq, pos, bs)
        for i in range(300):
            s, p = int(seq[i]), int(pos[i])
            if s < 0 or s >= 5 or p < 0 or p >= 7 * bs or tables[s, p // bs] < 0:
                assert got[i] == -1
            else:
                assert got[i] == int(tables[s, p // bs]) * bs + p % bs


# ------------------------------------------------------------------------------ append

def _pool_5d(pool, w):
    return pool.reshape(w.num_blocks, 2, w.num_kv_heads, w.block_size, w.head_dim)


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_append_readback_is_exact_and_touches_nothing_else(bs):
    w = W.small_decode("app", [3, 17, 40, 0], hq=4, hkv=2, d=64, bs=bs, seed=11)
    r = steps.decode_step(w)
    pool = _pool_5d(r["pool"], w)
    owned = np.zeros(pool.shape[:2] + (w.num_kv_heads, bs), bool)
    for s in range(w.num_seqs):
        k, v = W.logical_kv(w, s)
        for t in range(len(k)):
            b = w.block_tables[s, t // bs]
            assert np.array_equal(pool[b, 0, :, t % bs, :], k[t])
            assert np.array_equal(pool[b, 1, :, t % bs, :], v[t])
            owned[b, :, :, t % bs] = True
    assert np.all(pool[~owned] == W.NAN_BITS["f16"])


def test_append_fp8_power_of_two_scale_matches_torch():
    w = W.small_decode("app8", [5, 9], hq=4, hkv=2, d=64, bs=16, kv_dtype="fp8", seed=12)
    w.k_scale = np.array([0.25, 2.0], np.float32)   # divisions by powers of two are exact
    w.v_scale = np.array([1.0, 0.5], np.float32)
    r = steps.decode_step(w)
    pool = _pool_5d(r["pool"], w)
    for s in range(w.num_seqs):
        k, v = W.logical_kv(w, s)
        for kv, src, sc in ((0, k, w.k_scale), (1, v, w.v_scale)):
            x = (W.bits_to_float(src, "bf16") / sc[None, :, None]).astype(np.float32)
            ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            for t in range(len(src)):
                b = w.block_tables[s, t // 16]
                assert np.array_equal(pool[b, kv, :, t % 16, :], ref[t])


def test_append_skips_negative_and_counts_out_of_pool():
    pool = oracle.new_pool(2 * 2 * 1 * 4 * 8, "f16", 0x7E00)
    st = oracle.contiguous_strides(2, 1, 4, 8)
    k = np.arange(3 * 8, dtype=np.uint16).reshape(3, 1, 8)
    bad = oracle.kv_append(pool, st, "f16", 2, 4, 1, 8, k, k + 100, "f16", np.array([-1, 5, 8], np.int64))
    assert bad == 1
    p = pool.reshape(2, 2, 1, 4, 8)
    assert np.array_equal(p[1, 0, 0, 1], k[1, 0]) and np.array_equal(p[1, 1, 0, 1], k[1, 0] + 100)
    assert int(np.sum(p != 0x7E00)) == 16


# ------------------------------------------------------------------------------ decode

def brute_decode(w, out_dtype_bits=None):
    """Textbook attention on each sequence's contiguous logical K/V (no block tables)."""
    S, hq, d = w.q.shape
    G = hq // w.num_kv_heads
    q = W.bits_to_float(w.q, w.model_dtype)
    out = np.zeros((S, hq, d))
    for s in range(S):
        kb, vb = W.logical_kv(w, s)
        K, V = W.bits_to_float(kb, w.model_dtype), W.bits_to_float(vb, w.model_dtype)
        if w.kv_dtype == "fp8":
            Kq = torch.from_numpy((K / w.k_scale[None, :, None]).astype(np.float32)).to(torch.float8_e4m3fn)
            Vq = torch.from_numpy((V / w.v_scale[None, :, None]).astype(np.float32)).to(torch.float8_e4m3fn)
            K = Kq.to(torch.float64).numpy() * w.k_scale[None, :, None].astype(np.float64)
            V = Vq.to(torch.float64).numpy() * w.v_scale[None, :, None].astype(np.float64)
        for h in range(hq):
            x = float(w.scale) * (K[:, h // G, :] @ q[s, h])
            p = np.exp(x - x.max())
            p /= p.sum()
            out[s, h] = p @ V[:, h // G, :]
    return out


CASES = [
    dict(lens=[1, 15, 16, 37], hq=8, hkv=8, d=64, bs=16, kv_dtype="f16"),
    dict(lens=[0, 7, 33, 64, 100], hq=8, hkv=2, d=64, bs=8, kv_dtype="bf16"),
    dict(lens=[31, 32, 95], hq=4, hkv=1, d=128, bs=32, kv_dtype="f16"),
    dict(lens=[12, 70], hq=8, hkv=2, d=128, bs=16, kv_dtype="fp8"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{c['kv_dtype']}_G{c['hq'] // c['hkv']}_d{c['d']}_bs{c['bs']}")
def test_decode_matches_contiguous_brute_force(case):
    case = dict(case)
    w = W.small_decode("bf", case.pop("lens"), seed=21, **case)
    r = steps.decode_step(w, with_psum=True)
    ref = brute_decode(w)
    assert np.allclose(r["out"], ref, rtol=0, atol=1e-12)
    assert np.allclose(r["psum"], 1.0, atol=1e-12)


def test_decode_single_token_returns_v0_exactly():
    w = W.small_decode("one", [0, 0, 0], hq=4, hkv=2, d=64, bs=16, kv_dtype="bf16", seed=5)
    out = steps.decode_step(w)["out"]
    v = W.bits_to_float(w.new_v, "bf16")
    for s in range(3):
        for h in range(4):
            assert np.array_equal(out[s, h], v[s, h // 2])


def test_decode_equal_keys_gives_mean_of_v():
    w = W.small_decode("eq", [20, 45], hq=2, hkv=2, d=64, bs=16, seed=6)
    w.fill_k[:] = w.fill_k[0:1]
    w.new_k[:] = w.fill_k[0:1]
    out = steps.decode_step(w)["out"]
    for s in range(2):
        _, vb = W.logical_kv(w, s)
        mean = W.bits_to_float(vb, "f16").mean(axis=0)
        assert np.allclose(out[s], mean, rtol=0, atol=1e-13)


def test_decode_zero_length_gives_zero_row():
    w = W.small_decode("z", [3], hq=2, hkv=2, d=64, bs=16, seed=8)
    r = steps.decode_step(w)
    out = oracle.paged_decode(w.q, "f16", r["pool"], oracle.contiguous_strides(w.num_blocks, 2, 16, 64), "f16",
                              w.num_blocks, w.block_tables, np.array([0], np.int32), 2, 16, float(w.scale))
    assert np.all(out == 0)


def test_decode_invariant_to_physical_placement():
    a = W.small_decode("perm", [5, 40, 77], hq=4, hkv=4, d=64, bs=16, seed=9)
    b = W.small_decode("perm", [5, 40, 77], hq=4, hkv=4, d=64, bs=16, seed=9, num_blocks=a.num_blocks * 3,
                       placement_seed=123)
    assert not np.array_equal(a.block_tables, b.block_tables)
    assert np.array_equal(steps.decode_step(a)["out"], steps.decode_step(b)["out"])


def test_decode_shared_prefix_equals_private_copies():
    kw = dict(num_seqs=3, prefix_tokens=64, max_suffix=40, heads=2, d=64, bs=32)
    shared = W.prefix13b(**kw)
    private = W.prefix13b(private_prefix=True, **kw)
    assert shared.num_blocks < private.num_blocks
    prefix_blocks = shared.block_tables[:, :2]
    assert np.all(prefix_blocks == prefix_blocks[0:1])
    assert np.all(shared.ref_count[prefix_blocks[0]] == 3)
    assert np.array_equal(steps.decode_step(shared)["out"], steps.decode_step(private)["out"])
    assert np.allclose(steps.decode_step(shared)["out"], brute_decode(shared), atol=1e-12, rtol=0)


def test_decode_nan_in_unowned_slots_never_reaches_output():
    w = W.tiny()
    r = steps.decode_step(w)
    assert np.all(np.isfinite(r["out"]))
    nan_slots = np.sum(_pool_5d(r["pool"], w) == W.NAN_BITS["f16"])
    assert nan_slots > 0
    assert np.allclose(r["out"], brute_decode(w), atol=1e-12, rtol=0)


def test_decode_tail_is_masked_not_just_read():
    # a finite but huge value in the first unowned slot of a tail block would dominate if it were read
    w = W.small_decode("tail", [20], hq=2, hkv=2, d=64, bs=16, seed=10)
    r = steps.decode_step(w)
    pool = _pool_5d(r["pool"], w)
    b = w.block_tables[0, 1]
    pool[b, :, :, 21 % 16, :] = 0x7BFF   # 65504 in fp16
    out = oracle.paged_decode(w.q, "f16", r["pool"], oracle.contiguous_strides(w.num_blocks, 2, 16, 64), "f16",
                              w.num_blocks, w.block_tables, w.context_lens + 1, 2, 16, float(w.scale))
    assert np.array_equal(out, r["out"])


# ------------------------------------------------------------------------------ packed prefill

def brute_prefill(w):
    q = W.bits_to_float(w.q, w.dtype)
    k = W.bits_to_float(w.k, w.dtype)
    v = W.bits_to_float(w.v, w.dtype)
    G = w.num_q_heads // w.num_kv_heads
    out = np.zeros(q.shape)
    cu = w.cu_seqlens
    for i in range(len(w.lengths)):
        a, b = cu[i], cu[i + 1]
        n = b - a
        mask = np.triu(np.ones((n, n), bool), 1)
        for h in range(w.num_q_heads):
            x = float(w.scale) * (q[a:b, h] @ k[a:b, h // G].T)
            x[mask] = -np.inf
            p = np.exp(x - x.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            out[a:b, h] = p @ v[a:b, h // G]
    return out


def test_cu_seqlens_golden_and_packed_total():
    g = gold("cu_seqlens_discosf.json")
    w = W.prefill(lengths=g["lengths"], heads=1, d=64)
    assert w.cu_seqlens.tolist() == g["cu_seqlens"] and w.total_tokens == g["total_tokens"]
    p = gold("packed_lengths_discosf.json")
    assert sum(p["lengths"]) == p["packed_tokens"] != p["page_printed_total"]
    assert len(p["lengths"]) * max(p["lengths"]) == p["padded_tokens"]
    assert 1 - p["packed_tokens"] / p["padded_tokens"] > 0.6
    assert [W.blocks_for(n, 16) for n in p["lengths"]] == p["blocks_at_16"]
    assert 200 // 16 == p["length_200_full_blocks"] and 200 % 16 == p["length_200_tail_tokens"]


@pytest.mark.parametrize("heads,kv_heads,d", [(2, 2, 64), (4, 1, 128)])
def test_prefill_matches_causal_brute_force(heads, kv_heads, d):
    w = W.prefill(lengths=(3, 5, 2, 4, 33, 1), heads=heads, kv_heads=kv_heads, d=d, bs=16, seed=31)
    r = steps.prefill_step(w)
    assert np.allclose(r["out"], brute_prefill(w), atol=1e-12, rtol=0)


def test_prefill_sequences_are_independent():
    w = W.prefill(lengths=(17, 40, 9), heads=2, d=64, seed=32)
    base = steps.prefill_step(w)["out"]
    cu = w.cu_seqlens
    w.k[cu[1]:cu[2]] ^= 0x0400   # perturb sequence 1 only
    w.v[cu[1]:cu[2]] ^= 0x0400
    out = steps.prefill_step(w)["out"]
    for i in (0, 2):
        assert np.array_equal(out[cu[i]:cu[i + 1]], base[cu[i]:cu[i + 1]])
    assert not np.array_equal(out[cu[1]:cu[2]], base[cu[1]:cu[2]])


def test_prefill_first_row_is_v0_and_cache_holds_kv():
    w = W.prefill(lengths=(20, 1, 48), heads=2, kv_heads=1, d=64, bs=16, seed=33)
    r = steps.prefill_step(w)
    v = W.bits_to_float(w.v, "f16")
    for i in range(3):
        a = w.cu_seqlens[i]
        for h in range(2):
            assert np.array_equal(r["out"][a, h], v[a, 0])
    pool = r["pool"].reshape(w.num_blocks, 2, 1, 16, 64)
    for i, n in enumerate(w.lengths):
        for t in range(n):
            b = w.block_tables[i, t // 16]
            assert np.array_equal(pool[b, 0, 0, t % 16], w.k[w.cu_seqlens[i] + t, 0])
            assert np.array_equal(pool[b, 1, 0, t % 16], w.v[w.cu_seqlens[i] + t, 0])
