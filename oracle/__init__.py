"""CPU fp64 oracle for the paged KV cache hot path.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's CPU
baseline leg call it; the product path (the CUDA library and its binding)
never imports it.  It shares no code with the CUDA path: the arithmetic lives
in ``pagedkv_oracle.c`` (plain C99, fp64), built with gcc into
``oracle/_build/liboracle.so``; this module only marshals numpy arrays.

Each function states the passage it follows; the C source carries the same
citations.  Pins tying the oracle to things other than itself live in
``tests/test_oracle.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pagedkv_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

DTYPE = {"f16": 0, "bf16": 1, "fp8": 2}

_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (-O2, no fast-math, no FMA contraction, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.orc_f16_to_double.restype = ctypes.c_double
        lib.orc_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_bf16_to_double.restype = ctypes.c_double
        lib.orc_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.orc_e4m3_to_double.restype = ctypes.c_double
        lib.orc_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_slot_mapping.restype = None
        lib.orc_slot_mapping.argtypes = [_i32p, ctypes.c_int64, ctypes.c_int64, _i32p, _i32p, ctypes.c_int64,
                                         ctypes.c_int64, _i64p]
        lib.orc_kv_append.restype = ctypes.c_int64
        lib.orc_kv_append.argtypes = [_vp, _i64p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                      ctypes.c_int64, _u16p, _u16p, ctypes.c_int, _i64p, ctypes.c_int64, _f32p, _f32p]
        lib.orc_paged_decode.restype = ctypes.c_int64
        lib.orc_paged_decode.argtypes = [_u16p, ctypes.c_int, _vp, _i64p, ctypes.c_int, _f32p, _f32p, ctypes.c_int64,
                                         _i32p, ctypes.c_int64, _i32p, ctypes.c_int64, ctypes.c_int64,
                                         ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double, _f64p, _f64p]
        lib.orc_packed_prefill.restype = None
        lib.orc_packed_prefill.argtypes = [_u16p, _u16p, _u16p, ctypes.c_int, _i32p, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_int64, ctypes.c_double, _f64p]
        for name in ("orc_block_copy", "orc_block_swap_out", "orc_block_swap_in"):
            getattr(lib, name).restype = ctypes.c_int64
        lib.orc_block_copy.argtypes = [_vp, _i64p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.c_int64, _i32p, _i32p, ctypes.c_int64]
        lib.orc_block_swap_out.argtypes = [_vp, _i64p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                           ctypes.c_int64, _i32p, ctypes.c_int64, _vp]
        lib.orc_block_swap_in.argtypes = list(lib.orc_block_swap_out.argtypes)
        lib.orc_prefill_ctx.restype = ctypes.c_int64
        lib.orc_prefill_ctx.argtypes = [_u16p, ctypes.c_int, _vp, _i64p, ctypes.c_int, _f32p, _f32p, ctypes.c_int64,
                                        _i32p, ctypes.c_int64, _i32p, _i32p, ctypes.c_int64, ctypes.c_int64,
                                        ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_double, _f64p]
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_init()
        _lib = lib
        return lib


def _p(a: np.ndarray, t):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(t)


def num_threads() -> int:
    return int(_load().orc_num_threads())


# ----------------------------------------------------------------------------- scalar formats

def f16_to_double(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    return np.array([lib.orc_f16_to_double(int(b)) for b in np.asarray(bits, np.uint16).ravel()]).reshape(np.shape(bits))


def bf16_to_double(bits: np.ndarray) -> np.ndarray:
    lib = _load()
    return np.array([lib.orc_bf16_to_double(int(b)) for b in np.asarray(bits, np.uint16).ravel()]).reshape(np.shape(bits))


def e4m3_to_double(codes: np.ndarray) -> np.ndarray:
    lib = _load()
    return np.array([lib.orc_e4m3_to_double(int(c)) for c in np.asarray(codes, np.uint8).ravel()]).reshape(np.shape(codes))


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """OCP E4M3 code of each binary32 value (round-to-nearest-even, saturate to +-448, NaN -> 0x7F)."""
    lib = _load()
    x = np.asarray(x, np.float32)
    return np.array([lib.orc_e4m3_encode(float(v)) for v in x.ravel()], dtype=np.uint8).reshape(x.shape)


# ----------------------------------------------------------------------------- slot indexing

def slot_mapping(tables: np.ndarray, seq_ids: np.ndarray, positions: np.ndarray, block_size: int) -> np.ndarray:
    """slot = table[s][p // bs] * bs + p % bs  (discosf.com "Paged KV Cache 与 Packed Sequence", section 2.2)."""
    tables = np.ascontiguousarray(tables, np.int32)
    seq_ids = np.ascontiguousarray(seq_ids, np.int32)
    positions = np.ascontiguousarray(positions, np.int32)
    out = np.empty(len(positions), np.int64)
    _load().orc_slot_mapping(_p(tables, _i32p), tables.shape[0], tables.shape[1], _p(seq_ids, _i32p),
                             _p(positions, _i32p), len(positions), int(block_size), _p(out, _i64p))
    return out


# ----------------------------------------------------------------------------- pool model

def contiguous_strides(num_blocks, hkv, bs, d):
    """Element strides of a C-contiguous (block, K|V, head, offset, dim) pool."""
    return np.array([2 * hkv * bs * d, hkv * bs * d, bs * d, d, 1], np.int64)


def new_pool(num_elems: int, cache_dtype: str, fill_bits: int) -> np.ndarray:
    dt = np.uint8 if cache_dtype == "fp8" else np.uint16
    return np.full(int(num_elems), fill_bits, dtype=dt)


def kv_append(pool: np.ndarray, strides, cache_dtype: str, num_blocks: int, block_size: int, hkv: int, d: int,
              k_bits: np.ndarray, v_bits: np.ndarray, src_dtype: str, slots: np.ndarray,
              k_scale=None, v_scale=None) -> int:
    """Write each token's K/V at its slot (in place); returns the count of out-of-pool slots skipped."""
    strides = np.ascontiguousarray(strides, np.int64)
    k_bits = np.ascontiguousarray(k_bits, np.uint16)
    v_bits = np.ascontiguousarray(v_bits, np.uint16)
    slots = np.ascontiguousarray(slots, np.int64)
    if cache_dtype == "fp8":
        ks = np.ascontiguousarray(k_scale, np.float32)
        vs = np.ascontiguousarray(v_scale, np.float32)
        ksp, vsp = _p(ks, _f32p), _p(vs, _f32p)
    else:
        ksp = vsp = None
    return int(_load().orc_kv_append(pool.ctypes.data, _p(strides, _i64p), DTYPE[cache_dtype], num_blocks,
                                     block_size, hkv, d, _p(k_bits, _u16p), _p(v_bits, _u16p), DTYPE[src_dtype],
                                     _p(slots, _i64p), len(slots), ksp, vsp))


def paged_decode(q_bits: np.ndarray, q_dtype: str, pool: np.ndarray, strides, cache_dtype: str, num_blocks: int,
                 tables: np.ndarray, context_lens: np.ndarray, hkv: int, block_size: int, scale: float,
                 k_scale=None, v_scale=None, with_psum: bool = False):
    """fp64 paged decode attention (2kiu.com "PagedAttention 与前缀缓存", section 2.3).

    Returns out [S, Hq, D] float64 (and the per-row softmax weight sums when asked)."""
    q_bits = np.ascontiguousarray(q_bits, np.uint16)
    S, hq, d = q_bits.shape
    tables = np.ascontiguousarray(tables, np.int32)
    lens = np.ascontiguousarray(context_lens, np.int32)
    strides = np.ascontiguousarray(strides, np.int64)
    out = np.zeros((S, hq, d), np.float64)
    psum = np.zeros((S, hq), np.float64)
    if cache_dtype == "fp8":
        ks = np.ascontiguousarray(k_scale, np.float32)
        vs = np.ascontiguousarray(v_scale, np.float32)
        ksp, vsp = _p(ks, _f32p), _p(vs, _f32p)
    else:
        ksp = vsp = None
    bad = _load().orc_paged_decode(_p(q_bits, _u16p), DTYPE[q_dtype], pool.ctypes.data, _p(strides, _i64p),
                                   DTYPE[cache_dtype], ksp, vsp, num_blocks, _p(tables, _i32p), tables.shape[1],
                                   _p(lens, _i32p), S, hq, hkv, d, block_size, float(scale), _p(out, _f64p),
                                   _p(psum, _f64p))
    if bad:
        raise ValueError(f"{bad} (sequence, head) rows needed a block id outside the pool")
    return (out, psum) if with_psum else out


def packed_prefill(q_bits: np.ndarray, k_bits: np.ndarray, v_bits: np.ndarray, dtype: str, cu_seqlens: np.ndarray,
                   scale: float) -> np.ndarray:
    """fp64 block-diagonal causal attention over packed sequences (discosf.com section 3)."""
    q_bits = np.ascontiguousarray(q_bits, np.uint16)
    k_bits = np.ascontiguousarray(k_bits, np.uint16)
    v_bits = np.ascontiguousarray(v_bits, np.uint16)
    cu = np.ascontiguousarray(cu_seqlens, np.int32)
    T, hq, d = q_bits.shape
    hkv = k_bits.shape[1]
    out = np.zeros((T, hq, d), np.float64)
    _load().orc_packed_prefill(_p(q_bits, _u16p), _p(k_bits, _u16p), _p(v_bits, _u16p), DTYPE[dtype], _p(cu, _i32p),
                               len(cu) - 1, hq, hkv, d, float(scale), _p(out, _f64p))
    return out


# ----------------------------------------------------------------------------- whole-block copies

def _block_args(pool, strides, block_size, hkv, d):
    strides = np.ascontiguousarray(strides, np.int64)
    return pool.ctypes.data, strides, int(pool.itemsize), int(block_size), int(hkv), int(d)


def block_copy(pool: np.ndarray, strides, num_blocks: int, block_size: int, hkv: int, d: int,
               src_ids: np.ndarray, dst_ids: np.ndarray) -> int:
    """Copy-on-write (2kiu.com section 2.2, 4.3): block dst_ids[i] := block src_ids[i], in place.
    Returns the number of pairs skipped for an id outside the pool."""
    base, st, elt, bs, hkv, d = _block_args(pool, strides, block_size, hkv, d)
    src = np.ascontiguousarray(src_ids, np.int32)
    dst = np.ascontiguousarray(dst_ids, np.int32)
    assert len(src) == len(dst)
    return int(_load().orc_block_copy(base, _p(st, _i64p), elt, num_blocks, bs, hkv, d, _p(src, _i32p),
                                      _p(dst, _i32p), len(src)))


def block_swap_out(pool: np.ndarray, strides, num_blocks: int, block_size: int, hkv: int, d: int,
                   ids: np.ndarray):
    """Swap out (2kiu.com sections 2.2, 5.2): returns (buffer, skipped) with buffer block i = pool
    block ids[i] in the documented order [K|V][head][slot][dim]; skipped blocks stay zero."""
    base, st, elt, bs, hkv, d = _block_args(pool, strides, block_size, hkv, d)
    ids = np.ascontiguousarray(ids, np.int32)
    buf = np.zeros(len(ids) * 2 * hkv * bs * d, dtype=pool.dtype)
    bad = _load().orc_block_swap_out(base, _p(st, _i64p), elt, num_blocks, bs, hkv, d, _p(ids, _i32p), len(ids),
                                     buf.ctypes.data)
    return buf, int(bad)


def block_swap_in(pool: np.ndarray, strides, num_blocks: int, block_size: int, hkv: int, d: int,
                  ids: np.ndarray, buf: np.ndarray) -> int:
    """Swap in: pool block ids[i] := buffer block i, in place.  Returns the count of skipped ids."""
    base, st, elt, bs, hkv, d = _block_args(pool, strides, block_size, hkv, d)
    ids = np.ascontiguousarray(ids, np.int32)
    buf = np.ascontiguousarray(buf, pool.dtype)
    assert buf.size >= len(ids) * 2 * hkv * bs * d
    return int(_load().orc_block_swap_in(base, _p(st, _i64p), elt, num_blocks, bs, hkv, d, _p(ids, _i32p),
                                         len(ids), buf.ctypes.data))


# ----------------------------------------------------------------------------- prefill on a cached prefix

def prefill_ctx(q_bits: np.ndarray, q_dtype: str, pool: np.ndarray, strides, cache_dtype: str, num_blocks: int,
                tables: np.ndarray, cu_seqlens: np.ndarray, context_lens: np.ndarray, hkv: int, block_size: int,
                scale: float, k_scale=None, v_scale=None) -> np.ndarray:
    """fp64 attention of the tail tokens of each prompt over its cached prefix and itself, every key
    read from the pool through the table (2kiu.com section 4.3 steps 2-4).  The tail tokens' K/V
    must already be in the pool.  Returns out [T, Hq, D] float64."""
    q_bits = np.ascontiguousarray(q_bits, np.uint16)
    T, hq, d = q_bits.shape
    tables = np.ascontiguousarray(tables, np.int32)
    cu = np.ascontiguousarray(cu_seqlens, np.int32)
    ctx = np.ascontiguousarray(context_lens, np.int32)
    strides = np.ascontiguousarray(strides, np.int64)
    out = np.zeros((T, hq, d), np.float64)
    if cache_dtype == "fp8":
        ks = np.ascontiguousarray(k_scale, np.float32)
        vs = np.ascontiguousarray(v_scale, np.float32)
        ksp, vsp = _p(ks, _f32p), _p(vs, _f32p)
    else:
        ksp = vsp = None
    bad = _load().orc_prefill_ctx(_p(q_bits, _u16p), DTYPE[q_dtype], pool.ctypes.data, _p(strides, _i64p),
                                  DTYPE[cache_dtype], ksp, vsp, num_blocks, _p(tables, _i32p), tables.shape[1],
                                  _p(cu, _i32p), _p(ctx, _i32p), len(cu) - 1, hq, hkv, d, block_size, float(scale),
                                  _p(out, _f64p))
    if bad:
        raise ValueError(f"{bad} rows needed a block id outside the pool")
    return out
