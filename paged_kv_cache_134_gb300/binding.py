"""Thin ctypes binding over the C ABI of ``libpagedkv.so`` (include/pagedkv.h).

Argument marshalling only: tensors are checked for device, dtype, shape and contiguity and
passed as raw device pointers together with torch's current CUDA stream.  Every step of the
hot path runs in the library's kernels.  If the library has not been built, every call
raises ``RuntimeError``: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "lib", "libpagedkv.so")

PKV_F16, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2
_DT = {"f16": PKV_F16, "bf16": PKV_BF16, "fp8": PKV_FP8_E4M3}
_TORCH = {PKV_F16: torch.float16, PKV_BF16: torch.bfloat16}
DEVERR = {1: "block id", 2: "slot", 4: "length", 8: "cu_seqlens", 16: "timeout"}

_lock = threading.Lock()
_lib = None


class PagedKVError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"pagedkv status {status}: {msg}")
        self.status = status


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"CUDA library {LIB_PATH} is not built; run __graft_entry__.build() "
                               "(paged_kv_cache_134_gb300.build.build()) on a machine with nvcc")
        L = ctypes.CDLL(LIB_PATH)
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
        L.kv_cache_create.argtypes = [i64, i32, i32, i32, i32, i32, ctypes.POINTER(vp)]
        L.kv_cache_destroy.argtypes = [vp]
        L.kv_cache_set_scales.argtypes = [vp, vp, vp, vp]
        L.kv_cache_view.argtypes = [vp, ctypes.POINTER(vp), ctypes.POINTER(i64), ctypes.POINTER(i64)]
        L.kv_cache_reserve.argtypes = [vp, i32, i32, i32]
        L.kv_cache_check_error.argtypes = [vp, ctypes.POINTER(i32)]
        L.pkv_last_error.restype = ctypes.c_char_p
        L.paged_slot_mapping.argtypes = [vp, i32, i32, vp, vp, i64, i32, vp, vp]
        L.paged_kv_append.argtypes = [vp, vp, vp, vp, i64, vp]
        L.paged_kv_append_at.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp, i64, vp, vp]
        L.paged_decode_attention.argtypes = [vp, vp, vp, i32, vp, i32, i32, ctypes.c_float, vp, vp]
        L.paged_decode_attention_noalloc.argtypes = [vp, vp, vp, i32, vp, i32, i32, ctypes.c_float, vp, vp]
        L.packed_prefill_attention.argtypes = [vp, vp, vp, vp, i32, i32, i64, vp, i32, vp, i32, ctypes.c_float, vp,
                                               vp]
        L.paged_prefill_attention.argtypes = [vp, vp, vp, vp, vp, i32, i32, i64, vp, i32, vp, i32, ctypes.c_float, vp,
                                              vp]
        L.paged_block_copy.argtypes = [vp, vp, vp, i64, vp]
        L.paged_decode_attention_cascade.argtypes = [vp, vp, vp, i32, vp, i32, i32, i32, ctypes.c_float, vp, vp]
        L.pkv_block_hashes.argtypes = [vp, i64, i32, vp, i64, vp, vp, ctypes.POINTER(i64)]
        L.pkv_prefix_cache_create.argtypes = [i64, ctypes.POINTER(vp)]
        L.pkv_prefix_cache_destroy.argtypes = [vp]
        L.pkv_prefix_cache_match.argtypes = [vp, vp, i64, vp, ctypes.POINTER(i64)]
        L.pkv_prefix_cache_allocate.argtypes = [vp, i64, vp]
        L.pkv_prefix_cache_insert.argtypes = [vp, vp, vp, i64]
        L.pkv_prefix_cache_release.argtypes = [vp, vp, i64]
        L.pkv_prefix_cache_stats.argtypes = [vp, vp]
        L.paged_block_swap_out.argtypes = [vp, vp, i64, vp, vp]
        L.paged_block_swap_in.argtypes = [vp, vp, i64, vp, vp]
        L.kv_cache_profile_start.argtypes = [vp, ctypes.c_uint]
        L.kv_cache_profile_start_sampled.argtypes = [vp, ctypes.c_uint, ctypes.c_int]
        L.kv_cache_profile_read.argtypes = [vp, ctypes.c_void_p]
        L.pkv_kernel_launches.restype = i64
        L.kv_cache_selftest_wait_timeout.argtypes = [vp, ctypes.c_uint64, vp]
        _lib = L
        return L


class _Profile(ctypes.Structure):
    _fields_ = [("decode_launches", ctypes.c_int64), ("prefill_launches", ctypes.c_int64),
                ("append_launches", ctypes.c_int64), ("merge_launches", ctypes.c_int64),
                ("decode_ms", ctypes.c_double), ("prefill_ms", ctypes.c_double), ("append_ms", ctypes.c_double),
                ("merge_ms", ctypes.c_double), ("copy_launches", ctypes.c_int64), ("copy_ms", ctypes.c_double)]


def _check(status: int):
    if status != 0:
        raise PagedKVError(status, lib().pkv_last_error().decode(errors="replace"))


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _req(t: torch.Tensor, name: str, dtype=None, ndim=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {t.dim()}")


class _DevMem:
    """Exposes a raw device range through __cuda_array_interface__ for a zero-copy torch view."""

    def __init__(self, ptr: int, nbytes: int, owner):
        self.__cuda_array_interface__ = {"shape": (int(nbytes),), "typestr": "|u1", "data": (int(ptr), False),
                                         "version": 3, "strides": None}
        self._owner = owner


class KVCache:
    """A block pool on the current CUDA device (kv_cache_create)."""

    def __init__(self, num_blocks: int, block_size: int, num_kv_heads: int, head_dim: int,
                 kv_dtype: str = "f16", model_dtype: Optional[str] = None):
        L = lib()
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self.num_kv_heads, self.head_dim = int(num_kv_heads), int(head_dim)
        self.kv_dtype = kv_dtype
        self.model_dtype = model_dtype or (kv_dtype if kv_dtype != "fp8" else "bf16")
        h = ctypes.c_void_p()
        _check(L.kv_cache_create(self.num_blocks, self.block_size, self.num_kv_heads, self.head_dim,
                                 _DT[kv_dtype], _DT[self.model_dtype], ctypes.byref(h)))
        self._h = h
        self.torch_dtype = _TORCH[_DT[self.model_dtype]]

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None:
            raise RuntimeError("cache is closed")
        return self._h

    def close(self):
        if getattr(self, "_h", None) is not None:
            lib().kv_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def view(self):
        """(uint8 tensor over the whole pool, element strides of (block, K|V, head, offset, dim))."""
        base = ctypes.c_void_p()
        st = (ctypes.c_int64 * 5)()
        nbytes = ctypes.c_int64()
        _check(lib().kv_cache_view(self.handle, ctypes.byref(base), st, ctypes.byref(nbytes)))
        raw = torch.as_tensor(_DevMem(base.value, nbytes.value, self), device="cuda")
        return raw, [int(x) for x in st]

    def pool_elems(self) -> torch.Tensor:
        """The pool as a flat tensor of raw elements (int16 for 16-bit caches, uint8 for FP8)."""
        raw, _ = self.view()
        return raw if self.kv_dtype == "fp8" else raw.view(torch.int16)

    def set_scales(self, k_scale: torch.Tensor, v_scale: torch.Tensor):
        _req(k_scale, "k_scale", torch.float32, 1)
        _req(v_scale, "v_scale", torch.float32, 1)
        if k_scale.numel() != self.num_kv_heads or v_scale.numel() != self.num_kv_heads:
            raise ValueError("one scale per KV head")
        _check(lib().kv_cache_set_scales(self.handle, _ptr(k_scale), _ptr(v_scale), _stream()))

    def reserve(self, max_seqs: int, max_q_heads: int, max_blocks_per_seq: int):
        _check(lib().kv_cache_reserve(self.handle, int(max_seqs), int(max_q_heads), int(max_blocks_per_seq)))

    def check_error(self) -> int:
        """Synchronise and return (and clear) the device error bits; 0 when clean."""
        code = ctypes.c_int(0)
        st = lib().kv_cache_check_error(self.handle, ctypes.byref(code))
        if st not in (0, -5):
            _check(st)
        return int(code.value)

    def selftest_wait_timeout(self, limit_ns: int = 1_000_000):
        """Enqueue the bounded-wait self-test: a kernel waits on an mbarrier that never completes
        and gives up after limit_ns, setting the timeout bit that check_error then returns."""
        _check(lib().kv_cache_selftest_wait_timeout(self.handle, int(limit_ns), _stream()))

    PROFILE = {"decode": 1, "prefill": 2, "append": 4, "merge": 8, "copy": 16}

    @property
    def block_bytes(self) -> int:
        """Bytes of one physical block (K and V of every KV head)."""
        return 2 * self.num_kv_heads * self.block_size * self.head_dim * (1 if self.kv_dtype == "fp8" else 2)

    def profile_start(self, kinds=("decode", "prefill", "append", "merge"), every: int = 1):
        """Record CUDA events around the named kernels (events between kernels stop their overlap);
        with every > 1 only around every n-th launch of each kind."""
        mask = 0
        for k in kinds:
            mask |= self.PROFILE[k]
        _check(lib().kv_cache_profile_start_sampled(self.handle, mask, int(every)))

    def profile_read(self) -> dict:
        p = _Profile()
        _check(lib().kv_cache_profile_read(self.handle, ctypes.byref(p)))
        return {k: getattr(p, k) for k, _ in _Profile._fields_}


def kernel_launches() -> int:
    return int(lib().pkv_kernel_launches())


def paged_slot_mapping(block_tables: torch.Tensor, seq_ids: torch.Tensor, positions: torch.Tensor,
                       block_size: int, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    _req(block_tables, "block_tables", torch.int32, 2)
    _req(seq_ids, "seq_ids", torch.int32, 1)
    _req(positions, "positions", torch.int32, 1)
    n = positions.numel()
    if seq_ids.numel() != n:
        raise ValueError("seq_ids and positions differ in length")
    if out is None:
        out = torch.empty(n, dtype=torch.int64, device=positions.device)
    _req(out, "out", torch.int64, 1)
    _check(lib().paged_slot_mapping(_ptr(block_tables), block_tables.shape[0], block_tables.shape[1],
                                    _ptr(seq_ids), _ptr(positions), n, int(block_size), _ptr(out), _stream()))
    return out


def paged_kv_append(cache: KVCache, k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor) -> None:
    _req(k, "k", cache.torch_dtype, 3)
    _req(v, "v", cache.torch_dtype, 3)
    _req(slot_mapping, "slot_mapping", torch.int64, 1)
    n = k.shape[0]
    if tuple(k.shape) != (n, cache.num_kv_heads, cache.head_dim) or k.shape != v.shape:
        raise ValueError(f"k/v must be [T, {cache.num_kv_heads}, {cache.head_dim}]")
    if slot_mapping.numel() != n:
        raise ValueError("slot_mapping length != number of tokens")
    _check(lib().paged_kv_append(cache.handle, _ptr(k), _ptr(v), _ptr(slot_mapping), n, _stream()))


def paged_kv_append_at(cache: KVCache, k: torch.Tensor, v: torch.Tensor, block_tables: torch.Tensor,
                       seq_ids: torch.Tensor, positions: torch.Tensor,
                       slot_mapping: Optional[torch.Tensor] = None) -> Optional[torch.Tensor]:
    """Slot indexing + append in one launch; fills ``slot_mapping`` (int64) when given."""
    _req(k, "k", cache.torch_dtype, 3)
    _req(v, "v", cache.torch_dtype, 3)
    _req(block_tables, "block_tables", torch.int32, 2)
    _req(seq_ids, "seq_ids", torch.int32, 1)
    _req(positions, "positions", torch.int32, 1)
    n = k.shape[0]
    if tuple(k.shape) != (n, cache.num_kv_heads, cache.head_dim) or k.shape != v.shape:
        raise ValueError(f"k/v must be [T, {cache.num_kv_heads}, {cache.head_dim}]")
    if seq_ids.numel() != n or positions.numel() != n:
        raise ValueError("seq_ids/positions length != number of tokens")
    if slot_mapping is not None:
        _req(slot_mapping, "slot_mapping", torch.int64, 1)
        if slot_mapping.numel() != n:
            raise ValueError("slot_mapping length != number of tokens")
    _check(lib().paged_kv_append_at(cache.handle, _ptr(k), _ptr(v), _ptr(block_tables), block_tables.shape[0],
                                    block_tables.shape[1], _ptr(seq_ids), _ptr(positions), n, _ptr(slot_mapping),
                                    _stream()))
    return slot_mapping


def paged_decode_attention(q: torch.Tensor, cache: KVCache, block_tables: torch.Tensor,
                           context_lens: torch.Tensor, scale: float,
                           out: Optional[torch.Tensor] = None) -> torch.Tensor:
    _req(q, "q", cache.torch_dtype, 3)
    _req(block_tables, "block_tables", torch.int32, 2)
    _req(context_lens, "context_lens", torch.int32, 1)
    S, hq, d = q.shape
    if d != cache.head_dim or block_tables.shape[0] != S or context_lens.numel() != S:
        raise ValueError("shape mismatch between q, block_tables and context_lens")
    if out is None:
        out = torch.empty_like(q)
    _req(out, "out", cache.torch_dtype, 3)
    _check(lib().paged_decode_attention(_ptr(q), cache.handle, _ptr(block_tables), block_tables.shape[1],
                                        _ptr(context_lens), S, hq, ctypes.c_float(scale), _ptr(out), _stream()))
    return out


def paged_decode_attention_cascade(q: torch.Tensor, cache: KVCache, block_tables: torch.Tensor,
                                   context_lens: torch.Tensor, shared_prefix_len: int, scale: float,
                                   out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """paged_decode_attention for a batch whose tables share their first ``shared_prefix_len`` tokens."""
    _req(q, "q", cache.torch_dtype, 3)
    _req(block_tables, "block_tables", torch.int32, 2)
    _req(context_lens, "context_lens", torch.int32, 1)
    S, hq, d = q.shape
    if d != cache.head_dim or block_tables.shape[0] != S or context_lens.numel() != S:
        raise ValueError("shape mismatch between q, block_tables and context_lens")
    if out is None:
        out = torch.empty_like(q)
    _req(out, "out", cache.torch_dtype, 3)
    _check(lib().paged_decode_attention_cascade(_ptr(q), cache.handle, _ptr(block_tables), block_tables.shape[1],
                                                _ptr(context_lens), S, hq, int(shared_prefix_len),
                                                ctypes.c_float(scale), _ptr(out), _stream()))
    return out


def paged_decode_attention_noalloc(q: torch.Tensor, cache: KVCache, block_tables: torch.Tensor,
                                   context_lens: torch.Tensor, scale: float, out: torch.Tensor) -> torch.Tensor:
    """paged_decode_attention for callers that must not allocate device memory.

    The library keeps the split-K partials in a fixed 16 MiB array of its own (made resident when
    the cache was created) instead of the cache's growable workspace, so this call allocates
    nothing (the caller provides ``out``).  Calls that can overlap on the GPU share that array and
    must be serialised by the caller."""
    _req(q, "q", cache.torch_dtype, 3)
    _req(block_tables, "block_tables", torch.int32, 2)
    _req(context_lens, "context_lens", torch.int32, 1)
    _req(out, "out", cache.torch_dtype, 3)
    S, hq, d = q.shape
    if d != cache.head_dim or block_tables.shape[0] != S or context_lens.numel() != S or out.shape != q.shape:
        raise ValueError("shape mismatch between q, out, block_tables and context_lens")
    _check(lib().paged_decode_attention_noalloc(_ptr(q), cache.handle, _ptr(block_tables), block_tables.shape[1],
                                                _ptr(context_lens), S, hq, ctypes.c_float(scale), _ptr(out),
                                                _stream()))
    return out


def packed_prefill_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                             max_seqlen: int, block_tables: torch.Tensor, cache: KVCache, scale: float,
                             out: Optional[torch.Tensor] = None) -> torch.Tensor:
    for name, t in (("q", q), ("k", k), ("v", v)):
        _req(t, name, cache.torch_dtype, 3)
    _req(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _req(block_tables, "block_tables", torch.int32, 2)
    T, hq, d = q.shape
    if k.shape != (T, cache.num_kv_heads, d) or v.shape != k.shape or d != cache.head_dim:
        raise ValueError("q/k/v shape mismatch")
    nseq = cu_seqlens.numel() - 1
    if block_tables.shape[0] != nseq:
        raise ValueError("one block-table row per sequence")
    if out is None:
        out = torch.empty_like(q)
    _req(out, "out", cache.torch_dtype, 3)
    _check(lib().packed_prefill_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), nseq, int(max_seqlen), T,
                                          _ptr(block_tables), block_tables.shape[1], cache.handle, hq,
                                          ctypes.c_float(scale), _ptr(out), _stream()))
    return out


def _req_buffer(t: torch.Tensor, name: str, nbytes: int):
    """A contiguous byte buffer the GPU can reach: a CUDA tensor or page-locked host memory."""
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() * t.element_size() < nbytes:
        raise ValueError(f"{name} holds {t.numel() * t.element_size()} bytes, {nbytes} needed")


def paged_block_copy(cache: KVCache, src_blocks: torch.Tensor, dst_blocks: torch.Tensor) -> None:
    """Copy-on-write: block dst_blocks[i] := block src_blocks[i] (whole blocks)."""
    _req(src_blocks, "src_blocks", torch.int32, 1)
    _req(dst_blocks, "dst_blocks", torch.int32, 1)
    if src_blocks.numel() != dst_blocks.numel():
        raise ValueError("src_blocks and dst_blocks differ in length")
    _check(lib().paged_block_copy(cache.handle, _ptr(src_blocks), _ptr(dst_blocks), src_blocks.numel(), _stream()))


def paged_block_swap_out(cache: KVCache, block_ids: torch.Tensor, dst: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Gather whole blocks into ``dst`` (uint8, CUDA or pinned host; block i at i * block_bytes)."""
    _req(block_ids, "block_ids", torch.int32, 1)
    n = block_ids.numel()
    if dst is None:
        dst = torch.empty(n * cache.block_bytes, dtype=torch.uint8).pin_memory()
    _req_buffer(dst, "dst", n * cache.block_bytes)
    _check(lib().paged_block_swap_out(cache.handle, _ptr(block_ids), n, _ptr(dst), _stream()))
    return dst


def paged_block_swap_in(cache: KVCache, block_ids: torch.Tensor, src: torch.Tensor) -> None:
    """Scatter whole blocks back: block block_ids[i] := src[i * block_bytes : (i + 1) * block_bytes]."""
    _req(block_ids, "block_ids", torch.int32, 1)
    n = block_ids.numel()
    _req_buffer(src, "src", n * cache.block_bytes)
    _check(lib().paged_block_swap_in(cache.handle, _ptr(block_ids), n, _ptr(src), _stream()))


def paged_prefill_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens: torch.Tensor,
                            context_lens: torch.Tensor, max_seqlen: int, block_tables: torch.Tensor, cache: KVCache,
                            scale: float, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Prefill of each prompt's tail over the prefix its blocks already hold (writes the tail's K/V)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _req(t, name, cache.torch_dtype, 3)
    _req(cu_seqlens, "cu_seqlens", torch.int32, 1)
    _req(context_lens, "context_lens", torch.int32, 1)
    _req(block_tables, "block_tables", torch.int32, 2)
    T, hq, d = q.shape
    if k.shape != (T, cache.num_kv_heads, d) or v.shape != k.shape or d != cache.head_dim:
        raise ValueError("q/k/v shape mismatch")
    nseq = cu_seqlens.numel() - 1
    if block_tables.shape[0] != nseq or context_lens.numel() != nseq:
        raise ValueError("one block-table row and one context length per sequence")
    if out is None:
        out = torch.empty_like(q)
    _req(out, "out", cache.torch_dtype, 3)
    _check(lib().paged_prefill_attention(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens), _ptr(context_lens), nseq,
                                         int(max_seqlen), T, _ptr(block_tables), block_tables.shape[1], cache.handle,
                                         hq, ctypes.c_float(scale), _ptr(out), _stream()))
    return out


# ----------------------------------------------------------------------------- prefix cache (host)

def _np(a, dtype):
    import numpy as np
    return np.ascontiguousarray(a, dtype=dtype)


def block_hashes(tokens, block_size: int, extra: bytes = b"", init: Optional[bytes] = None):
    """Chained SHA-256 hashes of the full blocks of ``tokens`` (host); returns uint8 [n, 32]."""
    import numpy as np
    tok = _np(tokens, np.int32)
    n = len(tok) // int(block_size)
    out = np.zeros((n, 32), np.uint8)
    got = ctypes.c_int64(0)
    ex = ctypes.create_string_buffer(bytes(extra), len(extra)) if extra else None
    ini = ctypes.create_string_buffer(bytes(init), 32) if init is not None else None
    _check(lib().pkv_block_hashes(tok.ctypes.data, len(tok), int(block_size), ex, len(extra), ini,
                                  out.ctypes.data, ctypes.byref(got)))
    assert got.value == n
    return out


class PrefixCache:
    """Host prefix cache: hash -> physical block map, reference counts, LRU retention."""

    def __init__(self, num_blocks: int):
        h = ctypes.c_void_p()
        _check(lib().pkv_prefix_cache_create(int(num_blocks), ctypes.byref(h)))
        self._h = h

    def close(self):
        if getattr(self, "_h", None) is not None:
            lib().pkv_prefix_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def match(self, hashes):
        """Blocks of the longest cached prefix (attached: reference count + 1)."""
        import numpy as np
        hs = _np(hashes, np.uint8).reshape(-1, 32)
        out = np.zeros(len(hs), np.int32)
        hit = ctypes.c_int64(0)
        _check(lib().pkv_prefix_cache_match(self._h, hs.ctypes.data, len(hs), out.ctypes.data, ctypes.byref(hit)))
        return out[: hit.value]

    def allocate(self, n: int):
        import numpy as np
        out = np.zeros(int(n), np.int32)
        _check(lib().pkv_prefix_cache_allocate(self._h, int(n), out.ctypes.data))
        return out

    def insert(self, hashes, blocks):
        import numpy as np
        hs = _np(hashes, np.uint8).reshape(-1, 32)
        bl = _np(blocks, np.int32)
        assert len(hs) == len(bl)
        _check(lib().pkv_prefix_cache_insert(self._h, hs.ctypes.data, bl.ctypes.data, len(bl)))

    def release(self, blocks):
        import numpy as np
        bl = _np(blocks, np.int32)
        _check(lib().pkv_prefix_cache_release(self._h, bl.ctypes.data, len(bl)))

    def stats(self) -> dict:
        import numpy as np
        out = np.zeros(4, np.int64)
        _check(lib().pkv_prefix_cache_stats(self._h, out.ctypes.data))
        return dict(free=int(out[0]), cached_free=int(out[1]), in_use=int(out[2]), hashed=int(out[3]))
