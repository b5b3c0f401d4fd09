"""Oracle of the prefix cache: chained block hashes and the block map (TEST INFRASTRUCTURE ONLY).

Written from the notes "vLLM：PagedAttention 与前缀缓存" (sections on chained hashing, lookup and
reuse, reference counts and LRU, boundary conditions) and "PagedAttention 与前缀缓存" (2kiu.com,
section 3.2: hash each block, walk a new prompt block by block and stop at the first miss; mix
model and tokenizer versions into the hash; section 4.3 steps 2-3: attach hit blocks, reference
count + 1).  Shares no code with the library; hashlib's SHA-256 is the hash primitive.
"""
from __future__ import annotations

import collections
import hashlib
from typing import List, Optional, Sequence


def chained_hashes(tokens: Sequence[int], block_size: int, extra: bytes = b"",
                   init: Optional[bytes] = None) -> List[bytes]:
    """hash_i = SHA-256(hash_{i-1} || tokens of full block i as big-endian uint32 || extra), hash_{-1} =
    init or 32 zero bytes.  Only full blocks are hashed: a 100-token prompt with 16-token blocks has
    6 hashes (96 tokens)."""
    prev = bytes(32) if init is None else bytes(init)
    assert len(prev) == 32
    out = []
    for i in range(len(tokens) // block_size):
        blk = tokens[i * block_size:(i + 1) * block_size]
        payload = prev + b"".join(int(t).to_bytes(4, "big") for t in blk) + bytes(extra)
        prev = hashlib.sha256(payload).digest()
        out.append(prev)
    return out


class PrefixCacheModel:
    """Block bookkeeping as the notes describe it.

    * ``free``: blocks with no mapping, handed out in the order they became free;
    * ``lru``: released blocks that keep their mapping (least recently released first);
    * ``map``: hash -> block for every block that holds a published full block;
    * ``ref``: how many requests hold each block."""

    def __init__(self, num_blocks: int):
        self.ref = [0] * num_blocks
        self.hash_of = [None] * num_blocks
        self.map = {}
        self.free = collections.deque(range(num_blocks))
        self.lru = collections.OrderedDict()

    def match(self, hashes: Sequence[bytes]) -> List[int]:
        hit = []
        for h in hashes:
            b = self.map.get(bytes(h))
            if b is None:
                break                      # the first miss ends the hit
            if b in self.lru:
                del self.lru[b]            # a cached-free block is in use again
            self.ref[b] += 1
            hit.append(b)
        return hit

    def allocate(self, n: int) -> List[int]:
        if len(self.free) + len(self.lru) < n:
            raise MemoryError("KV cache block pool exhausted")
        out = []
        for _ in range(n):
            if self.free:
                b = self.free.popleft()
            else:
                b, _ = self.lru.popitem(last=False)   # evict the least recently released
                del self.map[self.hash_of[b]]
                self.hash_of[b] = None
            self.ref[b] = 1
            out.append(b)
        return out

    def insert(self, hashes: Sequence[bytes], blocks: Sequence[int]) -> None:
        for b in blocks:
            if self.ref[b] <= 0:
                raise ValueError(f"block {b} is not held by a request")
        for h, b in zip(hashes, blocks):
            h = bytes(h)
            if self.hash_of[b] == h or h in self.map:
                continue                   # an existing mapping for this prefix wins
            if self.hash_of[b] is not None:
                del self.map[self.hash_of[b]]
            self.map[h] = b
            self.hash_of[b] = h

    def release(self, blocks: Sequence[int]) -> None:
        for b, k in collections.Counter(int(b) for b in blocks).items():
            if self.ref[b] < k:
                raise ValueError(f"release of block {b} more often than requests hold it")
        for b in blocks:
            self.ref[b] -= 1
            if self.ref[b] == 0:
                if self.hash_of[b] is not None:
                    self.lru[b] = True     # most recently released last
                else:
                    self.free.append(b)

    def stats(self) -> dict:
        n = len(self.ref)
        return dict(free=len(self.free), cached_free=len(self.lru), in_use=n - len(self.free) - len(self.lru),
                    hashed=len(self.map))
