// Prefix cache on the host: chained block hashes and the hash -> physical block map with reference
// counts and LRU retention.
//
// What it computes ("vLLM：PagedAttention 与前缀缓存" notes, "链式哈希" / "查找与复用" / "引用计数与 LRU" /
// "边界条件"; "PagedAttention 与前缀缓存", 2kiu.com, sections 3.2 and 4.3 steps 2-3):
//   * every FULL block of a prompt gets hash_i = H(hash_{i-1}, the block's token ids, extra key);
//     the first block chains from a fixed initial value, so hash_i stands for the whole prefix up
//     to and including block i; a partial tail block is never hashed;
//   * lookup walks a prompt's hashes in order and stops at the first one not in the map; every hit
//     block is attached to the request (reference count + 1);
//   * a released block whose count reaches 0 keeps its hash mapping and joins an LRU queue of
//     cached-free blocks; allocation takes never-used (or unhashed) free blocks first and then evicts
//     the least recently released cached block, dropping its mapping.
// H is SHA-256 (FIPS 180-4) over  prev hash (32 bytes) || token ids as big-endian uint32 || extra
// bytes; the initial value is 32 zero bytes unless the caller gives one.  The SHA-256 round
// constants and initial state are derived exactly at start-up from their definition (the first 32
// bits of the fractional parts of the cube roots of the first 64 primes and of the square roots of
// the first 8 primes) with integer roots, not typed in.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <list>
#include <mutex>
#include <string>
#include <unordered_map>
#include <vector>

#include "pkv_internal.h"

namespace {

// ---------------------------------------------------------------- SHA-256 constants from their definition

typedef unsigned __int128 u128;

// floor(x^(1/k)) for k = 2 or 3, by binary search on 128-bit integers (x < 2^105: the root is below
// 2^36 and the search's cubes stay below 2^108)
u128 iroot(u128 x, int k) {
    u128 lo = 0, hi = (u128)1 << 36;
    while (hi - lo > 1) {
        const u128 mid = lo + (hi - lo) / 2;
        u128 p = mid * mid;
        if (k == 3) p *= mid;
        if (p <= x)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

struct ShaConsts {
    uint32_t k[64], h0[8];
    ShaConsts() {
        int primes[64], n = 0;
        for (int c = 2; n < 64; ++c) {
            bool prime = true;
            for (int d = 2; d * d <= c; ++d)
                if (c % d == 0) prime = false;
            if (prime) primes[n++] = c;
        }
        // cbrt(p) * 2^32 = cbrt(p * 2^96); its low 32 bits are the first 32 fractional bits
        for (int i = 0; i < 64; ++i) k[i] = (uint32_t)iroot((u128)primes[i] << 96, 3);
        for (int i = 0; i < 8; ++i) h0[i] = (uint32_t)iroot((u128)primes[i] << 64, 2);
    }
};

const ShaConsts &consts() {
    static const ShaConsts c;
    return c;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

class Sha256 {
  public:
    Sha256() {
        const ShaConsts &c = consts();
        std::memcpy(h_, c.h0, sizeof h_);
    }
    void update(const uint8_t *p, size_t n) {
        len_ += n;
        while (n) {
            const size_t take = std::min(n, (size_t)64 - fill_);
            std::memcpy(buf_ + fill_, p, take);
            fill_ += take;
            p += take;
            n -= take;
            if (fill_ == 64) {
                block(buf_);
                fill_ = 0;
            }
        }
    }
    void final(uint8_t out[32]) {
        const uint64_t bits = (uint64_t)len_ * 8;
        const uint8_t one = 0x80, zero = 0;
        update(&one, 1);
        while (fill_ != 56) update(&zero, 1);
        uint8_t l[8];
        for (int i = 0; i < 8; ++i) l[i] = (uint8_t)(bits >> (56 - 8 * i));
        update(l, 8);
        for (int i = 0; i < 8; ++i)
            for (int j = 0; j < 4; ++j) out[4 * i + j] = (uint8_t)(h_[i] >> (24 - 8 * j));
    }

  private:
    void block(const uint8_t *b) {
        const uint32_t *k = consts().k;
        uint32_t w[64];
        for (int i = 0; i < 16; ++i)
            w[i] = (uint32_t)b[4 * i] << 24 | (uint32_t)b[4 * i + 1] << 16 | (uint32_t)b[4 * i + 2] << 8 | b[4 * i + 3];
        for (int i = 16; i < 64; ++i) {
            const uint32_t s0 = rotr(w[i - 15], 7) ^ rotr(w[i - 15], 18) ^ (w[i - 15] >> 3);
            const uint32_t s1 = rotr(w[i - 2], 17) ^ rotr(w[i - 2], 19) ^ (w[i - 2] >> 10);
            w[i] = w[i - 16] + s0 + w[i - 7] + s1;
        }
        uint32_t a = h_[0], bb = h_[1], c = h_[2], d = h_[3], e = h_[4], f = h_[5], g = h_[6], h = h_[7];
        for (int i = 0; i < 64; ++i) {
            const uint32_t t1 = h + (rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25)) + ((e & f) ^ (~e & g)) + k[i] + w[i];
            const uint32_t t2 = (rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22)) + ((a & bb) ^ (a & c) ^ (bb & c));
            h = g;
            g = f;
            f = e;
            e = d + t1;
            d = c;
            c = bb;
            bb = a;
            a = t1 + t2;
        }
        h_[0] += a;
        h_[1] += bb;
        h_[2] += c;
        h_[3] += d;
        h_[4] += e;
        h_[5] += f;
        h_[6] += g;
        h_[7] += h;
    }
    uint32_t h_[8];
    uint8_t buf_[64];
    size_t fill_ = 0;
    uint64_t len_ = 0;
};

using Hash = std::string; // 32 raw bytes

} // namespace

struct pkv_prefix_cache {
    int64_t num_blocks = 0;
    std::vector<int32_t> ref;        // requests holding each block
    std::vector<Hash> hash_of;       // the block's mapping key ("" when unhashed)
    std::unordered_map<Hash, int32_t> map;
    std::list<int32_t> plain;        // free blocks without a mapping, taken from the front
    std::list<int32_t> lru;          // free blocks that keep their mapping, least recently released first
    std::vector<std::list<int32_t>::iterator> lru_pos;
    std::vector<uint8_t> in_lru;
    std::mutex mu;
};

extern "C" {

int pkv_block_hashes(const int32_t *tokens, int64_t num_tokens, int block_size, const void *extra, int64_t extra_bytes,
                     const uint8_t *init, uint8_t *hashes, int64_t *num_hashes) {
    if (num_tokens < 0 || block_size <= 0 || extra_bytes < 0) return pkv_fail(PKV_EINVAL, "bad size");
    if ((num_tokens > 0 && !tokens) || (extra_bytes > 0 && !extra) || !num_hashes)
        return pkv_fail(PKV_EINVAL, "NULL pointer");
    const int64_t n = num_tokens / block_size; // full blocks only
    if (n > 0 && !hashes) return pkv_fail(PKV_EINVAL, "NULL pointer");
    uint8_t prev[32];
    if (init)
        std::memcpy(prev, init, 32);
    else
        std::memset(prev, 0, 32);
    std::vector<uint8_t> be((size_t)block_size * 4);
    for (int64_t i = 0; i < n; ++i) {
        for (int t = 0; t < block_size; ++t) {
            const uint32_t x = (uint32_t)tokens[i * block_size + t];
            be[4 * t] = (uint8_t)(x >> 24);
            be[4 * t + 1] = (uint8_t)(x >> 16);
            be[4 * t + 2] = (uint8_t)(x >> 8);
            be[4 * t + 3] = (uint8_t)x;
        }
        Sha256 h;
        h.update(prev, 32);
        h.update(be.data(), be.size());
        if (extra_bytes) h.update(static_cast<const uint8_t *>(extra), (size_t)extra_bytes);
        h.final(hashes + 32 * i);
        std::memcpy(prev, hashes + 32 * i, 32);
    }
    *num_hashes = n;
    return PKV_OK;
}

int pkv_prefix_cache_create(int64_t num_blocks, pkv_prefix_cache_t *out) {
    if (num_blocks <= 0 || num_blocks > 0x7FFFFFFF || !out) return pkv_fail(PKV_EINVAL, "bad argument");
    pkv_prefix_cache *pc = new pkv_prefix_cache;
    pc->num_blocks = num_blocks;
    pc->ref.assign((size_t)num_blocks, 0);
    pc->hash_of.assign((size_t)num_blocks, Hash());
    pc->lru_pos.resize((size_t)num_blocks);
    pc->in_lru.assign((size_t)num_blocks, 0);
    for (int64_t b = 0; b < num_blocks; ++b) pc->plain.push_back((int32_t)b);
    *out = pc;
    return PKV_OK;
}

int pkv_prefix_cache_destroy(pkv_prefix_cache_t pc) {
    delete pc;
    return PKV_OK;
}

int pkv_prefix_cache_match(pkv_prefix_cache_t pc, const uint8_t *hashes, int64_t num_hashes, int32_t *blocks,
                           int64_t *num_hit) {
    if (!pc || num_hashes < 0 || !num_hit || (num_hashes > 0 && (!hashes || !blocks)))
        return pkv_fail(PKV_EINVAL, "bad argument");
    std::lock_guard<std::mutex> lk(pc->mu);
    int64_t i = 0;
    for (; i < num_hashes; ++i) {
        auto it = pc->map.find(Hash(reinterpret_cast<const char *>(hashes + 32 * i), 32));
        if (it == pc->map.end()) break; // the first miss ends the hit
        const int32_t b = it->second;
        if (pc->in_lru[b]) {
            pc->lru.erase(pc->lru_pos[b]);
            pc->in_lru[b] = 0;
        }
        pc->ref[b] += 1;
        blocks[i] = b;
    }
    *num_hit = i;
    return PKV_OK;
}

int pkv_prefix_cache_allocate(pkv_prefix_cache_t pc, int64_t n, int32_t *blocks) {
    if (!pc || n < 0 || (n > 0 && !blocks)) return pkv_fail(PKV_EINVAL, "bad argument");
    std::lock_guard<std::mutex> lk(pc->mu);
    if ((int64_t)(pc->plain.size() + pc->lru.size()) < n) return pkv_fail(PKV_ENOMEM, "KV cache block pool exhausted");
    for (int64_t i = 0; i < n; ++i) {
        int32_t b;
        if (!pc->plain.empty()) {
            b = pc->plain.front();
            pc->plain.pop_front();
        } else {
            // evict the least recently released cached block: its mapping goes with it
            b = pc->lru.front();
            pc->lru.pop_front();
            pc->in_lru[b] = 0;
            pc->map.erase(pc->hash_of[b]);
            pc->hash_of[b].clear();
        }
        pc->ref[b] = 1;
        blocks[i] = b;
    }
    return PKV_OK;
}

int pkv_prefix_cache_insert(pkv_prefix_cache_t pc, const uint8_t *hashes, const int32_t *blocks, int64_t n) {
    if (!pc || n < 0 || (n > 0 && (!hashes || !blocks))) return pkv_fail(PKV_EINVAL, "bad argument");
    std::lock_guard<std::mutex> lk(pc->mu);
    for (int64_t i = 0; i < n; ++i) {
        const int32_t b = blocks[i];
        if (b < 0 || b >= pc->num_blocks || pc->ref[b] <= 0)
            return pkv_fail(PKV_EINVAL, "block %d is not held by a request", (int)b);
    }
    for (int64_t i = 0; i < n; ++i) {
        const int32_t b = blocks[i];
        Hash h(reinterpret_cast<const char *>(hashes + 32 * i), 32);
        if (pc->hash_of[b] == h) continue;
        if (pc->map.count(h)) continue; // the prefix is cached in another block already: keep that one
        if (!pc->hash_of[b].empty()) pc->map.erase(pc->hash_of[b]);
        pc->map[h] = b;
        pc->hash_of[b] = h;
    }
    return PKV_OK;
}

int pkv_prefix_cache_release(pkv_prefix_cache_t pc, const int32_t *blocks, int64_t n) {
    if (!pc || n < 0 || (n > 0 && !blocks)) return pkv_fail(PKV_EINVAL, "bad argument");
    std::lock_guard<std::mutex> lk(pc->mu);
    std::unordered_map<int32_t, int32_t> times; // a block may appear more than once in one call
    for (int64_t i = 0; i < n; ++i) {
        const int32_t b = blocks[i];
        if (b < 0 || b >= pc->num_blocks || pc->ref[b] < ++times[b])
            return pkv_fail(PKV_EINVAL, "release of block %d more often than requests hold it", (int)b);
    }
    for (int64_t i = 0; i < n; ++i) {
        const int32_t b = blocks[i];
        if (--pc->ref[b] > 0) continue;
        if (!pc->hash_of[b].empty()) {
            pc->lru_pos[b] = pc->lru.insert(pc->lru.end(), b);
            pc->in_lru[b] = 1;
        } else {
            pc->plain.push_back(b);
        }
    }
    return PKV_OK;
}

int pkv_prefix_cache_stats(pkv_prefix_cache_t pc, int64_t out[4]) {
    if (!pc || !out) return pkv_fail(PKV_EINVAL, "NULL argument");
    std::lock_guard<std::mutex> lk(pc->mu);
    out[0] = (int64_t)pc->plain.size();
    out[1] = (int64_t)pc->lru.size();
    out[2] = pc->num_blocks - out[0] - out[1];
    out[3] = (int64_t)pc->map.size();
    return PKV_OK;
}

} // extern "C"
