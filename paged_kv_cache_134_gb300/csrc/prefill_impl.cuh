// Causal attention over packed or paged keys on the 5th-generation tensor cores: the packed prefill
// (with the paged K/V write fused in), the prefill over a cached prefix, and the prefix phase of the
// cascade decode.
//
// What it computes ("Paged KV Cache 与 Packed Sequence", discosf.com, sections 3.1-3.3, 4.2):
// sequences packed back to back, sequence i owning rows [cu[i], cu[i+1]); a query at in-sequence
// position r attends to the keys of its own sequence at positions c <= r (block-diagonal causal
// mask), out = softmax(scale q.k) v.  In packed mode every token's k/v is also written into the paged
// cache at block_table[i][r / bs], offset r % bs (the prompt-phase write of section 4.2, bounded by
// the sequence length so a partly filled tail block is never overrun).  In paged mode sequence i
// already holds ctx[i] tokens in its blocks ("PagedAttention 与前缀缓存", 2kiu.com, section 4.3): its
// rows sit at positions ctx[i] + r and every key is read from the pool through the block table.  In
// cascade mode the queries are the decode queries of a batch (one row per sequence) and the keys are
// a prefix shared by every table (section 3.3), cut into splits whose fp32 partials a merge combines.
//
// Design (one persistent CTA per SM, items taken from an atomic counter, heaviest first):
//  * An item is two 128-row query tiles A and B.  Packed and paged modes: consecutive tiles of one
//    (sequence, query head), which share every 128-key K/V tile (loaded once, used by both); cascade
//    mode: one tile of 128 sequences against two consecutive prefix splits (one Q tile, two key streams).
//  * Tensor memory (512 columns): S_A, S_B (128 fp32 columns each) and O_A, O_B (D columns each).  P
//    is written over S in place (fp16, or a bf16 hi + lo pair), and read by P V as the A operand from
//    tensor memory.
//  * Each tile has its own MMA-issuing warp, which issues per key step j: P V(j), then S(j+1).  While
//    one tile's softmax runs, the tensor pipe works on the other tile's products, so each softmax has
//    two MMAs' time (2 x 128 x 128 x D) to finish; S(j+1) of a tile is issued only after its P V(j),
//    which frees the S columns P occupies (tcgen05 operations of one thread complete in issue order).
//    Two issuing warps keep the pipe's queue fed while either waits for its softmax.
//  * Warp roles: 0 scheduler, Q loads and K loads; 2 V loads (each loader also writes the packed
//    mode's paged K/V rows, and widens the E4M3 tiles of FP8 caches); 1 and 3 the MMA issuers of tiles
//    A and B (warp 1 also owns tensor memory); 4-7 softmax of tile A, 8-11 softmax of tile B (one
//    thread per query row, tensor memory lane = row).
//  * O is rescaled in tensor memory only when a row's running maximum grows by more than 2^8 (the
//    exponent base stays fixed otherwise, which is exact algebra); the softmax thread does it, since
//    S(j) complete implies P V(j-1) complete.
//  * Item boundaries: the K loader issues the next item's first K tile, then its Q tiles as their
//    buffers free up; a tile's output (a whole tile of the sequence's rows) is staged in its own Q
//    buffer and written by TMA stores, and the Q buffer returns to the loader once they have read it.
//  * Every mbarrier wait is bounded; a timeout sets PKV_DEVERR_TIMEOUT and the CTA winds down.
#pragma once

#include <cuda.h>

#include "tcgen05.cuh"
#include "pkv_internal.h"

namespace pkv_prefill {

constexpr int BM = 128;          // query rows per tile (MMA M)
constexpr int BN = 128;          // keys per tile (MMA N of Q K^T, K of P V)
constexpr int kThreads = 384;    // 12 warps
constexpr uint32_t kTmemCols = 512;
constexpr float kRescale = 8.0f; // log2 units
constexpr int kCodeOff = 16384;  // E4M3 codes of a stage: row r at stage + kCodeOff + r * D

enum { MODE_PACKED = 0, MODE_PAGED = 1, MODE_CASCADE = 2 };

struct Args {
    const char *k, *v;  // packed [T][Hkv][D] (packed mode)
    void *out;          // packed [T][Hq][D]
    const int32_t *cu, *tables;
    char *pool;
    const float *k_scale, *v_scale; // FP8 caches: per KV head
    unsigned int *err;
    int *plan;          // [0] pair count, [1] next-item counter, [4 + 2i], [5 + 2i] = (sequence, pair) of list entry i
    const int32_t *ctx; // paged mode: tokens each sequence already holds in its blocks
    int64_t total_tokens, num_blocks, tile_elems;
    int num_seqs, max_seqlen, max_blocks, hq, hkv, bs, lg_bs, npairs_max, cost_bins;
    int64_t plan_cap;   // list entries the work list has room for
    int write_pool;     // packed mode: write K/V into the pool (16-bit caches; FP8 caches are written by the append)
    float scale_log2;
    // cascade mode: the decode queries of num_seqs sequences against a shared prefix of prefix_tokens
    // tokens (table row 0), cut into nps splits of split_tokens keys; each (sequence, query head, split)
    // leaves an fp32 partial (m, l, unnormalised o) in workspace slot split
    float *ws_o = nullptr, *ws_ml = nullptr;
    int max_splits = 0, prefix_tokens = 0, split_tokens = 0, nps = 0;
};

// TMA descriptors of one launch: q (and out) as [rows][Hq * D] with 64-column boxes of BM rows; packed
// k and v as [T][Hkv * D] with boxes of BN rows; the pool's rows (16-bit: bs rows x 64 dims; E4M3: bs
// whole rows)
struct Maps {
    CUtensorMap q, k, v, pool, out;
};

// Shared memory: two Q tiles, the K ring and the V ring.  A 16-bit tile is [D/64 halves][rows][128 B],
// 128-byte swizzled.  FP8 caches: the codes of a K or V tile land at stage + kCodeOff (row r at r * D)
// and are widened into the 16-bit layout of the same stage: for D = 128 the codes are the upper half
// of the stage, which each row's widening thread reads whole before it writes it; for D = 64 they
// follow the 16 KB tile.
template <int D, bool KV8>
struct Layout {
    static constexpr int NKS = D == 128 ? 3 : 4; // K stages (a K stage frees once S of both tiles is done)
    static constexpr int NVS = D == 128 ? 2 : 3; // V stages (a V stage frees after P V of both tiles)
    static constexpr int Q_TILE = BM * D * 2;
    static constexpr int TILE = BN * D * 2;
    static constexpr int STAGE = (KV8 && D == 64) ? TILE + BN * D : TILE;
    static constexpr int Q = 0;
    static constexpr int K0 = Q + 2 * Q_TILE;
    static constexpr int V0 = K0 + NKS * STAGE;
    static constexpr int BAR = V0 + NVS * STAGE;
    static constexpr int NBARS = 4 + 4 + 2 + 2 + 4 * NKS + 4 * NVS + 2 + 2 + 2 + 2 + 2 + 2;
    static constexpr int MISC = BAR + (NBARS * 8 + 15) / 16 * 16; // TMEM slot, abort flag; item slots at + 16
    static constexpr int TOTAL = MISC + 16 + 64;
    static_assert(TOTAL + 1024 <= 232448, "shared memory");
    static_assert(!KV8 || D == 64 || kCodeOff + BN * D <= STAGE, "code region");
};

// two floats -> packed fp16/bf16 pair (round-to-nearest-even), `lo` in the low half
PKV_DEV uint32_t pack2(float lo, float hi, int mt) {
    uint32_t r;
    if (mt == PKV_BF16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// two E4M3 codes (lo in bits 0-7) -> the model dtype's pair; exact (every E4M3 value is an fp16 and
// a bf16 value)
template <int MT>
PKV_DEV uint32_t widen2(uint32_t codes) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(codes)));
    if constexpr (MT == PKV_F16) {
        return h2;
    } else {
        const float lo = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xFFFFu)));
        const float hi = __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16)));
        return pack2(lo, hi, PKV_BF16);
    }
}

// Widen row r of an E4M3 tile (D codes at stage + kCodeOff + r * D) into the 128-byte-swizzled
// 16-bit layout of the same stage.  The whole code row is read before anything is written.
template <int D, int MT>
PKV_DEV void widen_row(uint8_t *stage, int r) {
    constexpr int NC = D / 16; // 16-byte chunks of codes
    uint4 c[NC];
#pragma unroll
    for (int i = 0; i < NC; ++i) c[i] = *reinterpret_cast<const uint4 *>(stage + kCodeOff + r * D + i * 16);
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        const uint32_t w[4] = {c[i].x, c[i].y, c[i].z, c[i].w};
        uint32_t o[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            o[2 * e] = widen2<MT>(w[e] & 0xFFFFu);
            o[2 * e + 1] = widen2<MT>(w[e] >> 16);
        }
        // codes 16 i .. 16 i + 15 = dims of two 8-element chunks u0 = 2 i, u0 + 1 (half = dims / 64)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int u = 2 * i + h, c2 = u >> 3, uu = u & 7;
            *reinterpret_cast<uint4 *>(stage + c2 * BN * 128 + r * 128 + ((uu ^ (r & 7)) << 4)) =
                make_uint4(o[4 * h], o[4 * h + 1], o[4 * h + 2], o[4 * h + 3]);
        }
    }
}

// query tiles of sequence i (0 for a malformed cu_seqlens entry or context length, which is reported)
PKV_DEV int seq_tiles(const Args &a, int i, bool report) {
    const int st = a.cu[i], en = a.cu[i + 1];
    if (st < 0 || en < st || en > a.total_tokens || en - st > a.max_seqlen) {
        if (report) set_error(a.err, PKV_DEVERR_CU_SEQLENS);
        return 0;
    }
    if (a.ctx) {
        // paged mode: the cached tokens plus the new ones must fit the sequence's table
        const int64_t c0 = a.ctx[i];
        if (c0 < 0 || c0 + (en - st) > (int64_t)a.max_blocks * a.bs) {
            if (report) set_error(a.err, PKV_DEVERR_LENGTH);
            return 0;
        }
    }
    return (en - st + BM - 1) / BM;
}

// one tile of an item as the roles see it
struct Tile {
    int n;     // key tiles (0: the tile is absent)
    int q0;    // first query row of the tile (in-sequence row; cascade: 0)
    int qlast; // last valid query row
    int qpos0; // absolute position of the tile's row 0 (causal mask)
    int k0;    // absolute position of the first key
    int kend;  // keys at or past kend hold no token of the sequence (or of the prefix split)
};

struct Item {
    int seq, pr, h; // seq < 0: no more items.  Cascade: seq = tile of 128 sequences, pr = split pair
    int start;      // packed row of the sequence's first token (cascade: first sequence of the tile)
    int n;          // rows of the sequence (cascade: sequences in the tile)
    int trow;       // block-table row of the keys
    Tile t[2];
};

PKV_DEV Item decode_item(const Args &a, int seq, int pr, int h) {
    Item it;
    it.seq = seq;
    it.pr = pr;
    it.h = h;
    if (seq < 0) return it;
    if (a.nps > 0) {
        it.start = seq * BM;
        it.n = min(BM, a.num_seqs - it.start);
        it.trow = 0;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
            const int sp = 2 * pr + t;
            Tile &x = it.t[t];
            x.q0 = 0;
            x.qlast = it.n - 1;
            x.qpos0 = 0;
            x.k0 = sp * a.split_tokens;
            x.kend = min(x.k0 + a.split_tokens, a.prefix_tokens);
            x.n = sp < a.nps ? (x.kend - x.k0 + BN - 1) / BN : 0;
        }
        return it;
    }
    it.start = a.cu[seq];
    it.n = a.cu[seq + 1] - it.start;
    it.trow = seq;
    const int c0 = a.ctx ? a.ctx[seq] : 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        Tile &x = it.t[t];
        x.q0 = (2 * pr + t) * BM;
        x.qlast = min(x.q0 + BM, it.n) - 1;
        x.qpos0 = c0 + x.q0;
        x.k0 = 0;
        x.kend = c0 + it.n;
        x.n = x.q0 < it.n ? (c0 + x.qlast) / BN + 1 : 0; // key tiles up to the tile's last row
    }
    return it;
}

// K (or V) ring index of key step j of tile t, counted from the item's first tile.  Packed and paged
// modes share one key tile per step; cascade mode has one per tile and step.
template <bool SHARED>
PKV_DEV int ring_index(const Item &it, int j, int t) {
    if constexpr (SHARED) {
        return j;
    } else {
        const int mn = min(it.t[0].n, it.t[1].n);
        const int before = 2 * min(j, mn) + max(0, j - mn);
        return before + ((t == 1 && j < it.t[0].n) ? 1 : 0);
    }
}
template <bool SHARED>
PKV_DEV int ring_count(const Item &it) {
    return SHARED ? max(it.t[0].n, it.t[1].n) : it.t[0].n + it.t[1].n;
}
// the tile (0 or 1) that ring entry e of the item belongs to, and its key step
template <bool SHARED>
PKV_DEV void ring_entry(const Item &it, int e, int &t, int &j) {
    if constexpr (SHARED) {
        t = 0;
        j = e;
    } else {
        const int mn = min(it.t[0].n, it.t[1].n);
        if (e < 2 * mn) {
            t = e & 1;
            j = e >> 1;
        } else {
            t = it.t[0].n > mn ? 0 : 1;
            j = mn + (e - 2 * mn);
        }
    }
}

template <int D, int MT, int MODE, bool KV8>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ Maps maps, const Args a) {
    const CUtensorMap &tq = maps.q, &tk = maps.k, &tv = maps.v, &tp = maps.pool, &to = maps.out;
    using L = Layout<D, KV8>;
    constexpr bool PAGED = MODE != MODE_PACKED;    // keys from the pool through the block table
    constexpr bool CASCADE = MODE == MODE_CASCADE; // no causal mask, fp32 split partials out
    constexpr bool SHARED = !CASCADE;              // both tiles use the same key tiles
    constexpr bool WRITER = MODE == MODE_PACKED;   // the loaders write the item's K/V rows into the pool
    constexpr int NP = MT == PKV_BF16 ? 2 : 1;     // P parts (bf16: hi + lo)
    constexpr int EB = KV8 ? 1 : 2;                // pool bytes per element
    constexpr int NKS = L::NKS, NVS = L::NVS;
    extern __shared__ __align__(1024) uint8_t smem[];

    pdl_trigger();
    if (smem_u32(smem) & 1023u) return; // the swizzled tiles need 1024-byte alignment (always true)

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR);
    // items go through a 4-slot ring: the scheduler publishes an item while the one before it is
    // still being loaded, so that nobody waits for the next item at an item boundary
    constexpr int kItemSlots = 4;
    uint64_t *item_full = bars, *item_empty = bars + kItemSlots;
    uint64_t *q_full = bars + 2 * kItemSlots, *q_empty = q_full + 2;
    uint64_t *k_full = q_empty + 2, *k_empty = k_full + NKS, *kc_full = k_empty + NKS, *k_spare = kc_full + NKS;
    uint64_t *v_full = k_spare + NKS, *v_empty = v_full + NVS, *vc_full = v_empty + NVS, *v_spare = vc_full + NVS;
    uint64_t *s_full = v_spare + NVS, *p_full = s_full + 2, *o_full = p_full + 2, *o_free = o_full + 2;
    uint64_t *fin = o_free + 2;
    uint64_t *epi = fin + 2; // a tile's output rows are staged (one arrival per softmax warp)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::MISC + 4);
    // exp phases the softmax of each tile has finished, counted per warp (4 per key step), monotonic
    int *sm_prog = reinterpret_cast<int *>(smem + L::MISC + 8); // [2]
    volatile int4 *item_slot = reinterpret_cast<volatile int4 *>(smem + L::MISC + 16); // [kItemSlots]
    (void)k_spare;
    (void)v_spare;
    // K / V tiles ready for the MMA: landed (16-bit) or landed and widened (E4M3)
    uint64_t *k_ready = KV8 ? kc_full : k_full;
    uint64_t *v_ready = KV8 ? vc_full : v_full;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // item consumers: V loader, the two MMA issuers, eight softmax warps
    constexpr int kItemConsumers = 11;
    // a K or V stage frees once every MMA warp whose tile reads it has released it (both tiles read
    // the shared key tiles of packed and paged modes; each cascade tile has key tiles of its own)
    constexpr int kStageReleasers = SHARED ? 2 : 1;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kItemSlots; ++s) {
            mbar_init(item_full + s, 1);
            mbar_init(item_empty + s, kItemConsumers);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(q_full + s, 1);
            mbar_init(q_empty + s, CASCADE ? 2 : 1); // cascade: one Q tile, read by both MMA warps
            mbar_init(s_full + s, 1);
            mbar_init(p_full + s, 4); // one arrival per softmax warp
            mbar_init(o_full + s, 1);
            mbar_init(o_free + s, 4);
        }
        for (int s = 0; s < NKS; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(k_empty + s, kStageReleasers);
            mbar_init(kc_full + s, 1);
        }
        for (int s = 0; s < NVS; ++s) {
            mbar_init(v_full + s, 1);
            mbar_init(v_empty + s, kStageReleasers);
            mbar_init(vc_full + s, 1);
        }
        mbar_init(fin, 1);
        mbar_init(fin + 1, 1);
        mbar_init(epi, 4);
        mbar_init(epi + 1, 4);
        *abort_flag = 0;
        sm_prog[0] = 0;
        sm_prog[1] = 0;
        fence_mbarrier_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    // everything above is private to this CTA; from here on global memory written by the previous
    // kernels on the stream (the work list, the inputs) is read.  Cascade mode runs right after the
    // suffix decode, which lets it launch once the decode itself has waited for its predecessors (the
    // plan of this call and everything before it): the prefix phase reads nothing the decode writes,
    // so it starts at once and fills the SMs the decode's CTAs leave, and waits for the decode only
    // before it exits (the merge after it then sees both).
    if constexpr (!CASCADE) pdl_wait();

    const int G = a.hq / a.hkv;
    auto fail = [&]() {
        set_error(a.err, PKV_DEVERR_TIMEOUT);
        *abort_flag = 1;
    };
    // the item in ring slot n % 4, once the scheduler has published it
    auto take_item = [&](int n, bool &ok) -> Item {
        const int sl = n & (kItemSlots - 1);
        ok = mbar_wait_hint(item_full + sl, (n / kItemSlots) & 1);
        if (!ok) return decode_item(a, -1, 0, 0);
        return decode_item(a, item_slot[sl].x, item_slot[sl].y, item_slot[sl].z);
    };
    // the item's keys of ring entry e: key step j of tile t (packed / paged: one tile serves both)
    // (tiles are selected, not indexed, so that the item stays in registers)
    auto key_base = [&](const Item &it, int e, int &t, int &j) -> int {
        ring_entry<SHARED>(it, e, t, j);
        return (t ? it.t[1].k0 : it.t[0].k0) + j * BN;
    };
    auto key_end = [&](const Item &it, int t) -> int {
        return (SHARED || t == 0) ? it.t[0].kend : it.t[1].kend;
    };

    if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 104;");
    if (warp == 0 || warp == 2) {
        // ---------------------------------------------------------------- loaders
        // Warp 0: the scheduler (lane 0), Q loads and K loads; warp 2: V loads.  Packed mode: lane 0
        // loads each tile (one box per half of D).  Paged and cascade modes: lane l loads block l of
        // each tile; blocks full of the keys' tokens arrive as TMA boxes, and every other row of a V
        // tile is written with plain stores: the tokens of a partly filled last block copied from the
        // pool, zeros for slots past the keys' end and for unusable block ids (P is 0 on those rows,
        // but 0 * NaN is NaN, and the pool's unused slots may hold anything); K rows past the end are
        // masked by the softmax instead.  FP8 caches: the codes land in the stage's code region, and
        // the loader widens each tile once it has landed, before it issues the next one.  Packed mode:
        // the paged write of an item's own rows (the keys of its last tiles) leaves a stage just before
        // the loader refills it (whole blocks as tiled TMA stores, one lane per block and half of D;
        // the rows of a partly filled last block as plain 16-byte stores, so no slot past the sequence
        // is touched), or at the end.
        const bool isK = warp == 0;
        constexpr int NS = 0; // (stage counts differ per ring; see ns below)
        (void)NS;
        const int ns = isK ? NKS : NVS;
        uint8_t *const ring = smem + (isK ? L::K0 : L::V0);
        uint64_t *const full = isK ? k_full : v_full;
        uint64_t *const empty = isK ? k_empty : v_empty;
        uint64_t *const ready = isK ? kc_full : vc_full; // E4M3: widened
        const int kvsel = isK ? 0 : 1;                   // K or V half of a pool block
        constexpr int CPR = D * EB / 16;                  // 16-byte chunks per pool row
        constexpr int RPI = 32 / CPR;                     // rows per warp instruction (never two blocks: bs >= 8)
        const int cc = lane % CPR, rsub = lane / CPR;
        if (lane == 0) {
            if (isK) tc::prefetch_tmap(&tq);
            tc::prefetch_tmap(PAGED ? &tp : (isK ? &tk : &tv));
        }
        // packed mode: the pending pool write of the entry each stage holds (j < 0: none), with the
        // item's rows and (lane l) the table entry of its logical block lb0 + l
        int wj[4] = {-1, -1, -1, -1}, wq0[4] = {}, wql[4] = {}, wkvh[4] = {}, wblk[4] = {}, wpar[4] = {};
        auto flush_write = [&](int st) {
            if constexpr (WRITER) {
                if (wj[st] < 0) return;
                const uint8_t *src = ring + st * L::STAGE;
                // the tile has landed long ago (it was loaded ns entries back); the wait is for the
                // rare case the loader is about to refill a stage whose tile still flies
                mbar_wait_hint(full + st, (uint32_t)wpar[st]);
                const int j = wj[st], q0 = wq0[st], qlast = wql[st], kvh = wkvh[st], blkv = wblk[st];
                const int lb0 = q0 >> a.lg_bs;
                const int lo = max(j * BN, q0), hi = min(j * BN + BN - 1, qlast);
                if (lo <= hi) {
                    const int bfirst = lo >> a.lg_bs;           // lo is a multiple of bs
                    const int nfull = (hi + 1 - lo) >> a.lg_bs; // whole blocks among the rows
                    {
                        const int lb = bfirst + lane;
                        const int blk = __shfl_sync(0xffffffffu, blkv, min(lb - lb0, 31));
                        if (lane < nfull) {
                            if (blk < 0 || blk >= a.num_blocks) {
                                set_error(a.err, PKV_DEVERR_BLOCK_ID);
                            } else {
                                const uint8_t *box = src + ((lb << a.lg_bs) - j * BN) * 128;
                                const int y = ((blk * 2 + kvsel) * a.hkv + kvh) << a.lg_bs;
#pragma unroll
                                for (int c = 0; c < D / 64; ++c) tc::tma_store_2d(&tp, c * 64, y, box + c * BN * 128);
                                tc::bulk_commit();
                            }
                        }
                    }
                    const int c2 = cc >> 3, u = cc & 7;
                    for (int p0 = lo + (nfull << a.lg_bs); p0 <= hi; p0 += RPI) { // fewer than bs rows
                        const int pp = p0 + rsub;
                        const int lb = pp >> a.lg_bs;
                        const int blk = __shfl_sync(0xffffffffu, blkv, min(lb - lb0, 31));
                        if (pp > hi) continue;
                        if (blk < 0 || blk >= a.num_blocks) {
                            if (cc == 0) set_error(a.err, PKV_DEVERR_BLOCK_ID);
                            continue;
                        }
                        const int rr = pp - j * BN;
                        const uint4 xv = *reinterpret_cast<const uint4 *>(src + c2 * BN * 128 + rr * 128 +
                                                                          ((u ^ (rr & 7)) << 4));
                        const int64_t dst = ((int64_t)(blk * 2 + kvsel) * a.hkv + kvh) * a.tile_elems +
                                            (int64_t)(pp - (lb << a.lg_bs)) * D + cc * 8;
                        *reinterpret_cast<uint4 *>(a.pool + dst * 2) = xv;
                    }
                }
                tc::bulk_wait_read_all(); // the stores have read the stage; it may be refilled
                __syncwarp();
                wj[st] = -1;
            }
        };
        // FP8: widen ring entry gw (landed), then release it to the MMAs
        auto widen = [&](int64_t gw) -> bool {
            const int st = (int)(gw % ns);
            if (!__all_sync(0xffffffffu, mbar_wait_hint(full + st, (uint32_t)((gw / ns) & 1)))) return false;
            uint8_t *stage = ring + st * L::STAGE;
            for (int r = lane; r < BN; r += 32) widen_row<D, MT>(stage, r);
            fence_proxy_async_smem(); // the MMAs read the widened tile through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(ready + st);
            return true;
        };
        const int total = a.plan[0] * a.hq;
        int64_t g = 0;      // tiles issued so far (all items)
        int nq[2] = {0, 0}; // Q loads per buffer so far (warp 0)
        int64_t pend = -1;  // FP8: the issued tile still to widen
        // FP8: widen the pending tile; done before this warp can block on anything an MMA of that tile
        // may be holding up (the next tile's stage, the next item, the next item's Q buffer)
        auto widen_pending = [&]() -> bool {
            if constexpr (KV8) {
                if (pend >= 0) {
                    const bool w = widen(pend);
                    pend = -1;
                    return w;
                }
            }
            return true;
        };
        bool ok = true;
        // the scheduler (warp 0): take item m from the work list and publish it in ring slot m % 4
        auto publish = [&](int m, bool &pok) -> Item {
            const int sl = m & (kItemSlots - 1);
            pok = true;
            if (m >= kItemSlots) pok = __all_sync(0xffffffffu, mbar_wait_hint(item_empty + sl, ((m / kItemSlots) - 1) & 1));
            int4 raw = make_int4(-1, 0, 0, 0);
            if (!pok) return decode_item(a, -1, 0, 0);
            if (lane == 0) {
                const int idx = *abort_flag ? total : atomicAdd(a.plan + 1, 1);
                if (idx < total) {
                    if constexpr (CASCADE) {
                        const int pair = idx / a.hq; // (tile of sequences, split pair)
                        const int npr = (a.nps + 1) / 2;
                        raw = make_int4(pair / npr, pair % npr, idx % a.hq, 0);
                    } else {
                        const int2 sq = reinterpret_cast<const int2 *>(a.plan + 4)[idx / a.hq];
                        raw = make_int4(sq.x, sq.y, idx % a.hq, 0);
                    }
                }
                item_slot[sl].x = raw.x;
                item_slot[sl].y = raw.y;
                item_slot[sl].z = raw.z;
                mbar_arrive(item_full + sl);
            }
            raw.x = __shfl_sync(0xffffffffu, raw.x, 0);
            raw.y = __shfl_sync(0xffffffffu, raw.y, 0);
            raw.z = __shfl_sync(0xffffffffu, raw.z, 0);
            return decode_item(a, raw.x, raw.y, raw.z);
        };
        for (int n = 0; ok; ++n) {
            Item it;
            if (!isK && !widen_pending()) ok = false; // before waiting for the next item
            if (!ok) break;
            if (isK) {
                // ---- scheduler: take the next item and publish it (once the previous item's last K
                // tile is issued, a few key steps before that item ends)
                it = publish(n, ok);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                if (n > 0 && it.seq >= 0 && lane == 0) {
                    // the item's Q tiles load only once the previous item's last S of each tile is done:
                    // staged in L2 now, they then arrive from L2
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        if (CASCADE ? b == 1 : it.t[b].n == 0) continue;
#pragma unroll
                        for (int c = 0; c < D / 64; ++c) tc::tma_prefetch_2d(&tq, it.h * D + c * 64, it.start + it.t[b].q0);
                    }
                }
            } else {
                it = take_item(n, ok);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
            }
            if (it.seq < 0) break;
            const int kvh = it.h / G;
            if (isK && !widen_pending()) ok = false; // before the Q loads wait for their buffers
            if (!ok) {
                if (lane == 0) fail();
                break;
            }
            // ---- Q (warp 0): buffer b holds tile b (cascade: buffer 0 holds the one query tile of both
            // splits).  Each load waits for the previous item's last S of that tile, so the loads are
            // interleaved with the K tiles in the order their buffers free up: K tile 0 (its stage frees
            // a few key steps before the previous item ends), Q_A, K tile 1, Q_B, the rest.  The first S
            // of each tile then finds both operands in place.
            // query row of each buffer's tile, -1: nothing to load
            const int qrow0 = it.t[0].n > 0 ? it.start + it.t[0].q0 : -1;
            const int qrow1 = !CASCADE && it.t[1].n > 0 ? it.start + it.t[1].q0 : -1;
            const int qcol = it.h * D;
            int qnext = 0; // next Q buffer to load
            auto issue_q = [&](int upto) {
                for (; qnext <= upto && qnext < 2 && ok; ++qnext) {
                    const int b = qnext;
                    const int row = b ? qrow1 : qrow0;
                    if (row < 0) continue;
                    if (lane == 0) {
                        const bool w = nq[b] < 1 || mbar_wait_hint(q_empty + b, (nq[b] - 1) & 1);
                        if (w) {
                            mbar_arrive_expect_tx(q_full + b, L::Q_TILE);
#pragma unroll
                            for (int c = 0; c < D / 64; ++c)
                                tc::tma_load_2d(smem + L::Q + b * L::Q_TILE + c * BM * 128, &tq, qcol + c * 64, row,
                                                q_full + b);
                        } else {
                            fail();
                        }
                        ok = w;
                    }
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    ++nq[b];
                }
            };
            const int ne = ring_count<SHARED>(it);
            // packed mode: this item writes the K/V of its own rows (the first query head of each KV
            // group does), from the key tiles that hold them
            const int q0 = it.t[0].q0, qlast = it.t[1].n > 0 ? it.t[1].qlast : it.t[0].qlast;
            const bool writes = WRITER && a.write_pool && it.h % G == 0;
            int blkv = -1;
            if (writes) {
                const int lb = (q0 >> a.lg_bs) + lane;
                if ((lb << a.lg_bs) <= qlast && lb < a.max_blocks) blkv = a.tables[(int64_t)it.seq * a.max_blocks + lb];
            }
            // paged / cascade: lane l's table entry of block l of ring entry e (-1: no token there)
            auto entry = [&](int e) -> int {
                int t, j;
                const int kb = key_base(it, e, t, j);
                const int lb = (kb >> a.lg_bs) + lane;
                return (lane < (BN >> a.lg_bs) && (lb << a.lg_bs) < key_end(it, t))
                           ? a.tables[(int64_t)it.trow * a.max_blocks + lb]
                           : -1;
            };
            int nxt = PAGED && ne > 0 ? entry(0) : -1;
            int issued = 0;
            for (int e = 0; e < ne && ok; ++e) {
                const int64_t gg = g + e;
                const int st = (int)(gg % ns);
                const int64_t round = gg / ns;
                // FP8: the previous tile is widened first (an MMA waits for it), then this one loads
                if (!widen_pending()) ok = false;
                flush_write(st); // the stage's previous tile leaves for the pool before the refill
                if (ok && round >= 1) ok = __all_sync(0xffffffffu, mbar_wait_hint(empty + st, (round - 1) & 1));
                if (!ok || __any_sync(0xffffffffu, *abort_flag != 0)) break;
                uint8_t *stage = ring + st * L::STAGE;
                if constexpr (PAGED) {
                    int t, j;
                    const int kbase = key_base(it, e, t, j), send = key_end(it, t);
                    const int nbt = BN >> a.lg_bs;
                    int b = nxt;
                    if (e + 1 < ne) nxt = entry(e + 1);
                    const int lb = (kbase >> a.lg_bs) + lane;
                    const bool has = lane < nbt && (lb << a.lg_bs) < send;
                    const bool good = has && b >= 0 && b < a.num_blocks;
                    if (!isK && has && !good) set_error(a.err, PKV_DEVERR_BLOCK_ID);
                    // K: every usable block whole (rows past the end are masked); V: only full blocks
                    const bool full_blk = good && (isK || ((lb + 1) << a.lg_bs) <= send);
                    const unsigned fullmask = __ballot_sync(0xffffffffu, full_blk);
                    if (lane == 0) mbar_expect_tx(full + st, (uint32_t)__popc(fullmask) * (uint32_t)(a.bs * D * EB));
                    __syncwarp();
                    if (full_blk) {
                        const int y = ((b * 2 + kvsel) * a.hkv + kvh) << a.lg_bs;
                        if constexpr (KV8) {
                            tc::tma_load_2d(stage + kCodeOff + (lane << a.lg_bs) * D, &tp, 0, y, full + st);
                        } else {
#pragma unroll
                            for (int c = 0; c < D / 64; ++c)
                                tc::tma_load_2d(stage + c * BN * 128 + ((lane << a.lg_bs) * 128), &tp, c * 64, y,
                                                full + st);
                        }
                    }
                    const unsigned allmask = nbt == 32 ? 0xffffffffu : (1u << nbt) - 1u;
                    if (!isK) {
                        for (int r0 = 0; fullmask != allmask && r0 < BN; r0 += RPI) {
                            const int r = r0 + rsub, l = r >> a.lg_bs;
                            const int bl = __shfl_sync(0xffffffffu, good ? b : -1, l);
                            if ((fullmask >> l) & 1u) continue;
                            uint4 x = make_uint4(0u, 0u, 0u, 0u);
                            if (bl >= 0 && kbase + r < send)
                                x = *reinterpret_cast<const uint4 *>(
                                    a.pool + ((((int64_t)bl * 2 + 1) * a.hkv + kvh) * a.tile_elems +
                                              (int64_t)(r - (l << a.lg_bs)) * D) * EB + cc * 16);
                            if constexpr (KV8) {
                                *reinterpret_cast<uint4 *>(stage + kCodeOff + r * D + cc * 16) = x;
                            } else {
                                const int c2 = cc >> 3, u = cc & 7;
                                *reinterpret_cast<uint4 *>(stage + c2 * BN * 128 + r * 128 + ((u ^ (r & 7)) << 4)) = x;
                            }
                        }
                        if constexpr (!KV8) fence_proxy_async_smem(); // the plain stores are read by the MMA
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(full + st);
                } else {
                    if (lane == 0) {
                        mbar_arrive_expect_tx(full + st, L::TILE);
#pragma unroll
                        for (int c = 0; c < D / 64; ++c)
                            tc::tma_load_2d(stage + c * BN * 128, isK ? &tk : &tv, kvh * D + c * 64, it.start + e * BN,
                                            full + st);
                    }
                    if (writes && e >= q0 / BN) {
                        // the tile holds some of the item's own rows: write them before the stage is refilled
                        wj[st] = e;
                        wq0[st] = q0;
                        wql[st] = qlast;
                        wkvh[st] = kvh;
                        wblk[st] = blkv;
                        wpar[st] = (int)(round & 1);
                    }
                }
                issued = e + 1;
                if constexpr (KV8) pend = gg;
                if (isK && e < 2) issue_q(e); // Q_A after K tile 0, Q_B after K tile 1
            }
            if (isK) issue_q(1); // items of fewer than two key tiles
            g += issued; // tiles issued so far, all items
            if (!isK && lane == 0) mbar_arrive(item_empty + (n & (kItemSlots - 1)));
            if (!ok) {
                if (lane == 0) fail();
                break;
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        }
        // FP8: the last tile issued is widened too (an MMA may still be waiting for it)
        if (ok && !widen_pending() && lane == 0) fail();
        // pending pool writes leave now; every store has completed before the CTA exits
        for (int st = 0; st < ns; ++st) flush_write(st);
        if constexpr (WRITER) tc::bulk_wait_all();
        // the last loads must land before this CTA's shared memory goes away
        if (lane == 0) {
            for (int64_t gg = g > ns ? g - ns : 0; gg < g; ++gg)
                if (!mbar_wait_hint(full + gg % ns, (gg / ns) & 1)) set_error(a.err, PKV_DEVERR_TIMEOUT);
            if (isK)
                for (int b = 0; b < 2; ++b)
                    if (nq[b] >= 1 && !mbar_wait_hint(q_full + b, (nq[b] - 1) & 1)) set_error(a.err, PKV_DEVERR_TIMEOUT);
        }
    } else if (warp == 1 || warp == 3) {
        // ---------------------------------------------------------------- MMA issuers
        // Warp 1 issues the products of tile A, warp 3 those of tile B, each from a converged warp with
        // one elected lane issuing (waits agreed with __all_sync).  Per tile: S(0), then per key step
        // j: P V(j), S(j+1).  S(j+1) follows P V(j) from the same thread, so it overwrites the S
        // columns only after P V(j) has read P from them.  Two issuers keep the tensor pipe's queue fed
        // while either waits for its softmax.  Commits track the issuing thread's own MMAs.
        const int t = warp == 1 ? 0 : 1;
        constexpr uint32_t IQK = tc::idesc_f16(MT == PKV_BF16 ? 1u : 0u, 0u, BM, BN);
        constexpr uint32_t IPV = tc::idesc_f16(MT == PKV_BF16 ? 1u : 0u, 1u, BM, D);
        // one descriptor per operand layout; the address field counts 16-byte units, so a tile at byte
        // offset `off` from the base is the base descriptor plus off / 16
        const uint64_t dQ = tc::smem_desc(smem_u32(smem + L::Q), 16, 1024);
        const uint64_t dK = tc::smem_desc(smem_u32(smem + L::K0), 16, 1024);
        const uint64_t dV = tc::smem_desc(smem_u32(smem + L::V0), BN * 128, 1024);
        const uint32_t tS = tmem + (uint32_t)(t * BN), tO = tmem + (uint32_t)(2 * BN + t * D);
        bool any_mma = false, ok = true;
        // ring cursors: the stage of the K (V) entry to look at next and the parity of its phase
        uint32_t kst = 0, kph = 0, vst = 0, vph = 0;
        uint32_t pph = 0, oph = 0, qph = 0; // phase parities of this tile's barriers
        bool o_used = false;
        auto adv = [](uint32_t &st, uint32_t &ph, int nstage) {
            if (++st == (uint32_t)nstage) {
                st = 0;
                ph ^= 1u;
            }
        };
        for (int n = 0; ok; ++n) {
            const Item it = take_item(n, ok);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok || it.seq < 0) break;
            const int nt = t ? it.t[1].n : it.t[0].n;
            // shared modes: key entries j >= n_other are read by this tile alone, which then gives the
            // stage's release for both tiles (two commits), so the other tile's issuer skips them
            // without waiting for their loads
            const int n_other = t ? it.t[0].n : it.t[1].n;
            const int ne = ring_count<SHARED>(it);
            const int qb = CASCADE ? 0 : t;
            // ring entries of the item this warp has passed (cascade: the other tile's are skipped)
            int ke = 0, ve = 0;
            auto owner = [&](int e) -> int {
                int tt, jj;
                ring_entry<SHARED>(it, e, tt, jj);
                return tt;
            };
            // move a cursor to this tile's next entry (cascade: over the other tile's entries)
            auto skip_others = [&](int &pos, uint32_t &st, uint32_t &ph, int nstage) {
                if (!SHARED) {
                    while (pos < ne && owner(pos) != t) {
                        adv(st, ph, nstage);
                        ++pos;
                    }
                }
            };
            // S(j) = Q K^T into the tile's S columns (its MMAs only; the caller commits)
            auto mmas_s = [&]() {
                const uint64_t a0 = dQ + (uint64_t)((qb * L::Q_TILE) >> 4);
                const uint64_t b0 = dK + (uint64_t)(kst * (L::STAGE >> 4));
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const int c = k >> 2, kk = k & 3;
                    tc::mma_f16_warp(tS, a0 + (uint64_t)((c * BM * 128 + kk * 32) >> 4),
                                     b0 + (uint64_t)((c * BN * 128 + kk * 32) >> 4), IQK, k > 0 ? 1u : 0u);
                }
            };
            // after S(j): S complete, this warp's share of the K stage, and Q after the tile's last S
            auto commit_s = [&](int j) {
                tc::commit_warp(s_full + t);
                tc::commit_warp(k_empty + kst); // this warp's share of the K stage
                if (SHARED && j >= n_other) tc::commit_warp(k_empty + kst); // and the other tile's
                adv(kst, kph, NKS);
                ++ke;
                if (j == nt - 1) {
                    // cascade: the last S of the tile has read Q (other modes: the epilogue, which stages
                    // the tile's output in the Q buffer, frees it)
                    if constexpr (CASCADE) tc::commit_warp(q_empty + qb);
                    qph ^= 1u;
                }
            };
            // S(0): Q and the first K tile
            auto first_s = [&]() -> bool {
                skip_others(ke, kst, kph, NKS);
                if (!__all_sync(0xffffffffu, mbar_wait(k_ready + kst, kph) && mbar_wait(q_full + qb, qph))) return false;
                tc::fence_after_sync();
                any_mma = true;
                mmas_s();
                commit_s(0);
                return true;
            };
            // O += P(j) V(j), then S(j + 1) right behind it: the pipe gets both groups back to back.
            // P is read from tensor memory where the softmax left it (over S), and S(j + 1) overwrites
            // those columns only after P V(j) has read them (one thread's MMAs complete in order).
            auto step = [&](int j) -> bool {
                skip_others(ve, vst, vph, NVS);
                const bool more = j + 1 < nt;
                // the next K tile is normally in place already; checked first, so that nothing but the
                // softmax is waited for between the two groups
                if (more) {
                    skip_others(ke, kst, kph, NKS);
                    if (!__all_sync(0xffffffffu, mbar_wait(k_ready + kst, kph))) return false;
                }
                bool w = mbar_wait(v_ready + vst, vph) && mbar_wait(p_full + t, pph);
                // the previous item's epilogue of this tile has read O out of tensor memory
                if (j == 0 && o_used) w = w && mbar_wait(o_free + t, oph ^ 1u);
                if (!__all_sync(0xffffffffu, w)) return false;
                pph ^= 1u;
                tc::fence_after_sync();
                const uint64_t b0 = dV + (uint64_t)(vst * (L::STAGE >> 4));
#pragma unroll
                for (int part = 0; part < NP; ++part)
#pragma unroll
                    for (int k = 0; k < BN / 16; ++k)
                        tc::mma_f16_ts_warp(tO, tS + (uint32_t)(part * (BN / 2) + k * 8), b0 + (uint64_t)((k * 2048) >> 4),
                                            IPV, (j > 0 || k > 0 || part > 0) ? 1u : 0u);
                // the V stage share goes out before S(j + 1) is issued (a commit covers every earlier MMA of
                // this thread, so issued later it would hold the stage until S(j + 1) completes too); the
                // P V MMAs queued ahead keep the pipe busy meanwhile
                tc::commit_warp(v_empty + vst); // this warp's share of the V stage
                if (SHARED && j >= n_other) tc::commit_warp(v_empty + vst); // and the other tile's
                adv(vst, vph, NVS);
                ++ve;
                if (more) mmas_s();
                if (!more) {
                    tc::commit_warp(o_full + t); // the tile's O is complete once this commit arrives
                    oph ^= 1u;
                    o_used = true;
                } else {
                    commit_s(j + 1);
                }
                return true;
            };
            if (nt > 0) ok = first_s();
            for (int j = 0; j < nt && ok; ++j) ok = step(j);
            if constexpr (SHARED) {
                // key tiles only the other tile reads: released by that tile (see n_other)
                for (; ke < ne; ++ke, ++ve) {
                    adv(kst, kph, NKS);
                    adv(vst, vph, NVS);
                }
            } else {
                // the other tile's remaining entries
                for (; ke < ne; ++ke) adv(kst, kph, NKS);
                for (; ve < ne; ++ve) adv(vst, vph, NVS);
                if (nt == 0 && ok) {
                    // cascade: no split for this tile; its share of the Q buffer once Q has landed
                    ok = __all_sync(0xffffffffu, mbar_wait_hint(q_full + qb, qph));
                    if (ok && lane == 0) mbar_arrive(q_empty + qb);
                    qph ^= 1u;
                }
            }
            if (lane == 0) mbar_arrive(item_empty + (n & (kItemSlots - 1)));
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        }
        if (!ok && lane == 0) fail();
        // every MMA issued by this warp's elected lane has completed before TMEM is released (a warp that
        // issued none has nothing to wait for)
        if (any_mma) {
            tc::commit_warp(fin + t);
            if (!__all_sync(0xffffffffu, mbar_wait_hint(fin + t, 0)) && lane == 0) set_error(a.err, PKV_DEVERR_TIMEOUT);
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 200;");
        // ---------------------------------------------------------------- softmax, one thread per row
        const int t = (warp - 4) >> 2;          // tile A (warps 4-7) or B (warps 8-11)
        const int r = (warp & 3) * 32 + lane;   // query row of the tile = tensor-memory lane
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + lane_off + (uint32_t)(t * BN);
        const uint32_t tO = tmem + lane_off + (uint32_t)(2 * BN + t * D);
        bool ok = true;
        int ns = 0, no = 0, nepi = 0;
        int steps0 = 0, steps1 = 0; // key steps of tiles A and B in earlier items
        // The two tiles' softmaxes take turns on the exponentials (they share the SMSPs and their
        // transcendental units; run together, each takes twice as long and the MMAs of both tiles
        // wait): in an item, A's step j follows B's step j - 1, and B's step j follows A's step j.
        // The wait reads the other tile's monotonic count of finished steps, polled with a bound.
        auto wait_turn = [&](int other, int target) -> bool {
            volatile int *prog = sm_prog + other;
            if (*prog >= target) return true;
            const uint64_t t0 = global_timer_ns();
            for (uint32_t i = 0; i < 0x80000000u; ++i) {
                if (*prog >= target) return true;
                __nanosleep(32);
                if ((i & 63u) == 0u && global_timer_ns() - t0 > PKV_WAIT_LIMIT_NS) return false;
            }
            return false;
        };
        for (int n = 0; ok; ++n) {
            const Item it = take_item(n, ok);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok || it.seq < 0) break;
            const Tile x = t ? it.t[1] : it.t[0];
            const int n0 = it.t[0].n, n1 = it.t[1].n;
            if (x.n > 0) {
                const int kvh = it.h / G;
                const float sl = KV8 ? a.scale_log2 * a.k_scale[kvh] : a.scale_log2;
                const int qpos = x.qpos0 + r; // absolute position of this row (causal modes)
                float m_use = -INFINITY, l = 0.f;
                for (int j = 0; j < x.n && ok; ++j) {
                    // (spinning: S complete is on the critical path; a suspended wait wakes later)
                    ok = __all_sync(0xffffffffu, mbar_wait(s_full + t, ns & 1));
                    if (!ok) break;
                    ++ns;
                    tc::fence_after_sync();
                    uint32_t sr[BN];
#pragma unroll
                    for (int c = 0; c < BN / 32; ++c)
                        tc::ld32(tS + c * 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[c * 32]));
                    tc::wait_ld();
                    const int kbase = x.k0 + j * BN;
                    if constexpr (CASCADE) {
                        // every query sees the whole split: only keys past its end are masked
                        if (kbase + BN > x.kend) {
                            const int lim = x.kend - kbase;
#pragma unroll
                            for (int c = 0; c < BN; ++c)
                                if (c >= lim) sr[c] = 0xFF800000u; // -inf
                        }
                    } else if (kbase + BN - 1 > x.qpos0) {
                        // causal mask, only on tiles that reach past the tile's first query row
                        const int lim = qpos - kbase + 1; // keys c < lim are at or before this row
#pragma unroll
                        for (int c = 0; c < BN; ++c)
                            if (c >= lim) sr[c] = 0xFF800000u; // -inf
                    }
                    // row maximum: eight independent chains of three-input maxima, then a short tree
                    float mc[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) mc[q] = __uint_as_float(sr[q]);
#pragma unroll
                    for (int c = 8; c < BN; c += 16) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) mc[q] = max3(mc[q], __uint_as_float(sr[c + q]), __uint_as_float(sr[c + 8 + q]));
                    }
                    const float mx = fmaxf(max3(mc[0], mc[1], mc[2]), max3(mc[3], mc[4], max3(mc[5], mc[6], mc[7]))) *
                                     sl; // scale > 0 keeps the order
                    const bool up = mx > m_use + kRescale;
                    const float m_new = up ? mx : m_use;
                    const float alpha = up ? fast_exp2(m_use - m_new) : 1.f;
                    m_use = m_new;
                    const float nbase = m_use == -INFINITY ? 0.f : -m_use; // a row with no live key yet keeps p = 0
                    // O rescale (rows whose base moved): P V(j - 1) has completed, since S(j) has
                    if (j > 0 && __any_sync(0xffffffffu, up)) {
#pragma unroll
                        for (int cc = 0; cc < D / 16; ++cc) {
                            uint32_t o[16];
                            tc::ld16(tO + cc * 16, o);
                            tc::wait_ld();
#pragma unroll
                            for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                            tc::st16(tO + cc * 16, o);
                        }
                    }
                    // this tile's turn on the exponentials (see wait_turn)
                    if (t == 0 ? (j >= 1 && j - 1 < n1) : (j < n0)) {
                        const int target = 4 * (t == 0 ? steps1 + j : steps0 + j + 1);
                        ok = __all_sync(0xffffffffu, wait_turn(1 - t, target));
                        if (!ok) break;
                    }
                    float2 rs = make_float2(0.f, 0.f);
                    const float2 sc2 = make_float2(sl, sl), nb2 = make_float2(nbase, nbase);
                    // P over the S columns: packed pairs, key c in column c / 2 (bf16: lo parts from BN / 2)
                    // (keys per store: 32 for fp16 P, 16 for a bf16 hi + lo pair, to keep registers for S)
                    constexpr int KC = NP == 2 ? 16 : 32;
#pragma unroll
                    for (int q = 0; q < BN / KC; ++q) {
                        uint32_t phi[KC / 2], plo[NP == 2 ? KC / 2 : 1];
#pragma unroll
                        for (int c = 0; c < KC / 2; ++c) {
                            const int k = q * KC + 2 * c;
                            const float2 xx =
                                fma2(make_float2(__uint_as_float(sr[k]), __uint_as_float(sr[k + 1])), sc2, nb2);
                            const float p0 = fast_exp2(xx.x), p1 = fast_exp2(xx.y);
                            rs = add2(rs, make_float2(p0, p1));
                            phi[c] = pack2(p0, p1, MT);
                            if constexpr (NP == 2) // remainders after bf16 rounding, themselves rounded to bf16
                                plo[c] = pack2(p0 - __uint_as_float(phi[c] << 16),
                                               p1 - __uint_as_float(phi[c] & 0xFFFF0000u), MT);
                        }
                        if constexpr (NP == 2) {
                            tc::stn<8>(tS + q * 8, phi);
                            tc::stn<8>(tS + BN / 2 + q * 8, plo);
                        } else {
                            tc::st16(tS + q * 16, phi);
                        }
                    }
                    l = l * alpha + (rs.x + rs.y);
                    tc::wait_st();
                    tc::fence_before_sync();
                    __syncwarp(); // every lane's P is stored; one arrival for the warp
                    if (lane == 0) {
                        mbar_arrive(p_full + t);
                        atomicAdd(sm_prog + t, 1); // this warp's exp phase of the step is done
                    }
                }
                // the tile's O is complete
                if (ok) ok = __all_sync(0xffffffffu, mbar_wait_hint(o_full + t, no & 1));
                if (!ok) break;
                ++no;
                tc::fence_after_sync();
                using T = typename ModelT<MT>::T;
                const float vs = KV8 ? a.v_scale[kvh] : 1.f;
                if constexpr (CASCADE) {
                    // fp32 partial of (sequence it.start + r, head it.h, split 2 pr + t): unnormalised o
                    // and (m, l) with m the row's exponent base in log2 units, as the split merge expects
                    const bool valid = r < it.n;
                    const int64_t idx = ((int64_t)(it.start + r) * a.hq + it.h) * a.max_splits + 2 * it.pr + t;
                    float *wo = a.ws_o + idx * D;
                    uint32_t o[D]; // the whole row in one tensor-memory round trip
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) tc::ld32(tO + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[cc * 32]));
                    tc::wait_ld();
                    if (valid) {
                        float4 *dst = reinterpret_cast<float4 *>(wo);
#pragma unroll
                        for (int e = 0; e < D / 4; ++e)
                            dst[e] = make_float4(__uint_as_float(o[4 * e]) * vs, __uint_as_float(o[4 * e + 1]) * vs,
                                                 __uint_as_float(o[4 * e + 2]) * vs, __uint_as_float(o[4 * e + 3]) * vs);
                    }
                    if (valid) reinterpret_cast<float2 *>(a.ws_ml)[idx] = make_float2(m_use, l);
                } else {
                    const int row = x.q0 + r;
                    const float inv = vs / l;
                    uint32_t o[D]; // the whole row in one tensor-memory round trip
#pragma unroll
                    for (int cc = 0; cc < D / 32; ++cc) tc::ld32(tO + cc * 32, *reinterpret_cast<uint32_t(*)[32]>(&o[cc * 32]));
                    tc::wait_ld();
                    const bool lead = (warp & 3) == 0 && lane == 0;
                    if (x.q0 + BM <= it.n) {
                        // a whole tile of the sequence's rows: staged in this tile's Q buffer (free, since the
                        // tile's last S has completed) in the Q tile's own 128-byte swizzled layout, then one TMA
                        // store per 64 columns writes coalesced rows; the buffer goes back to the Q loader once
                        // the stores have read it
                        uint8_t *stage = smem + L::Q + t * L::Q_TILE;
#pragma unroll
                        for (int cc = 0; cc < D / 8; ++cc) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                w[e] = pack2(__uint_as_float(o[8 * cc + 2 * e]) * inv, __uint_as_float(o[8 * cc + 2 * e + 1]) * inv, MT);
                            const int h = cc >> 3, u = cc & 7;
                            *reinterpret_cast<uint4 *>(stage + h * BM * 128 + r * 128 + ((u ^ (r & 7)) << 4)) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                        }
                        fence_proxy_async_smem(); // the stores read the tile through the async proxy
                        __syncwarp();
                        if (lane == 0) mbar_arrive(epi + t);
                        if (lead) {
                            // the four warps' rows are staged (bounded wait: a warp that gave up never arrives)
                            if (mbar_wait(epi + t, nepi & 1)) {
#pragma unroll
                                for (int h = 0; h < D / 64; ++h)
                                    tc::tma_store_2d(&to, it.h * D + h * 64, it.start + x.q0, stage + h * BM * 128);
                                tc::bulk_commit();
                                tc::bulk_wait_read_all();
                                mbar_arrive(q_empty + t);
                            } else {
                                ok = false;
                            }
                        }
                        ++nepi;
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                    } else {
                        // the sequence's last, partial tile: row by row, so that no row of the next sequence is
                        // written; the Q buffer is not used here and is free already
                        if (lead) mbar_arrive(q_empty + t);
                        if (row < it.n) {
                            T *orow = static_cast<T *>(a.out) + ((int64_t)(it.start + row) * a.hq + it.h) * D;
#pragma unroll
                            for (int cc = 0; cc < D / 8; ++cc) {
                                uint32_t w[4];
#pragma unroll
                                for (int e = 0; e < 4; ++e)
                                    w[e] = pack2(__uint_as_float(o[8 * cc + 2 * e]) * inv,
                                                 __uint_as_float(o[8 * cc + 2 * e + 1]) * inv, MT);
                                reinterpret_cast<uint4 *>(orow)[cc] = make_uint4(w[0], w[1], w[2], w[3]);
                            }
                        }
                    }
                }
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(o_free + t); // O has been read out; the tile's next first P V may overwrite it
            }
            steps0 += n0;
            steps1 += n1;
            __syncwarp();
            if (lane == 0) mbar_arrive(item_empty + (n & (kItemSlots - 1)));
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        }
        if (!ok) fail();
        // the output tiles' TMA stores have completed before the CTA exits
        if (!CASCADE && (warp & 3) == 0 && lane == 0) tc::bulk_wait_all();
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if constexpr (CASCADE) pdl_wait(); // the grid completes after the suffix decode (see above)
}

// launch of one instantiation (prefill_packed.cu, prefill_paged.cu, prefill_cascade.cu)
template <int D, int MT, int MODE, bool KV8>
cudaError_t launch_attn(const Maps &m, const Args &a, int64_t max_ctas, int num_sms, cudaStream_t st) {
    auto kern = attn_kernel<D, MT, MODE, KV8>;
    const int smem = Layout<D, KV8>::TOTAL;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(max_ctas, (int64_t)num_sms);
    return pdl_launch(kern, dim3((unsigned)grid), dim3(kThreads), smem, st, m, a);
}

#define PKV_ATTN_EXTERN(MODE, KV8)                                                                                     \
    extern template cudaError_t launch_attn<128, PKV_F16, MODE, KV8>(const Maps &, const Args &, int64_t, int, cudaStream_t);  \
    extern template cudaError_t launch_attn<128, PKV_BF16, MODE, KV8>(const Maps &, const Args &, int64_t, int, cudaStream_t); \
    extern template cudaError_t launch_attn<64, PKV_F16, MODE, KV8>(const Maps &, const Args &, int64_t, int, cudaStream_t);   \
    extern template cudaError_t launch_attn<64, PKV_BF16, MODE, KV8>(const Maps &, const Args &, int64_t, int, cudaStream_t);
#define PKV_ATTN_INSTANTIATE(MODE, KV8)                                                                         \
    template cudaError_t launch_attn<128, PKV_F16, MODE, KV8>(const Maps &, const Args &, int64_t, int, cudaStream_t);  \
    template cudaError_t launch_attn<128, PKV_BF16, MODE, KV8>(const Maps &, const Args &, int64_t, int, cudaStream_t); \
    template cudaError_t launch_attn<64, PKV_F16, MODE, KV8>(const Maps &, const Args &, int64_t, int, cudaStream_t);   \
    template cudaError_t launch_attn<64, PKV_BF16, MODE, KV8>(const Maps &, const Args &, int64_t, int, cudaStream_t);

PKV_ATTN_EXTERN(MODE_PACKED, false)
PKV_ATTN_EXTERN(MODE_PAGED, false)
PKV_ATTN_EXTERN(MODE_PAGED, true)
PKV_ATTN_EXTERN(MODE_CASCADE, false)
PKV_ATTN_EXTERN(MODE_CASCADE, true)

} // namespace pkv_prefill
