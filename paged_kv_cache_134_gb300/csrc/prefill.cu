// Packed causal prefill on the 5th-generation tensor cores, with the paged K/V write fused in.
//
// What it computes ("Paged KV Cache 与 Packed Sequence", discosf.com, sections 3.1-3.3, 4.2):
// sequences packed back to back, sequence i owning rows [cu[i], cu[i+1]); a query at in-sequence
// position r attends to the keys of its own sequence at positions c <= r (block-diagonal causal
// mask), out = softmax(scale q.k) v.  Every token's k/v is also written into the paged cache at
// block_table[i][r / bs], offset r % bs (the prompt-phase write of section 4.2, bounded by the
// sequence length so a partly filled tail block is never overrun).
//
// Work items are (sequence, 128-query tile, query head) triples.  A one-CTA plan kernel lists the
// (sequence, query tile) pairs heaviest first; a persistent grid (as many CTAs as fit, two per SM
// for fp16 models at D = 128) then takes items one at a time from an atomic counter, so an SM
// whose item ends early starts the next one at once instead of waiting for the hardware to
// dispatch a new CTA.  Warp roles inside a CTA:
//   warp 0     lane 0: takes the next item and hands it to the other roles through a 2-entry ring
//              in shared memory, then loads its Q tile and its K tiles of 64 keys into a 2-stage
//              ring; lane 1 loads the V tiles into another 2-stage ring (tiled TMA, 128-byte
//              swizzle, out-of-range rows zero-filled); a K stage frees when S = Q K^T of its tile is
//              done and the writer warps have passed it, a V stage likewise after P V;
//   warp 1     tensor-memory owner and MMA issuer (one thread): S = Q K^T into one of two TMEM S
//              buffers (M=128, N=64, fp32), then O += P V into the TMEM O accumulator (M=128, N=D);
//   warps 2-5  softmax, one thread per query row (TMEM lane = row): mask, exp2, row sums, P written
//              to shared memory in the 128-byte-swizzled K-major layout the MMA reads (fp16 P for
//              fp16 models; for bf16 models P = hi + lo, two bf16 tiles and two accumulating MMAs);
//              O in TMEM is rescaled only when a row's running max grows by more than 2^8 (the
//              exponent base stays fixed otherwise, which is exact algebra); then the epilogue;
//   warps 6-7  paged K/V writer for the item's rows, straight from the K/V tiles already in shared
//              memory as they land (only items of the first query head of each KV group write, so
//              every (token, KV head) is written once).
// Every barrier phase is counted across items (a global K/V tile counter, an item counter), so the
// pipeline runs on from one item into the next.  The diagonal tiles are masked per element; tiles
// entirely above the diagonal are never issued.  Every mbarrier wait is bounded; a timeout sets
// PKV_DEVERR_TIMEOUT and the CTA winds down.
#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "tcgen05.cuh"
#include "pkv_internal.h"

namespace pkv_prefill {

constexpr int BM = 128;          // query rows per tile (MMA M)
constexpr int BN = 64;           // keys per tile (MMA N of Q K^T, K of P V)
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 256; // S [0,64), P buffers [64,128), O [128, 128+D)
constexpr float kRescale = 8.0f; // log2 units

struct Args {
    const char *k, *v;  // packed [T][Hkv][D]
    void *out;          // packed [T][Hq][D]
    const int32_t *cu, *tables;
    char *pool;
    unsigned int *err;
    int *plan;          // [0] item count, [1] next-item counter, [4 + 2i], [5 + 2i] = (sequence, query tile) of item i
    const int32_t *ctx; // paged mode: tokens each sequence already holds in its blocks (else NULL)
    int64_t total_tokens, num_blocks, tile_elems;
    int num_seqs, max_seqlen, max_blocks, hq, hkv, bs, lg_bs, nqt_max;
    float scale_log2;
    // cascade mode: the decode queries of num_seqs sequences against a shared prefix of
    // prefix_tokens tokens (table row 0), cut into nps splits of split_tokens keys; each (sequence,
    // query head, split) leaves an fp32 partial (m, l, unnormalised o) in workspace slot split
    float *ws_o = nullptr, *ws_ml = nullptr;
    int max_splits = 0, prefix_tokens = 0, split_tokens = 0, nps = 0;
};

enum { MODE_PACKED = 0, MODE_PAGED = 1, MODE_CASCADE = 2 };

constexpr int NKS = 3;           // K stages (a K stage frees as soon as S = Q K^T of its tile is done)
constexpr int NVS = 2;           // V stages (a V stage frees after P V)

// Shared memory: Q, the K ring and the V ring (P lives in tensor memory).  bf16 models keep P as a
// hi + lo pair of bf16 halves (P = hi + lo to ~2^-16 relative), because one bf16 rounding of P
// (2^-9 relative) alone would exceed the accuracy the outputs are held to; fp16 P (2^-12) is one.
template <int D, int MT>
struct Layout {
    static constexpr int NP = MT == PKV_BF16 ? 2 : 1;
    // P buffers in tensor memory (columns [BN, 2 BN)): two fp16 P tiles of BN/2 columns, or one bf16
    // hi + lo pair; with two, the softmax never waits for P V before writing the next P
    static constexpr int NPB = NP == 1 ? 2 : 1;
    static constexpr int Q = 0;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2; // one K or V tile
    static constexpr int K0 = Q + Q_BYTES;
    static constexpr int V0 = K0 + NKS * KV_BYTES;
    static constexpr int BAR = V0 + NVS * KV_BYTES;
    static constexpr int TOTAL = BAR + 256; // 24 mbarriers, the TMEM slot, a flag, two 16-byte item slots
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

// two CTAs per SM whenever the shared memory allows it (then at most 128 registers a thread)
template <int D, int MT>
constexpr int min_blocks() {
    return 2 * (Layout<D, MT>::TOTAL + 1024) <= 233472 ? 2 : 1;
}

constexpr int kPlanThreads = 1024;
constexpr int kItemConsumers = 7;  // V loader, MMA issuer, 4 softmax warps, the writer warp
constexpr int kStageReleasers = 2; // a K or V stage frees after the MMA that reads it and the writer warp

// query tiles of sequence i (0 for a malformed cu_seqlens entry, which is reported)
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

// in-place inclusive prefix sum of x[0, n) by the whole CTA (kPlanThreads threads)
PKV_DEV void cta_inclusive_scan(int *x, int n, int *warp_sums) {
    const int per = (n + kPlanThreads - 1) / kPlanThreads;
    const int b = min((int)threadIdx.x * per, n), e = min(b + per, n);
    int own = 0;
    for (int i = b; i < e; ++i) own += x[i];
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int v = own;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    if (lane == 31) warp_sums[w] = v;
    __syncthreads();
    if (w == 0) {
        int u = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, u, o);
            if (lane >= o) u += t;
        }
        warp_sums[lane] = u;
    }
    __syncthreads();
    int run = v - own + (w > 0 ? warp_sums[w - 1] : 0);
    for (int i = b; i < e; ++i) {
        run += x[i];
        x[i] = run;
    }
    __syncthreads();
}

// The work list.  Rank r holds every sequence's r-th heaviest query tile (its (nq-1-r)-th): with
// gt[r] = #{i : nq_i > r} items in rank r, rank r starts at gt[0] + ... + gt[r-1].  Inside a rank
// the order is whatever the atomics give; it only decides which CTA computes an item, never what
// the item computes.  Also resets the next-item counter the attention kernel draws from.
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(const Args a) {
    extern __shared__ int sh[];
    const int R = a.nqt_max + 1;
    int *hist = sh;          // hist[c] = #{i : nq_i == c}, then rank starts
    int *cnt = sh + R;       // items placed so far in each rank
    int *warp_sums = sh + 2 * R;
    pdl_trigger();
    pdl_wait();
    if (a.nps > 0) {
        // cascade: the items are the (tile of query rows, prefix split) pairs, taken in order
        if (threadIdx.x == 0) {
            a.plan[0] = ((a.num_seqs + BM - 1) / BM) * a.nps;
            a.plan[1] = 0;
        }
        return;
    }
    for (int x = threadIdx.x; x < R; x += kPlanThreads) {
        hist[x] = 0;
        cnt[x] = 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < a.num_seqs; i += kPlanThreads) atomicAdd(&hist[min(seq_tiles(a, i, true), a.nqt_max)], 1);
    __syncthreads();
    cta_inclusive_scan(hist, R, warp_sums);                             // hist[r] = #{i : nq_i <= r}
    for (int x = threadIdx.x; x < R; x += kPlanThreads) hist[x] = a.num_seqs - hist[x]; // gt[r]
    __syncthreads();
    cta_inclusive_scan(hist, R, warp_sums);                             // hist[r] = gt[0] + ... + gt[r]
    int2 *list = reinterpret_cast<int2 *>(a.plan + 4);
    for (int i = threadIdx.x; i < a.num_seqs; i += kPlanThreads) {
        const int nq = min(seq_tiles(a, i, false), a.nqt_max);
        for (int r = 0; r < nq; ++r) {
            const int pos = (r > 0 ? hist[r - 1] : 0) + atomicAdd(&cnt[r], 1);
            list[pos] = make_int2(i, nq - 1 - r);
        }
    }
    if (threadIdx.x == 0) {
        a.plan[0] = hist[R - 1];
        a.plan[1] = 0;
    }
}

// one item as the roles see it
struct Item {
    int seq, qt, h; // seq < 0: no more items
    int start, n, q0, qlast, nkv;
    int c0;   // paged mode: cached tokens ahead of the item's sequence rows (absolute position of row 0)
    int k0;   // absolute position of the item's first key (cascade: its split's start; else 0)
    int kend; // keys at or past kend hold no token of the sequence (or of the prefix)
    int trow; // block-table row of the item's keys
};

PKV_DEV Item decode_item(const Args &a, int4 raw) {
    Item it;
    it.seq = raw.x;
    it.qt = raw.y;
    it.h = raw.z;
    if (it.seq >= 0 && a.nps > 0) {
        // cascade: seq = tile of 128 query rows (sequences), qt = prefix split
        it.start = it.seq * BM;
        it.n = min(BM, a.num_seqs - it.start);
        it.q0 = 0;
        it.qlast = it.n - 1;
        it.c0 = 0;
        it.k0 = it.qt * a.split_tokens;
        it.kend = min(it.k0 + a.split_tokens, a.prefix_tokens);
        it.nkv = (it.kend - it.k0 + BN - 1) / BN;
        it.trow = 0;
        return it;
    }
    if (it.seq >= 0) {
        it.start = a.cu[it.seq];
        it.n = a.cu[it.seq + 1] - it.start;
        it.q0 = it.qt * BM;
        it.qlast = min(it.q0 + BM, it.n) - 1;
        it.c0 = a.ctx ? a.ctx[it.seq] : 0;
        it.nkv = (it.c0 + it.qlast) / BN + 1; // key tiles up to the item's last row
        it.k0 = 0;
        it.kend = it.c0 + it.n;
        it.trow = it.seq;
    }
    return it;
}

template <int D, int MT, int MODE>
__global__ void __launch_bounds__(kThreads, min_blocks<D, MT>())
    prefill_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tp, const Args a) {
    using L = Layout<D, MT>;
    constexpr bool PAGED = MODE != MODE_PACKED;     // keys from the pool through the block table
    constexpr bool CASCADE = MODE == MODE_CASCADE;  // no causal mask, fp32 split partials out
    extern __shared__ __align__(1024) uint8_t smem[];

    pdl_trigger();
    if (smem_u32(smem) & 1023u) return; // the swizzled tiles need 1024-byte alignment (always true)

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR);
    uint64_t *q_full = bars + 0, *q_empty = bars + 1;
    uint64_t *k_full = bars + 2, *k_empty = k_full + NKS;          // [NKS] each
    uint64_t *v_full = k_empty + NKS, *v_empty = v_full + NVS;     // [NVS] each
    uint64_t *s_full = v_empty + NVS, *s_free = s_full + 1;        // phase t: S of global tile t
    // p_full[t % 2] / t_full[t % 2]: P of global tile t written / P V of tile t done (phase t / 2).
    // Pairs of barriers, so that a parity wait for tile t only needs tile t - 2 to be complete (which
    // every waiter knows already) while tile t + 2 cannot be: the softmax may run one tile ahead of
    // the P V issue, never two.
    uint64_t *p_full = s_full + 2, *t_full = p_full + 2, *o_free = t_full + 2;
    uint64_t *item_full = o_free + 1, *item_empty = item_full + 2, *fin = item_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(fin + 2);
    volatile int4 *item_slot = reinterpret_cast<volatile int4 *>(fin + 3); // [2], 16-byte aligned

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int s = 0; s < NKS; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(k_empty + s, kStageReleasers);
        }
        for (int s = 0; s < NVS; ++s) {
            mbar_init(v_full + s, 1);
            mbar_init(v_empty + s, kStageReleasers);
        }
        mbar_init(s_full, 1);
        mbar_init(s_free, 128);
        for (int s = 0; s < 2; ++s) {
            mbar_init(item_full + s, 1);
            mbar_init(item_empty + s, kItemConsumers);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(p_full + s, 128);
            mbar_init(t_full + s, 1);
        }
        mbar_init(o_free, 128);
        mbar_init(fin, 1);
        *abort_flag = 0;
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
    // suffix decode, which lets it launch once the decode itself has waited for its predecessors
    // (the plan of this call and everything before it): the prefix phase reads nothing the decode
    // writes, so it starts at once and fills the SMs the decode's CTAs leave, and waits for the
    // decode only before it exits (the merge after it then sees both).
    if constexpr (!CASCADE) pdl_wait();

    const int G = a.hq / a.hkv;
    auto fail = [&]() {
        set_error(a.err, PKV_DEVERR_TIMEOUT);
        *abort_flag = 1;
    };
    // the item in ring slot n % 2, once the scheduler has published it
    auto take_item = [&](int n, bool &ok) -> Item {
        Item it;
        it.seq = -1;
        ok = mbar_wait(item_full + (n & 1), (n >> 1) & 1);
        if (!ok) return it;
        const int4 raw = make_int4(item_slot[n & 1].x, item_slot[n & 1].y, item_slot[n & 1].z, 0);
        return decode_item(a, raw);
    };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ scheduler, Q and K loads
            tc::prefetch_tmap(&tq);
            tc::prefetch_tmap(&tk);
            const int total = a.plan[0] * a.hq;
            int n = 0, last_q = -1;
            int64_t g = 0; // K tiles issued so far (all items)
            for (;; ++n) {
                const int s = n & 1;
                if (n >= 2 && !mbar_wait(item_empty + s, ((n >> 1) - 1) & 1)) {
                    fail();
                    break;
                }
                const int idx = *abort_flag ? total : atomicAdd(a.plan + 1, 1);
                int4 raw = make_int4(-1, 0, 0, 0);
                if (idx < total) {
                    if constexpr (CASCADE) {
                        const int pair = idx / a.hq; // (tile of query rows, prefix split)
                        raw = make_int4(pair / a.nps, pair % a.nps, idx % a.hq, 0);
                    } else {
                        const int2 sq = reinterpret_cast<const int2 *>(a.plan + 4)[idx / a.hq];
                        raw = make_int4(sq.x, sq.y, idx % a.hq, 0);
                    }
                }
                item_slot[s].x = raw.x;
                item_slot[s].y = raw.y;
                item_slot[s].z = raw.z;
                mbar_arrive(item_full + s);
                if (raw.x < 0) break;
                const Item it = decode_item(a, raw);
                const int kvh = it.h / G;
                if (n >= 1 && !mbar_wait(q_empty, (n - 1) & 1)) {
                    fail();
                    break;
                }
                mbar_arrive_expect_tx(q_full, L::Q_BYTES);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tc::tma_load_2d(smem + L::Q + c * BM * 128, &tq, it.h * D + c * 64, it.start + it.q0, q_full);
                last_q = n;
                bool ok = true;
                int issued = 0;
                // paged mode: table entries of the blocks of one key tile (-1: no token of the sequence)
                int ent[BN / 8];
                auto read_entries = [&](const Item &itm, int jj) {
                    const int lb0 = (itm.k0 + jj * BN) >> a.lg_bs, nbt = BN >> a.lg_bs;
#pragma unroll
                    for (int l = 0; l < BN / 8; ++l)
                        ent[l] = (l < nbt && ((lb0 + l) << a.lg_bs) < itm.kend)
                                     ? a.tables[(int64_t)itm.trow * a.max_blocks + lb0 + l]
                                     : -1;
                };
                if constexpr (PAGED) read_entries(it, 0);
                for (int j = 0; j < it.nkv && ok; ++j) {
                    const int64_t gg = g + j;
                    const int st = (int)(gg % NKS);
                    const int64_t round = gg / NKS;
                    if (round >= 1) ok = mbar_wait(k_empty + st, (round - 1) & 1);
                    if (!ok || *abort_flag) break;
                    if constexpr (PAGED) {
                        // the tile's blocks that hold tokens of the sequence, one box of bs rows per
                        // block and half of D from the pool; rows past the sequence's end are masked
                        // by the softmax, and unusable block ids (reported by the V loader) are skipped.
                        // The table entries of tile j + 1 are read now, ahead of their use.
                        int blk[BN / 8];
                        uint32_t bytes = 0;
#pragma unroll
                        for (int l = 0; l < BN / 8; ++l) {
                            blk[l] = ent[l];
                            if (blk[l] >= a.num_blocks) blk[l] = -1;
                            if (blk[l] >= 0) bytes += (uint32_t)(a.bs * D * 2);
                        }
                        if (j + 1 < it.nkv) read_entries(it, j + 1);
                        mbar_arrive_expect_tx(k_full + st, bytes);
#pragma unroll
                        for (int l = 0; l < BN / 8; ++l)
                            if (blk[l] >= 0) {
                                const int y = (blk[l] * 2 * a.hkv + kvh) << a.lg_bs;
#pragma unroll
                                for (int c = 0; c < D / 64; ++c)
                                    tc::tma_load_2d(smem + L::K0 + st * L::KV_BYTES + c * BN * 128 +
                                                        ((l << a.lg_bs) * 128),
                                                    &tp, c * 64, y, k_full + st);
                            }
                    } else {
                        mbar_arrive_expect_tx(k_full + st, L::KV_BYTES);
#pragma unroll
                        for (int c = 0; c < D / 64; ++c)
                            tc::tma_load_2d(smem + L::K0 + st * L::KV_BYTES + c * BN * 128, &tk, kvh * D + c * 64,
                                            it.start + j * BN, k_full + st);
                    }
                    issued = j + 1;
                }
                g += issued; // tiles issued so far, all items
                if (!ok) {
                    fail();
                    break;
                }
                if (*abort_flag) break;
            }
            // the last loads must land before this CTA's shared memory goes away
            for (int64_t gg = g > NKS ? g - NKS : 0; gg < g; ++gg)
                if (!mbar_wait(k_full + gg % NKS, (gg / NKS) & 1)) set_error(a.err, PKV_DEVERR_TIMEOUT);
            if (last_q >= 0 && !mbar_wait(q_full, last_q & 1)) set_error(a.err, PKV_DEVERR_TIMEOUT);
        }
    } else if (warp == 7 && PAGED) {
        // ------------------------------------------------------------ V loads from the pool (whole warp)
        // Lane l handles block l of the tile.  Blocks full of the sequence's tokens arrive as TMA boxes;
        // every other row of the tile is written with plain stores: the tokens of a partly filled last
        // block copied from the pool, zeros for slots past the sequence and for unusable block ids.  P
        // is 0 on those rows, but 0 * NaN is NaN, and the pool's unused slots may hold anything.
        constexpr int CPR = D / 8;    // 16-byte chunks per row
        constexpr int RPI = 32 / CPR; // rows per warp instruction (never two blocks: bs >= 8)
        const int cc = lane % CPR, rsub = lane / CPR, c2 = cc >> 3, u = cc & 7;
        if (lane == 0) tc::prefetch_tmap(&tp);
        int64_t g = 0;
        bool ok = true;
        for (int n = 0;; ++n) {
            const Item it = take_item(n, ok);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok || it.seq < 0) break;
            const int kvh = it.h / G, send = it.kend, nbt = BN >> a.lg_bs;
            // lane l: table entry of block l of a key tile, read one tile ahead of its use
            auto entry = [&](int jj) -> int {
                const int lbl = ((it.k0 + jj * BN) >> a.lg_bs) + lane;
                return (lane < nbt && (lbl << a.lg_bs) < send) ? a.tables[(int64_t)it.trow * a.max_blocks + lbl] : -1;
            };
            int nxt = entry(0);
            int issued = 0;
            for (int j = 0; j < it.nkv && ok; ++j) {
                const int64_t gg = g + j;
                const int st = (int)(gg % NVS);
                const int64_t round = gg / NVS;
                const int b = nxt;
                if (j + 1 < it.nkv) nxt = entry(j + 1);
                if (round >= 1) ok = __all_sync(0xffffffffu, mbar_wait(v_empty + st, (round - 1) & 1));
                if (!ok || __any_sync(0xffffffffu, *abort_flag != 0)) break;
                const int kbase = it.k0 + j * BN, lb = (kbase >> a.lg_bs) + lane;
                const bool has = lane < nbt && (lb << a.lg_bs) < send;
                const bool good = has && b >= 0 && b < a.num_blocks;
                if (has && !good) set_error(a.err, PKV_DEVERR_BLOCK_ID);
                const bool full = good && ((lb + 1) << a.lg_bs) <= send;
                const unsigned fullmask = __ballot_sync(0xffffffffu, full);
                uint8_t *stage = smem + L::V0 + st * L::KV_BYTES;
                if (lane == 0) mbar_expect_tx(v_full + st, (uint32_t)__popc(fullmask) * (uint32_t)(a.bs * D * 2));
                __syncwarp();
                if (full) {
                    const int y = ((b * 2 + 1) * a.hkv + kvh) << a.lg_bs;
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tc::tma_load_2d(stage + c * BN * 128 + ((lane << a.lg_bs) * 128), &tp, c * 64, y, v_full + st);
                }
                for (int r0 = 0; fullmask != (1u << nbt) - 1u && r0 < BN; r0 += RPI) {
                    const int r = r0 + rsub, l = r >> a.lg_bs;
                    const int bl = __shfl_sync(0xffffffffu, good ? b : -1, l);
                    if ((fullmask >> l) & 1u) continue;
                    uint4 x = make_uint4(0u, 0u, 0u, 0u);
                    if (bl >= 0 && kbase + r < send)
                        x = *reinterpret_cast<const uint4 *>(
                            a.pool + ((((int64_t)bl * 2 + 1) * a.hkv + kvh) * a.tile_elems +
                                      (int64_t)(r - (l << a.lg_bs)) * D + cc * 8) * 2);
                    *reinterpret_cast<uint4 *>(stage + c2 * BN * 128 + r * 128 + ((u ^ (r & 7)) << 4)) = x;
                }
                fence_proxy_async_smem(); // the plain stores are read by the MMA (async proxy)
                __syncwarp();
                if (lane == 0) mbar_arrive(v_full + st);
                issued = j + 1;
            }
            g += issued; // tiles issued so far, all items
            if (lane == 0) mbar_arrive(item_empty + (n & 1));
            if (!ok || __any_sync(0xffffffffu, *abort_flag != 0)) break;
        }
        if (!ok && lane == 0) fail();
        if (lane == 0)
            for (int64_t gg = g > NVS ? g - NVS : 0; gg < g; ++gg)
                if (!mbar_wait(v_full + gg % NVS, (gg / NVS) & 1)) set_error(a.err, PKV_DEVERR_TIMEOUT);
    } else if (warp == 7) {
        // a warp of its own: sharing one with the K loader, whose lane spins on its own barriers,
        // held V loads back by thousands of cycles at every item start
        if (lane == 0) {
            // ------------------------------------------------------------ V loads
            tc::prefetch_tmap(&tv);
            int64_t g = 0;
            for (int n = 0;; ++n) {
                bool ok;
                const Item it = take_item(n, ok);
                if (!ok) fail();
                if (!ok || it.seq < 0) break;
                const int kvh = it.h / G;
                int issued = 0;
                for (int j = 0; j < it.nkv && ok; ++j) {
                    const int64_t gg = g + j;
                    const int st = (int)(gg % NVS);
                    const int64_t round = gg / NVS;
                    if (round >= 1) ok = mbar_wait(v_empty + st, (round - 1) & 1);
                    if (!ok || *abort_flag) break;
                    mbar_arrive_expect_tx(v_full + st, L::KV_BYTES);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tc::tma_load_2d(smem + L::V0 + st * L::KV_BYTES + c * BN * 128, &tv, kvh * D + c * 64,
                                        it.start + j * BN, v_full + st);
                    issued = j + 1;
                }
                g += issued; // tiles issued so far, all items
                mbar_arrive(item_empty + (n & 1));
                if (!ok) {
                    fail();
                    break;
                }
                if (*abort_flag) break;
            }
            for (int64_t gg = g > NVS ? g - NVS : 0; gg < g; ++gg)
                if (!mbar_wait(v_full + gg % NVS, (gg / NVS) & 1)) set_error(a.err, PKV_DEVERR_TIMEOUT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // the whole warp runs the issue loop in step (waits agreed with __all_sync); one elected lane
        // issues each MMA and commit
        {
            constexpr uint32_t IQK = tc::idesc_f16(MT == PKV_BF16 ? 1u : 0u, 0u, BM, BN);
            constexpr uint32_t IPV = tc::idesc_f16(MT == PKV_BF16 ? 1u : 0u, 1u, BM, D);
            const uint32_t tO = tmem + 2 * BN;
            // one descriptor per operand layout; the address field counts 16-byte units, so a tile at
            // byte offset `off` from the base is the base descriptor plus off / 16 (shared memory stays
            // below the field's 256 KB): each MMA adds a constant instead of rebuilding its descriptors
            const uint64_t dQ = tc::smem_desc(smem_u32(smem + L::Q), 16, 1024);
            const uint64_t dK = tc::smem_desc(smem_u32(smem + L::K0), 16, 1024);
            const uint64_t dV = tc::smem_desc(smem_u32(smem + L::V0), BN * 128, 1024);
            bool any_mma = false;
            // S of global tile gg = Q K^T, once the softmax has read S of tile gg - 1 out of the single
            // S buffer; the K stage is released as soon as S is done
            auto issue_s = [&](int64_t gg) -> bool {
                const int st = (int)(gg % NKS);
                if (!__all_sync(0xffffffffu, mbar_wait(k_full + st, (gg / NKS) & 1) &&
                                                 (gg < 1 || mbar_wait(s_free, (gg - 1) & 1))))
                    return false;
                tc::fence_after_sync();
                any_mma = true;
                const uint64_t b0 = dK + (uint64_t)((st * L::KV_BYTES) >> 4);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const int c = k >> 2, kk = k & 3;
                    tc::mma_f16_warp(tmem, dQ + (uint64_t)((c * BM * 128 + kk * 32) >> 4),
                                     b0 + (uint64_t)((c * BN * 128 + kk * 32) >> 4), IQK, k > 0 ? 1u : 0u);
                }
                tc::commit_warp(s_full);
                tc::commit_warp(k_empty + st);
                return true;
            };
            bool ok = true;
            int64_t g = 0;
            for (int n = 0; ok; ++n) {
                const Item it = take_item(n, ok);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok || it.seq < 0) break;
                ok = __all_sync(0xffffffffu, mbar_wait(q_full, n & 1)) && issue_s(g);
                for (int j = 0; j < it.nkv && ok; ++j) {
                    const int64_t gg = g + j;
                    if (j + 1 < it.nkv) {
                        ok = issue_s(gg + 1);
                        if (!ok) break;
                    } else {
                        tc::commit_warp(q_empty); // the item's last S has been issued: Q may be replaced
                    }
                    const int sv = (int)(gg % NVS);
                    ok = __all_sync(0xffffffffu, mbar_wait(p_full + (gg & 1), (gg >> 1) & 1) && mbar_wait(v_full + sv, (gg / NVS) & 1));
                    // the epilogue of the previous item has read O out of TMEM
                    if (ok && j == 0 && n >= 1) ok = __all_sync(0xffffffffu, mbar_wait(o_free, (n - 1) & 1));
                    if (!ok) break;
                    tc::fence_after_sync();
                    // O += P V, P (A operand) read from tensor memory where the softmax left it
                    const uint32_t a0 = tmem + (uint32_t)(BN + (int)(gg % L::NPB) * (BN / 2));
                    const uint64_t b0 = dV + (uint64_t)((sv * L::KV_BYTES) >> 4);
#pragma unroll
                    for (int part = 0; part < L::NP; ++part)
#pragma unroll
                        for (int k = 0; k < BN / 16; ++k)
                            tc::mma_f16_ts_warp(tO, a0 + (uint32_t)(part * (BN / 2) + k * 8), b0 + (uint64_t)((k * 2048) >> 4),
                                                IPV, (j > 0 || k > 0 || part > 0) ? 1u : 0u);
                    tc::commit_warp(t_full + (gg & 1));
                    tc::commit_warp(v_empty + sv);
                }
                g += it.nkv;
                if (lane == 0) mbar_arrive(item_empty + (n & 1));
                if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            }
            if (!ok && lane == 0) fail();
            // every MMA issued by the elected lane has completed before TMEM is released (a CTA that found
            // no item issued none and has nothing to wait for)
            if (any_mma) {
                tc::commit_warp(fin);
                if (!__all_sync(0xffffffffu, mbar_wait(fin, 0)) && lane == 0) set_error(a.err, PKV_DEVERR_TIMEOUT);
            }
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ softmax, one thread per row
        const int lw = warp & 3;
        const int r = lw * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(lw * 32) << 16;
        bool ok = true;
        int64_t g = 0;
        for (int n = 0; ok; ++n) {
            Item it = take_item(n, ok);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok || it.seq < 0) break;
            // absolute positions: row r of the item sits at c0 + q0 + r (c0 = 0 without a cached prefix)
            const int q0 = it.c0 + it.q0, qpos = it.q0 + r;
            float m_use = -INFINITY, l = 0.f;
            for (int j = 0; j < it.nkv && ok; ++j) {
                const int64_t gg = g + j;
                ok = __all_sync(0xffffffffu, mbar_wait(s_full, gg & 1));
                if (!ok) break;
                tc::fence_after_sync();
                uint32_t sr[64];
                {
                    uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
                    uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
                    tc::ld32(tmem + lane_off, lo);
                    tc::ld32(tmem + lane_off + 32, hi);
                }
                tc::wait_ld();
                tc::fence_before_sync();
                mbar_arrive(s_free); // the S buffer may take the next tile
                const int kbase = it.k0 + j * BN;
                if constexpr (CASCADE) {
                    // every query sees the whole prefix: only keys past its end are masked
                    if (kbase + BN > it.kend) {
                        const int lim = it.kend - kbase;
#pragma unroll
                        for (int c = 0; c < BN; ++c)
                            if (c >= lim) sr[c] = 0xFF800000u; // -inf
                    }
                } else if (kbase + BN - 1 > q0) {
                    // causal mask, only on tiles that reach past the item's first query row
                    const int lim = q0 + r - kbase + 1; // keys c < lim are at or before this row
#pragma unroll
                    for (int c = 0; c < BN; ++c)
                        if (c >= lim) sr[c] = 0xFF800000u; // -inf
                }
                float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
                for (int c = 0; c < BN; c += 4) {
                    mx0 = max3(mx0, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
                    mx1 = max3(mx1, __uint_as_float(sr[c + 2]), __uint_as_float(sr[c + 3]));
                }
                const float mx = fmaxf(mx0, mx1) * a.scale_log2; // scale > 0 keeps the order
                const bool up = mx > m_use + kRescale;
                const float m_new = up ? mx : m_use;
                const float alpha = up ? fast_exp2(m_use - m_new) : 1.f;
                m_use = m_new;
                const float nbase = m_use == -INFINITY ? 0.f : -m_use; // a row with no live key yet keeps p = 0
                float2 rs = make_float2(0.f, 0.f);
                const float2 sc2 = make_float2(a.scale_log2, a.scale_log2), nb2 = make_float2(nbase, nbase);
                uint32_t phi[BN / 2], plo[L::NP == 2 ? BN / 2 : 1];
#pragma unroll
                for (int c = 0; c < BN / 2; ++c) {
                    const float2 x = fma2(make_float2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sc2, nb2);
                    const float p0 = fast_exp2(x.x), p1 = fast_exp2(x.y);
                    rs = add2(rs, make_float2(p0, p1));
                    phi[c] = pack2(p0, p1, MT);
                    if constexpr (L::NP == 2) // remainders after bf16 rounding, themselves rounded to bf16
                        plo[c] = pack2(p0 - __uint_as_float(phi[c] << 16), p1 - __uint_as_float(phi[c] & 0xFFFF0000u), MT);
                }
                l = l * alpha + (rs.x + rs.y);
                // P V of the previous tile must have finished when O is rescaled (only when a row's
                // base moved) and, with a single P buffer, before P is overwritten.  The wait is
                // unambiguous: S of this tile is done, hence P V of tile gg - 2 (issued before it), and
                // P V of tile gg + 1 cannot start before this thread's later p_full arrivals.  With two
                // P buffers, the one of tile gg was last read by P V of tile gg - 2, already done.  At
                // j = 0 the previous item's epilogue has waited for its last P V.
                const bool moved = __any_sync(0xffffffffu, up);
                if (j > 0 && (L::NPB == 1 || moved)) {
                    ok = __all_sync(0xffffffffu, mbar_wait(t_full + ((gg - 1) & 1), ((gg - 1) >> 1) & 1));
                    if (!ok) break;
                    tc::fence_after_sync();
                }
                if (j > 0 && moved) {
#pragma unroll
                    for (int cc = 0; cc < D / 16; ++cc) {
                        uint32_t o[16];
                        tc::ld16(tmem + lane_off + 2 * BN + cc * 16, o);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc::st16(tmem + lane_off + 2 * BN + cc * 16, o);
                    }
                }
                // P into its tensor-memory buffer: packed pairs, key c in column c / 2
                const uint32_t pcol = (uint32_t)(BN + (int)(gg % L::NPB) * (BN / 2));
                tc::st32(tmem + lane_off + pcol, phi);
                if constexpr (L::NP == 2) tc::st32(tmem + lane_off + pcol + BN / 2, plo);
                tc::wait_st();
                tc::fence_before_sync();
                mbar_arrive(p_full + (gg & 1));
            }
            g += it.nkv;
            // the commit after P V of the item's last tile covers every earlier MMA as well
            if (ok) ok = __all_sync(0xffffffffu, mbar_wait(t_full + ((g - 1) & 1), ((g - 1) >> 1) & 1));
            if (!ok) break;
            tc::fence_after_sync();
            const float inv = 1.f / l;
            using T = typename ModelT<MT>::T;
            if constexpr (CASCADE) {
                // fp32 partial of (sequence it.start + qpos, head it.h, split it.qt): unnormalised o and
                // (m, l) with m the row's exponent base in log2 units, as the split merge expects
                const int64_t idx = ((int64_t)(it.start + qpos) * a.hq + it.h) * a.max_splits + it.qt;
                float *wo = a.ws_o + idx * D;
#pragma unroll
                for (int cc = 0; cc < D / 16; ++cc) {
                    uint32_t o[16];
                    tc::ld16(tmem + lane_off + 2 * BN + cc * 16, o);
                    tc::wait_ld();
                    if (qpos < it.n) {
                        float4 *dst = reinterpret_cast<float4 *>(wo + cc * 16);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_float4(__uint_as_float(o[4 * e]), __uint_as_float(o[4 * e + 1]),
                                                 __uint_as_float(o[4 * e + 2]), __uint_as_float(o[4 * e + 3]));
                    }
                }
                if (qpos < it.n) reinterpret_cast<float2 *>(a.ws_ml)[idx] = make_float2(m_use, l);
            } else {
                T *orow = static_cast<T *>(a.out) + ((int64_t)(it.start + qpos) * a.hq + it.h) * D;
#pragma unroll
                for (int cc = 0; cc < D / 16; ++cc) {
                    uint32_t o[16];
                    tc::ld16(tmem + lane_off + 2 * BN + cc * 16, o);
                    tc::wait_ld();
                    uint32_t w[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        w[e] = pack2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv, MT);
                    if (qpos < it.n) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 16);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
            }
            tc::fence_before_sync();
            mbar_arrive(o_free); // O has been read out; the next item's first P V may overwrite it
            __syncwarp();
            if (lane == 0) mbar_arrive(item_empty + (n & 1));
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        }
        if (!ok) fail();
    } else {
        // ------------------------------------------------------------ paged K/V write of the item's rows
        // The item's own rows q0..qlast are the keys of its last K/V tiles (q0/BN .. nkv-1).  This
        // warp follows every K tile and every V tile of the rings in order (so a stage's phase is
        // never more than one ahead of it) and holds each stage until it is done with it: a stage
        // frees only after the MMA that reads it and this warp.  K and V are released independently,
        // so a K stage never waits for its V tile to land.  Whole blocks of the item's rows leave
        // shared memory as tiled TMA stores (one lane per block; one box of bs rows x 64 dims per
        // half of D, the 128-byte swizzle undone by the copy engine) into their (block, K|V, head)
        // tile of the pool; the rows of a partly filled last block (a sequence whose length is not a
        // multiple of bs) go out as plain 16-byte stores, so no slot past the sequence is touched.
        // The block-table entries of the item's rows are read once, at the start of the item.
        constexpr int CPR = D / 8;   // 16-byte chunks per row
        constexpr int RPI = 32 / CPR; // rows per warp instruction
        const int cc = lane % CPR, rsub = lane / CPR;
        const int c2 = cc >> 3, u = cc & 7;
        if (lane == 0) tc::prefetch_tmap(&tp);
        bool ok = true;
        int64_t g = 0;
        for (int n = 0; ok; ++n) {
            const Item it = take_item(n, ok);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok || it.seq < 0) break;
            const bool writes = !PAGED && it.h % G == 0; // paged mode: the K/V were appended before
            const int kvh = it.h / G, lb0 = it.q0 >> a.lg_bs;
            // lane l: table entry of logical block lb0 + l (at most BM / bs <= 16 of them)
            int blkv = -1;
            {
                const int lb = lb0 + lane;
                if (writes && (lb << a.lg_bs) <= it.qlast && lb < a.max_blocks)
                    blkv = a.tables[(int64_t)it.seq * a.max_blocks + lb];
            }
            // the item's rows of tile j, from `src` (a K or a V stage) into the K (kv = 0) or V half
            auto write_tile = [&](int j, const uint8_t *src, int kv) {
                const int lo = max(j * BN, it.q0), hi = min(j * BN + BN - 1, it.qlast);
                if (lo > hi) return;
                const int bfirst = lo >> a.lg_bs;            // lo is a multiple of bs
                const int nfull = (hi + 1 - lo) >> a.lg_bs;  // whole blocks among the rows
                {
                    const int lb = bfirst + lane;
                    const int blk = __shfl_sync(0xffffffffu, blkv, min(lb - lb0, 31));
                    if (lane < nfull) {
                        if (blk < 0 || blk >= a.num_blocks) {
                            set_error(a.err, PKV_DEVERR_BLOCK_ID);
                        } else {
                            const uint8_t *box = src + ((lb << a.lg_bs) - j * BN) * 128;
                            const int y = ((blk * 2 + kv) * a.hkv + kvh) << a.lg_bs;
#pragma unroll
                            for (int c = 0; c < D / 64; ++c) tc::tma_store_2d(&tp, c * 64, y, box + c * BN * 128);
                            tc::bulk_commit();
                        }
                    }
                }
                for (int p0 = lo + (nfull << a.lg_bs); p0 <= hi; p0 += RPI) { // fewer than bs rows
                    const int p = p0 + rsub;
                    const int lb = p >> a.lg_bs;
                    const int blk = __shfl_sync(0xffffffffu, blkv, min(lb - lb0, 31));
                    if (p > hi) continue;
                    if (blk < 0 || blk >= a.num_blocks) {
                        if (cc == 0) set_error(a.err, PKV_DEVERR_BLOCK_ID);
                        continue;
                    }
                    const int r = p - j * BN;
                    const int sw = c2 * BN * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((u ^ (r & 7)) << 4);
                    const uint4 x = *reinterpret_cast<const uint4 *>(src + sw);
                    const int64_t dst = ((int64_t)(blk * 2 + kv) * a.hkv + kvh) * a.tile_elems +
                                        (int64_t)(p - (lb << a.lg_bs)) * D + cc * 8;
                    *reinterpret_cast<uint4 *>(a.pool + dst * 2) = x;
                }
                tc::bulk_wait_read_all(); // the stores have read the stage; it may be released
            };
            for (int j = 0; j < it.nkv && ok; ++j) {
                const int64_t gg = g + j;
                const bool mine = writes && j >= it.q0 / BN;
                const int sk = (int)(gg % NKS), sv = (int)(gg % NVS);
                ok = __all_sync(0xffffffffu, mbar_wait(k_full + sk, (gg / NKS) & 1));
                if (!ok) break;
                if (mine) write_tile(j, smem + L::K0 + sk * L::KV_BYTES, 0);
                __syncwarp();
                if (lane == 0) mbar_arrive(k_empty + sk);
                ok = __all_sync(0xffffffffu, mbar_wait(v_full + sv, (gg / NVS) & 1));
                if (!ok) break;
                if (mine) write_tile(j, smem + L::V0 + sv * L::KV_BYTES, 1);
                __syncwarp();
                if (lane == 0) mbar_arrive(v_empty + sv);
            }
            if (!ok) break;
            g += it.nkv;
            if (lane == 0) mbar_arrive(item_empty + (n & 1));
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        }
        tc::bulk_wait_all(); // the pool writes have completed before the CTA exits
        if (!ok && lane == 0) fail();
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
    if constexpr (CASCADE) pdl_wait(); // the grid completes after the suffix decode (see above)
}

using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
    static EncodeFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeFn>(p);
    });
    return fn;
}

// 2-D view [rows = tokens][cols = heads * D] of a packed tensor; box = 64 columns x box_rows rows.
// mt = PKV_FP8_E4M3: one-byte elements, boxes of 128 columns (one 128-byte swizzle row).
bool make_map(CUtensorMap *m, const void *base, int mt, int64_t rows, int64_t cols, int box_rows) {
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    const bool bytes = mt == PKV_FP8_E4M3;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * (bytes ? 1 : 2)};
    const cuuint32_t box[2] = {bytes ? 128u : 64u, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = bytes                ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : mt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUresult r = enc(m, dt, 2,
                           const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, int MT, int MODE>
cudaError_t launch_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tp,
                     const Args &a, int64_t max_ctas, int num_sms, cudaStream_t st) {
    auto kern = prefill_kernel<D, MT, MODE>;
    const int smem = Layout<D, MT>::TOTAL;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    // all of the unified L1/shared array as shared memory: two CTAs of ~113 KB then fit an SM
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    // resident CTAs per SM: what the launch bounds and the shared-memory size were chosen for (the
    // occupancy query answers 1 here, though two CTAs of this size do run side by side on an SM)
    int per_sm = min_blocks<D, MT>();
    if (const char *v = std::getenv("PAGEDKV_PREFILL_CTAS")) {
        // resident CTAs per SM, for tuning sweeps (persistent CTAs beyond what fits simply run later)
        const int x = std::atoi(v);
        if (x > 0 && x <= 4) per_sm = x;
    }
    const int64_t grid = std::min<int64_t>(max_ctas, (int64_t)num_sms * std::max(per_sm, 1));
    return pdl_launch(kern, dim3((unsigned)grid), dim3(kThreads), smem, st, tq, tk, tv, tp, a);
}

cudaError_t launch_plan(const Args &a, cudaStream_t st) {
    const int smem = (2 * (a.nqt_max + 1) + 32) * (int)sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return pdl_launch(plan_kernel, dim3(1), dim3(kPlanThreads), smem, st, a);
}

} // namespace pkv_prefill

bool pkv_tmap_2d(CUtensorMap *m, const void *base, int mt, int64_t rows, int64_t cols, int box_rows) {
    return pkv_prefill::make_map(m, base, mt, rows, cols, box_rows);
}

bool pkv_tmap_rows128_grouped(CUtensorMap *m, const void *base, int mt, int64_t rows, int box_rows) {
    using namespace pkv_prefill;
    EncodeFn enc = encode_fn();
    if (!enc || rows % 8 || box_rows % 8 || box_rows > 256 * 8) return false;
    // rows of 128 16-bit elements = 256 bytes, seen as (64 elements, row in its group of 8, half, group):
    // a box of (64, 8, 2, box_rows / 8) lands as [group][half][8 rows][128 bytes]
    const cuuint64_t dims[4] = {64, 8, 2, (cuuint64_t)(rows / 8)};
    const cuuint64_t strides[3] = {256, 128, 2048};
    const cuuint32_t box[4] = {64u, 8u, 2u, (cuuint32_t)(box_rows / 8)};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    const CUtensorMapDataType dt = mt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUresult r = enc(m, dt, 4, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

cudaError_t launch_prefill(pkv_cache *c, const PrefillLaunch &p, cudaStream_t st) {
    using namespace pkv_prefill;
    if (p.total_tokens <= 0) return cudaSuccess;
    const int D = c->head_dim;
    const int mt = c->model_dtype;
    Args a;
    a.k = static_cast<const char *>(p.k);
    a.v = static_cast<const char *>(p.v);
    a.out = p.out;
    a.cu = p.cu;
    a.ctx = p.ctx;
    a.tables = p.tables;
    a.pool = static_cast<char *>(c->pool);
    a.err = c->err;
    a.total_tokens = p.total_tokens;
    a.num_blocks = c->num_blocks;
    a.tile_elems = (int64_t)c->block_size * D;
    a.num_seqs = p.num_seqs;
    a.max_seqlen = p.max_seqlen;
    a.max_blocks = p.max_blocks;
    a.hq = p.num_q_heads;
    a.hkv = c->num_kv_heads;
    a.bs = c->block_size;
    a.lg_bs = 0;
    while ((1 << a.lg_bs) < c->block_size) ++a.lg_bs;
    a.nqt_max = (p.max_seqlen + BM - 1) / BM;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    // (sequence, query tile) items: sum_i ceil(n_i / BM) <= T / BM + num_seqs
    const int64_t items = std::min<int64_t>((int64_t)a.nqt_max * p.num_seqs, p.total_tokens / BM + p.num_seqs);
    if (items == 0) return cudaSuccess;
    if (items * p.num_q_heads > 0x7FFFFFFF) return cudaErrorNotSupported;
    // the plan kernel's two rank arrays live in shared memory
    if ((2 * ((int64_t)a.nqt_max + 1) + 32) * (int64_t)sizeof(int) > 200 * 1024) return cudaErrorNotSupported;
    const int64_t plan_bytes = (4 + 2 * items) * (int64_t)sizeof(int);
    if (plan_bytes > c->plan_bytes) {
        if (c->plan) cudaFree(c->plan);
        c->plan = nullptr;
        c->plan_bytes = 0;
        cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&c->plan), (size_t)plan_bytes);
        if (e != cudaSuccess) {
            c->plan = nullptr;
            return e;
        }
        c->plan_bytes = plan_bytes;
    }
    a.plan = c->plan;
    // the pool as rows [(block, K|V, head, slot)][D] for the tiled stores of whole blocks; row
    // coordinates are 32-bit
    const int64_t pool_rows = c->num_blocks * 2 * c->num_kv_heads * c->block_size;
    if (pool_rows > 0x7FFFFFFFLL) return cudaErrorNotSupported;
    CUtensorMap tq, tk, tv, tp;
    if (!make_map(&tq, p.q, mt, p.total_tokens, (int64_t)p.num_q_heads * D, BM) ||
        !make_map(&tk, p.k, mt, p.total_tokens, (int64_t)c->num_kv_heads * D, BN) ||
        !make_map(&tv, p.v, mt, p.total_tokens, (int64_t)c->num_kv_heads * D, BN) ||
        !make_map(&tp, c->pool, mt, pool_rows, D, c->block_size))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (p.ctx) {
        // a cached prefix: the new tokens' K/V go to their slots first, then attention reads every
        // key through the block table
        e = launch_append_ranges(c, p.k, p.v, p.tables, p.num_seqs, p.max_blocks, p.cu, p.ctx, p.total_tokens, st);
        if (e != cudaSuccess) return e;
    }
    PkvTimer timer(c, PKV_KIND_PREFILL, st);
    e = launch_plan(a, st);
    g_pkv_launches++;
    if (e != cudaSuccess) return e;
    const int64_t max_ctas = items * p.num_q_heads;
    const int mode = p.ctx != nullptr ? MODE_PAGED : MODE_PACKED;
    e = cudaErrorInvalidValue;
#define PKV_PREFILL_CASE(DD, MM, MO) \
    if (D == DD && mt == MM && mode == MO) e = launch_t<DD, MM, MO>(tq, tk, tv, tp, a, max_ctas, c->num_sms, st);
    PKV_PREFILL_CASE(128, PKV_F16, MODE_PACKED)
    PKV_PREFILL_CASE(128, PKV_BF16, MODE_PACKED)
    PKV_PREFILL_CASE(64, PKV_F16, MODE_PACKED)
    PKV_PREFILL_CASE(64, PKV_BF16, MODE_PACKED)
    PKV_PREFILL_CASE(128, PKV_F16, MODE_PAGED)
    PKV_PREFILL_CASE(128, PKV_BF16, MODE_PAGED)
    PKV_PREFILL_CASE(64, PKV_F16, MODE_PAGED)
    PKV_PREFILL_CASE(64, PKV_BF16, MODE_PAGED)
#undef PKV_PREFILL_CASE
    g_pkv_launches++;
    return e;
}

int cascade_split_tokens(const pkv_cache *c, int num_seqs, int num_q_heads, int prefix_tokens) {
    using namespace pkv_prefill;
    if (const char *v = std::getenv("PAGEDKV_CASCADE_SPLIT_TOKENS")) {
        // keys per prefix split, for tuning sweeps (rounded up to whole 64-key tiles)
        const int x = std::atoi(v);
        if (x > 0) return (x + 63) / 64 * 64;
    }
    // The prefix phase runs as one wave of items where it can: as many splits per (query-row tile,
    // head) as leave every item a resident CTA (a split past one wave makes the whole phase wait for
    // a second), each of at least 256 keys so that an item's fixed costs (Q load, epilogue, partial
    // write) stay small next to its key tiles, in whole 64-key tiles.
    int per_sm = 1;
    if (c->head_dim == 128)
        per_sm = c->model_dtype == PKV_BF16 ? min_blocks<128, PKV_BF16>() : min_blocks<128, PKV_F16>();
    else
        per_sm = c->model_dtype == PKV_BF16 ? min_blocks<64, PKV_BF16>() : min_blocks<64, PKV_F16>();
    const int64_t slots = (int64_t)c->num_sms * per_sm;
    const int64_t rows = (int64_t)((num_seqs + BM - 1) / BM) * num_q_heads;
    const int64_t nps = std::max<int64_t>(1, slots / std::max<int64_t>(rows, 1));
    int64_t split = (prefix_tokens + nps - 1) / nps;
    split = std::max<int64_t>(split, 256);
    return (int)((split + 63) / 64 * 64);
}

cudaError_t launch_cascade_prefix(pkv_cache *c, const CascadePrefixLaunch &p, cudaStream_t st, int part) {
    using namespace pkv_prefill;
    if (p.num_seqs <= 0 || p.prefix_tokens <= 0) return cudaSuccess;
    const int D = c->head_dim;
    const int mt = c->model_dtype;
    Args a;
    a.k = a.v = nullptr;
    a.out = nullptr;
    a.cu = nullptr;
    a.ctx = nullptr;
    a.tables = p.tables;
    a.pool = static_cast<char *>(c->pool);
    a.err = c->err;
    a.total_tokens = p.num_seqs;
    a.num_blocks = c->num_blocks;
    a.tile_elems = (int64_t)c->block_size * D;
    a.num_seqs = p.num_seqs;
    a.max_seqlen = 0;
    a.max_blocks = p.max_blocks;
    a.hq = p.num_q_heads;
    a.hkv = c->num_kv_heads;
    a.bs = c->block_size;
    a.lg_bs = 0;
    while ((1 << a.lg_bs) < c->block_size) ++a.lg_bs;
    a.nqt_max = 0;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    a.ws_o = p.ws_o;
    a.ws_ml = p.ws_ml;
    a.max_splits = p.max_splits;
    a.prefix_tokens = p.prefix_tokens;
    a.split_tokens = p.split_tokens;
    a.nps = (p.prefix_tokens + p.split_tokens - 1) / p.split_tokens;
    const int64_t pairs = (int64_t)((p.num_seqs + BM - 1) / BM) * a.nps;
    if (pairs * p.num_q_heads > 0x7FFFFFFF) return cudaErrorNotSupported;
    if (c->plan_bytes < 16) {
        if (c->plan) cudaFree(c->plan);
        c->plan = nullptr;
        c->plan_bytes = 0;
        cudaError_t e = cudaMalloc(reinterpret_cast<void **>(&c->plan), 64);
        if (e != cudaSuccess) return e;
        c->plan_bytes = 64;
    }
    a.plan = c->plan;
    const int64_t pool_rows = c->num_blocks * 2 * c->num_kv_heads * c->block_size;
    if (pool_rows > 0x7FFFFFFFLL) return cudaErrorNotSupported;
    // q [S][Hq][D] as rows of sequences: a box of 128 sequences x 64 dims of one head
    CUtensorMap tq, tp;
    if (!make_map(&tq, p.q, mt, p.num_seqs, (int64_t)p.num_q_heads * D, BM) ||
        !make_map(&tp, c->pool, mt, pool_rows, D, c->block_size))
        return cudaErrorInvalidValue;
    cudaError_t e;
    if (part == 1) {
        e = launch_plan(a, st);
        g_pkv_launches++;
        return e;
    }
    e = cudaErrorInvalidValue;
    if (D == 128)
        e = mt == PKV_BF16 ? launch_t<128, PKV_BF16, MODE_CASCADE>(tq, tp, tp, tp, a, pairs * p.num_q_heads, c->num_sms, st)
                           : launch_t<128, PKV_F16, MODE_CASCADE>(tq, tp, tp, tp, a, pairs * p.num_q_heads, c->num_sms, st);
    else
        e = mt == PKV_BF16 ? launch_t<64, PKV_BF16, MODE_CASCADE>(tq, tp, tp, tp, a, pairs * p.num_q_heads, c->num_sms, st)
                           : launch_t<64, PKV_F16, MODE_CASCADE>(tq, tp, tp, tp, a, pairs * p.num_q_heads, c->num_sms, st);
    g_pkv_launches++;
    return e;
}
