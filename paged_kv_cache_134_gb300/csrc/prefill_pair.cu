// Packed causal prefill, two query tiles per CTA ("Paged KV Cache 与 Packed Sequence", discosf.com,
// sections 3.1-3.3 and 4.2): the same attention and the same paged K/V write as prefill.cu's packed
// mode, organised so that one SM keeps two independent softmax chains in flight on one K/V stream.
//
// Work item = (sequence, pair of consecutive 128-row query tiles A and B, query head).  Both tiles
// read the same K/V tiles of 128 keys; tile A needs the key tiles 0 .. 2p, tile B 0 .. 2p + 1 (the
// diagonal tile of each is masked per element, no tile above a diagonal is computed).  One CTA per
// SM, persistent, taking items from the heaviest-first work list of a one-CTA plan kernel.
//
// Tensor memory (512 columns): S_A [0,128), S_B [128,256), O_A [256, 256 + D), O_B [384, 384 + D).
// P (fp16) is written over the first 64 columns of its S buffer once the row has been read: the
// MMAs of one issuing thread run in issue order, so the next S, issued after the P V that reads P,
// cannot overwrite P early.  The MMA warp issues, per key tile j:
//     [P_A(j) ready] P V_A(j), S_A(j + 1)     [P_B(j) ready] P V_B(j), S_B(j + 1)
// so that the softmax warps of one tile work while the tensor pipe runs the other tile's MMAs.
// S = Q K^T is M = 128, N = 128 (8 KB of shared memory per 64-cycle MMA, the shared-memory rate);
// P V takes P from tensor memory.
//
// Warps: 0 scheduler + Q + K loads (lane 0), 1 MMA issuer (converged warp, elected lane), 2-5
// softmax of tile A, 6-9 softmax of tile B (one thread per query row, the row's TMEM lane), 10 V
// loads (lane 0), 11 paged K/V writer of the item's own rows (whole blocks by tiled TMA stores,
// a partly filled last block row by row).  Every mbarrier wait is bounded; a timeout sets
// PKV_DEVERR_TIMEOUT and the CTA winds down.  fp16 models only (bf16 models keep P as a hi + lo
// pair, which does not fit in the S columns; they run prefill.cu's kernel).
#include <algorithm>
#include <cstdlib>

#include "tcgen05.cuh"
#include "pkv_internal.h"

namespace pkv_prefill_pair {

constexpr int BM = 128;        // query rows per tile (MMA M)
constexpr int BN = 128;        // keys per tile (MMA N of Q K^T, K of P V)
constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t TS_A = 0, TS_B = 128, TO_A = 256, TO_B = 384; // tensor-memory columns
constexpr float kRescale = 8.0f;  // log2 units
constexpr int NKS = 2, NVS = 3;   // K and V stages
constexpr int kItemConsumers = 11; // MMA, 8 softmax warps, V loader, writer
constexpr int kStageReleasers = 2; // a K or V stage frees after the MMAs that read it and the writer
constexpr int kPlanThreads = 1024;

struct Args {
    const char *k, *v;  // packed [T][Hkv][D]
    void *out;          // packed [T][Hq][D]
    const int32_t *cu, *tables;
    char *pool;
    unsigned int *err;
    int *plan;          // [0] item count, [1] next-item counter, [4 + 2i], [5 + 2i] = (sequence, pair) of item i
    int64_t total_tokens, num_blocks, tile_elems;
    int num_seqs, max_seqlen, max_blocks, hq, hkv, bs, lg_bs, npr_max;
    float scale_log2;
};

template <int D>
struct Layout {
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2; // one K or V tile: [D / 64][128 rows][128 B]
    static constexpr int QA = 0, QB = QA + Q_BYTES;
    static constexpr int K0 = QB + Q_BYTES;
    static constexpr int V0 = K0 + NKS * KV_BYTES;
    static constexpr int BAR = V0 + NVS * KV_BYTES;
    static constexpr int TOTAL = BAR + 512; // mbarriers, the TMEM slot, a flag, two 16-byte item slots
};

// two floats -> packed fp16 pair (round-to-nearest-even), `lo` in the low half
PKV_DEV uint32_t pack_h2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// query-tile pairs of sequence i (0 for a malformed cu_seqlens entry, which is reported)
PKV_DEV int seq_pairs(const Args &a, int i, bool report) {
    const int st = a.cu[i], en = a.cu[i + 1];
    if (st < 0 || en < st || en > a.total_tokens || en - st > a.max_seqlen) {
        if (report) set_error(a.err, PKV_DEVERR_CU_SEQLENS);
        return 0;
    }
    const int nqt = (en - st + BM - 1) / BM;
    return (nqt + 1) / 2;
}

// in-place inclusive prefix sum of x[0, n) by the whole CTA (kPlanThreads threads)
PKV_DEV void cta_scan(int *x, int n, int *warp_sums) {
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

// The work list: rank r holds every sequence's r-th heaviest pair (its (np - 1 - r)-th, the
// heavier the later in the sequence).  With gt[r] = #{i : np_i > r} items in rank r, rank r starts
// at gt[0] + ... + gt[r - 1]; inside a rank the order is whatever the atomics give (it only decides
// which CTA computes an item).  Also resets the next-item counter.
__global__ void __launch_bounds__(kPlanThreads) plan_pairs_kernel(const Args a) {
    extern __shared__ int sh[];
    const int R = a.npr_max + 1;
    int *hist = sh, *cnt = sh + R, *warp_sums = sh + 2 * R;
    pdl_trigger();
    pdl_wait();
    for (int x = threadIdx.x; x < R; x += kPlanThreads) {
        hist[x] = 0;
        cnt[x] = 0;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < a.num_seqs; i += kPlanThreads) atomicAdd(&hist[min(seq_pairs(a, i, true), a.npr_max)], 1);
    __syncthreads();
    cta_scan(hist, R, warp_sums); // hist[r] = #{i : np_i <= r}
    for (int x = threadIdx.x; x < R; x += kPlanThreads) hist[x] = a.num_seqs - hist[x];
    __syncthreads();
    cta_scan(hist, R, warp_sums); // hist[r] = gt[0] + ... + gt[r]
    int2 *list = reinterpret_cast<int2 *>(a.plan + 4);
    for (int i = threadIdx.x; i < a.num_seqs; i += kPlanThreads) {
        const int np = min(seq_pairs(a, i, false), a.npr_max);
        for (int r = 0; r < np; ++r) {
            const int pos = (r > 0 ? hist[r - 1] : 0) + atomicAdd(&cnt[r], 1);
            list[pos] = make_int2(i, np - 1 - r);
        }
    }
    if (threadIdx.x == 0) {
        a.plan[0] = hist[R - 1];
        a.plan[1] = 0;
    }
}

// one item as the roles see it
struct Item {
    int seq, pr, h;  // seq < 0: no more items
    int start, n;    // the sequence's packed rows [start, start + n)
    int qa0;         // first row of tile A (tile B starts at qa0 + BM)
    bool has_b;
    int nkva, nkvb;  // key tiles of tile A (0 .. nkva - 1) and of tile B (0 if none)
    int nkv;         // key tiles the item loads: max(nkva, nkvb)
    int qlast;       // the item's last row
};

PKV_DEV Item make_item(const Args &a, int seq, int pr, int h) {
    Item it;
    it.seq = seq;
    it.pr = pr;
    it.h = h;
    if (seq < 0) return it;
    it.start = a.cu[seq];
    it.n = a.cu[seq + 1] - it.start;
    it.qa0 = pr * 2 * BM;
    it.has_b = it.qa0 + BM < it.n;
    it.nkva = 2 * pr + 1;
    it.nkvb = it.has_b ? 2 * pr + 2 : 0;
    it.nkv = it.has_b ? it.nkvb : it.nkva;
    it.qlast = min(it.qa0 + 2 * BM, it.n) - 1;
    return it;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tp, const Args a) {
    using L = Layout<D>;
    extern __shared__ __align__(1024) uint8_t smem[];

    pdl_trigger();
    if (smem_u32(smem) & 1023u) return; // the swizzled tiles need 1024-byte alignment (always true)

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR);
    // Q tile A / B loaded, and free again once the item's last S of that tile is done (per item)
    uint64_t *qa_full = bars + 0, *qa_empty = bars + 1, *qb_full = bars + 2, *qb_empty = bars + 3;
    uint64_t *k_full = bars + 4, *k_empty = k_full + NKS;      // [NKS] each
    uint64_t *v_full = k_empty + NKS, *v_empty = v_full + NVS; // [NVS] each
    // per tile of A (of B), counted over all items: S done, P written, P V done
    uint64_t *sa_full = v_empty + NVS, *sb_full = sa_full + 1;
    uint64_t *pa_full = sb_full + 1, *pb_full = pa_full + 1;
    uint64_t *ta_full = pb_full + 1, *tb_full = ta_full + 1;
    // per item: O of tile A (B) read out by the epilogue (B: also when the item has no tile B)
    uint64_t *oa_free = tb_full + 1, *ob_free = oa_free + 1;
    uint64_t *item_full = ob_free + 1, *item_empty = item_full + 2, *fin = item_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(fin + 2);
    volatile int4 *item_slot = reinterpret_cast<volatile int4 *>(bars + 30); // [2], 16-byte aligned

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(qa_full, 1);
        mbar_init(qa_empty, 1);
        mbar_init(qb_full, 1);
        mbar_init(qb_empty, 1);
        for (int s = 0; s < NKS; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(k_empty + s, kStageReleasers);
        }
        for (int s = 0; s < NVS; ++s) {
            mbar_init(v_full + s, 1);
            mbar_init(v_empty + s, kStageReleasers);
        }
        mbar_init(sa_full, 1);
        mbar_init(sb_full, 1);
        mbar_init(pa_full, 128);
        mbar_init(pb_full, 128);
        mbar_init(ta_full, 1);
        mbar_init(tb_full, 1);
        mbar_init(oa_free, 128);
        mbar_init(ob_free, 128);
        for (int s = 0; s < 2; ++s) {
            mbar_init(item_full + s, 1);
            mbar_init(item_empty + s, kItemConsumers);
        }
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
    // kernels on the stream (the work list, the inputs) is read
    pdl_wait();

    const int G = a.hq / a.hkv;
    auto fail = [&]() {
        set_error(a.err, PKV_DEVERR_TIMEOUT);
        *abort_flag = 1;
    };
    // the item in ring slot n % 2, once the scheduler has published it
    auto take_item = [&](int n, bool &ok) -> Item {
        ok = mbar_wait_sleep(item_full + (n & 1), (n >> 1) & 1);
        if (!ok) return make_item(a, -1, 0, 0);
        return make_item(a, item_slot[n & 1].x, item_slot[n & 1].y, item_slot[n & 1].z);
    };

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------------------ scheduler, Q and K loads
            tc::prefetch_tmap(&tq);
            tc::prefetch_tmap(&tk);
            const int total = a.plan[0] * a.hq;
            int n = 0, last_q = -1;
            int64_t g = 0; // K tiles issued so far (all items)
            bool ok = true;
            for (;; ++n) {
                const int s = n & 1;
                if (n >= 2 && !mbar_wait_sleep(item_empty + s, ((n >> 1) - 1) & 1)) {
                    ok = false;
                    break;
                }
                const int idx = *abort_flag ? total : atomicAdd(a.plan + 1, 1);
                int4 raw = make_int4(-1, 0, 0, 0);
                if (idx < total) {
                    const int2 sp = reinterpret_cast<const int2 *>(a.plan + 4)[idx / a.hq];
                    raw = make_int4(sp.x, sp.y, idx % a.hq, 0);
                }
                item_slot[s].x = raw.x;
                item_slot[s].y = raw.y;
                item_slot[s].z = raw.z;
                mbar_arrive(item_full + s);
                if (raw.x < 0) break;
                const Item it = make_item(a, raw.x, raw.y, raw.z);
                const int kvh = it.h / G;
                // both Q tiles, tile B also when the item has none (its rows are then those of the next
                // sequence or out of range and zero-filled; nothing reads them), so that the Q
                // barriers count items
                if (n >= 1 && !(mbar_wait_sleep(qa_empty, (n - 1) & 1) && mbar_wait_sleep(qb_empty, (n - 1) & 1))) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(qa_full, L::Q_BYTES);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tc::tma_load_2d(smem + L::QA + c * BM * 128, &tq, it.h * D + c * 64, it.start + it.qa0, qa_full);
                mbar_arrive_expect_tx(qb_full, L::Q_BYTES);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tc::tma_load_2d(smem + L::QB + c * BM * 128, &tq, it.h * D + c * 64, it.start + it.qa0 + BM,
                                    qb_full);
                last_q = n;
                for (int j = 0; j < it.nkv; ++j) {
                    const int64_t gg = g + j;
                    const int st = (int)(gg % NKS);
                    const int64_t round = gg / NKS;
                    if (round >= 1 && !mbar_wait_sleep(k_empty + st, (round - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    if (*abort_flag) break;
                    mbar_arrive_expect_tx(k_full + st, L::KV_BYTES);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tc::tma_load_2d(smem + L::K0 + st * L::KV_BYTES + c * BN * 128, &tk, kvh * D + c * 64,
                                        it.start + j * BN, k_full + st);
                }
                if (!ok || *abort_flag) break;
                g += it.nkv;
            }
            if (!ok) fail();
            // the last loads must land before this CTA's shared memory goes away
            for (int64_t gg = g > NKS ? g - NKS : 0; gg < g; ++gg)
                if (!mbar_wait_sleep(k_full + gg % NKS, (gg / NKS) & 1)) set_error(a.err, PKV_DEVERR_TIMEOUT);
            // the Q loads of the last item loaded (the earlier ones were waited for by the MMA warp
            // before it released their buffers)
            if (last_q >= 0 && !(mbar_wait_sleep(qa_full, last_q & 1) && mbar_wait_sleep(qb_full, last_q & 1)))
                set_error(a.err, PKV_DEVERR_TIMEOUT);
        }
    } else if (warp == 10) {
        if (lane == 0) {
            // ------------------------------------------------------------ V loads
            tc::prefetch_tmap(&tv);
            int64_t g = 0;
            bool ok = true;
            for (int n = 0;; ++n) {
                const Item it = take_item(n, ok);
                if (!ok || it.seq < 0) break;
                const int kvh = it.h / G;
                for (int j = 0; j < it.nkv && ok; ++j) {
                    const int64_t gg = g + j;
                    const int st = (int)(gg % NVS);
                    const int64_t round = gg / NVS;
                    if (round >= 1) ok = mbar_wait_sleep(v_empty + st, (round - 1) & 1);
                    if (!ok || *abort_flag) break;
                    mbar_arrive_expect_tx(v_full + st, L::KV_BYTES);
#pragma unroll
                    for (int c = 0; c < D / 64; ++c)
                        tc::tma_load_2d(smem + L::V0 + st * L::KV_BYTES + c * BN * 128, &tv, kvh * D + c * 64,
                                        it.start + j * BN, v_full + st);
                }
                if (!ok || *abort_flag) break;
                g += it.nkv;
                mbar_arrive(item_empty + (n & 1));
            }
            if (!ok) fail();
            for (int64_t gg = g > NVS ? g - NVS : 0; gg < g; ++gg)
                if (!mbar_wait_sleep(v_full + gg % NVS, (gg / NVS) & 1)) set_error(a.err, PKV_DEVERR_TIMEOUT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // the whole warp runs the issue loop in step (waits agreed with __all_sync); one elected lane
        // issues each MMA and commit
        constexpr uint32_t IQK = tc::idesc_f16(0u, 0u, BM, BN); // fp16, A = Q and B = K both K-major
        constexpr uint32_t IPV = tc::idesc_f16(0u, 1u, BM, D);  // fp16, A = P (tensor memory), B = V MN-major
        // one descriptor per operand; the address field counts 16-byte units, so a tile at byte
        // offset `off` is the base descriptor plus off / 16
        const uint64_t dQA = tc::smem_desc(smem_u32(smem + L::QA), 16, 1024);
        const uint64_t dQB = tc::smem_desc(smem_u32(smem + L::QB), 16, 1024);
        const uint64_t dK = tc::smem_desc(smem_u32(smem + L::K0), 16, 1024);
        const uint64_t dV = tc::smem_desc(smem_u32(smem + L::V0), BN * 128, 1024);
        bool any_mma = false;
        // S = Q K^T of key tile in K stage ks into the S buffer at column ts
        auto issue_s = [&](uint32_t ts, uint64_t dq, int ks) {
            const uint64_t b0 = dK + (uint64_t)((ks * L::KV_BYTES) >> 4);
#pragma unroll
            for (int k = 0; k < D / 16; ++k) {
                const int c = k >> 2, kk = k & 3;
                tc::mma_f16_warp(tmem + ts, dq + (uint64_t)((c * BM * 128 + kk * 32) >> 4),
                                 b0 + (uint64_t)((c * BN * 128 + kk * 32) >> 4), IQK, k > 0 ? 1u : 0u);
            }
        };
        // O += P V of the key tile in V stage vs, P (the A operand) in tensor memory at column ts
        auto issue_pv = [&](uint32_t to, uint32_t ts, int vs, bool first) {
            const uint64_t b0 = dV + (uint64_t)((vs * L::KV_BYTES) >> 4);
#pragma unroll
            for (int k = 0; k < BN / 16; ++k)
                tc::mma_f16_ts_warp(tmem + to, tmem + ts + (uint32_t)(k * 8), b0 + (uint64_t)((k * 2048) >> 4), IPV,
                                    (!first || k > 0) ? 1u : 0u);
        };
        auto wait_all = [&](uint64_t *bar, uint32_t parity) { return __all_sync(0xffffffffu, mbar_wait_sleep(bar, parity)); };
        bool ok = true;
        int64_t g = 0, ta = 0, tb = 0; // K/V tiles, A tiles and B tiles so far (all items)
        for (int n = 0; ok; ++n) {
            const Item it = take_item(n, ok);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok || it.seq < 0) break;
            // both Q tiles in place and the first key tile: S_A(0), S_B(0)
            ok = wait_all(qa_full, n & 1) && wait_all(qb_full, n & 1) && wait_all(k_full + (int)(g % NKS), (g / NKS) & 1);
            if (!ok) break;
            tc::fence_after_sync();
            any_mma = true;
            issue_s(TS_A, dQA, (int)(g % NKS));
            tc::commit_warp(sa_full);
            if (it.nkva == 1) tc::commit_warp(qa_empty); // Q_A has no later use in this item
            if (it.has_b) {
                issue_s(TS_B, dQB, (int)(g % NKS));
                tc::commit_warp(sb_full);
            } else {
                tc::commit_warp(qb_empty);
            }
            tc::commit_warp(k_empty + (int)(g % NKS));
            for (int j = 0; j < it.nkv && ok; ++j) {
                const int64_t gg = g + j;
                const int vs = (int)(gg % NVS), ks1 = (int)((gg + 1) % NKS);
                ok = wait_all(v_full + vs, (gg / NVS) & 1);
                if (!ok) break;
                bool k1 = false; // key tile j + 1 has landed (waited for once)
                if (j < it.nkva) {
                    // O_A += P_A(j) V(j), then S_A(j + 1) over P_A (it runs after that P V)
                    ok = wait_all(pa_full, (uint32_t)((ta + j) & 1));
                    if (ok && j == 0 && n >= 1) ok = wait_all(oa_free, (n - 1) & 1);
                    if (!ok) break;
                    tc::fence_after_sync();
                    issue_pv(TO_A, TS_A, vs, j == 0);
                    tc::commit_warp(ta_full);
                    if (j + 1 < it.nkva) {
                        ok = wait_all(k_full + ks1, ((gg + 1) / NKS) & 1);
                        if (!ok) break;
                        k1 = true;
                        tc::fence_after_sync();
                        issue_s(TS_A, dQA, ks1);
                        tc::commit_warp(sa_full);
                        if (j + 2 == it.nkva) tc::commit_warp(qa_empty);
                    }
                }
                if (j < it.nkvb) {
                    ok = wait_all(pb_full, (uint32_t)((tb + j) & 1));
                    if (ok && j == 0 && n >= 1) ok = wait_all(ob_free, (n - 1) & 1);
                    if (!ok) break;
                    tc::fence_after_sync();
                    issue_pv(TO_B, TS_B, vs, j == 0);
                    tc::commit_warp(tb_full);
                    if (j + 1 < it.nkvb) {
                        if (!k1) ok = wait_all(k_full + ks1, ((gg + 1) / NKS) & 1);
                        if (!ok) break;
                        tc::fence_after_sync();
                        issue_s(TS_B, dQB, ks1);
                        tc::commit_warp(sb_full);
                        if (j + 2 == it.nkvb) tc::commit_warp(qb_empty);
                    }
                }
                tc::commit_warp(v_empty + vs);
                if (j + 1 < it.nkv) tc::commit_warp(k_empty + ks1);
            }
            if (!ok) break;
            g += it.nkv;
            ta += it.nkva;
            tb += it.nkvb;
            if (lane == 0) mbar_arrive(item_empty + (n & 1));
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        }
        if (!ok && lane == 0) fail();
        // every MMA issued by the elected lane has completed before tensor memory is released
        if (any_mma) {
            tc::commit_warp(fin);
            if (!__all_sync(0xffffffffu, mbar_wait_sleep(fin, 0)) && lane == 0) set_error(a.err, PKV_DEVERR_TIMEOUT);
        }
    } else if (warp < 10) {
        // ------------------------------------------------------------ softmax, one thread per query row
        const bool tile_b = warp >= 6; // warps 2-5: tile A, 6-9: tile B
        const int lw = warp & 3;
        const int r = lw * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(lw * 32) << 16;
        const uint32_t ts = tmem + lane_off + (tile_b ? TS_B : TS_A);
        const uint32_t to = tmem + lane_off + (tile_b ? TO_B : TO_A);
        uint64_t *s_full = tile_b ? sb_full : sa_full, *p_full = tile_b ? pb_full : pa_full;
        uint64_t *t_full = tile_b ? tb_full : ta_full, *o_free = tile_b ? ob_free : oa_free;
        bool ok = true;
        int64_t t0 = 0; // this tile's key tiles so far (all items)
        for (int n = 0; ok; ++n) {
            const Item it = take_item(n, ok);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok || it.seq < 0) break;
            const int nk = tile_b ? it.nkvb : it.nkva;
            const int q0 = it.qa0 + (tile_b ? BM : 0); // the tile's first row (= its diagonal key tile's first key)
            float m_use = -INFINITY, l = 0.f;
            for (int j = 0; j < nk && ok; ++j) {
                const int64_t t = t0 + j;
                ok = __all_sync(0xffffffffu, mbar_wait_sleep(s_full, (uint32_t)(t & 1)));
                if (!ok) break;
                tc::fence_after_sync();
                // the diagonal key tile (the last one) keeps keys c <= r of the row; the others are whole
                const bool diag = j + 1 == nk;
                // One pass over S in two halves of 64 keys (two TMEM loads in flight per wait).  Each
                // half's maximum is checked against the row's base first; P = exp2(scale s - base) goes
                // out as fp16 pairs over the S columns already read (P of half hp takes columns
                // [32 hp, 32 hp + 32), inside S half hp).  The base moves only when a score passes it by
                // more than kRescale; the P already written (values <= 2^kRescale, finite in fp16) is
                // then scaled to the new base.
                const float m_start = m_use;
                float2 rs = make_float2(0.f, 0.f);
                const float2 sc2 = make_float2(a.scale_log2, a.scale_log2);
#pragma unroll
                for (int hp = 0; hp < BN / 64; ++hp) {
                    uint32_t s[64];
                    {
                        uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[0]);
                        uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32]);
                        tc::ld32(ts + hp * 64, s0);
                        tc::ld32(ts + hp * 64 + 32, s1);
                    }
                    tc::wait_ld();
                    if (diag) {
#pragma unroll
                        for (int c = 0; c < 64; ++c)
                            if (hp * 64 + c > r) s[c] = 0xFF800000u; // -inf: p = 0
                    }
                    float cm0 = -INFINITY, cm1 = -INFINITY;
#pragma unroll
                    for (int c = 0; c < 64; c += 4) {
                        cm0 = max3(cm0, __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
                        cm1 = max3(cm1, __uint_as_float(s[c + 2]), __uint_as_float(s[c + 3]));
                    }
                    const float cms = fmaxf(cm0, cm1) * a.scale_log2; // scale > 0 keeps the order
                    const bool move = cms > m_use + kRescale;          // false while cms = -inf
                    if (__any_sync(0xffffffffu, move)) {
                        const float mn = move ? cms : m_use;
                        const float al = move ? fast_exp2(m_use - mn) : 1.f; // 0 from a base of -inf
                        if (hp > 0) {
#pragma unroll
                            for (int c2 = 0; c2 < 2; ++c2) {
                                uint32_t pw[16];
                                tc::ld16(ts + c2 * 16, pw);
                                tc::wait_ld();
#pragma unroll
                                for (int e = 0; e < 16; ++e) {
                                    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&pw[e]));
                                    pw[e] = pack_h2(f.x * al, f.y * al);
                                }
                                tc::st16(ts + c2 * 16, pw);
                            }
                        }
                        rs.x *= al;
                        rs.y *= al;
                        m_use = mn;
                    }
                    const float nbase = m_use == -INFINITY ? 0.f : -m_use; // a row with no live key keeps p = 0
                    const float2 nb2 = make_float2(nbase, nbase);
                    uint32_t pp[32];
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float2 x = fma2(make_float2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), sc2, nb2);
                        const float2 pv = make_float2(fast_exp2(x.x), fast_exp2(x.y));
                        rs = add2(rs, pv);
                        pp[c] = pack_h2(pv.x, pv.y);
                    }
                    tc::st32(ts + hp * 32, pp);
                }
                const bool up = m_use != m_start;
                const float alpha = up ? fast_exp2(m_start - m_use) : 1.f; // 0 from a base of -inf
                l = l * alpha + (rs.x + rs.y);
                // O is rescaled when a row's base moved, after P V of the previous key tile is done (that
                // wait is unambiguous: P V of key tile t + 1 needs this thread's next P)
                if (j > 0 && __any_sync(0xffffffffu, up)) {
                    ok = __all_sync(0xffffffffu, mbar_wait_sleep(t_full, (uint32_t)((t - 1) & 1)));
                    if (!ok) break;
                    tc::fence_after_sync();
#pragma unroll
                    for (int cc = 0; cc < D / 16; ++cc) {
                        uint32_t o[16];
                        tc::ld16(to + cc * 16, o);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc::st16(to + cc * 16, o);
                    }
                }
                tc::wait_st();
                tc::fence_before_sync();
                mbar_arrive(p_full);
            }
            if (!ok) break;
            if (nk > 0) {
                // ---- epilogue: O / l of the tile's rows inside the sequence, after its last P V
                t0 += nk;
                ok = __all_sync(0xffffffffu, mbar_wait_sleep(t_full, (uint32_t)((t0 - 1) & 1)));
                if (!ok) break;
                tc::fence_after_sync();
                const float inv = 1.f / l;
                const int qrow = q0 + r;
                __half *orow = static_cast<__half *>(a.out) + ((int64_t)(it.start + qrow) * a.hq + it.h) * D;
#pragma unroll
                for (int cc = 0; cc < D / 16; ++cc) {
                    uint32_t o[16];
                    tc::ld16(to + cc * 16, o);
                    tc::wait_ld();
                    uint32_t w[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) w[e] = pack_h2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv);
                    if (qrow < it.n) {
                        uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 16);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                    }
                }
                tc::fence_before_sync();
            }
            // O may take the next item's first P V (for an item without tile B: at once)
            mbar_arrive(o_free);
            __syncwarp();
            if (lane == 0) mbar_arrive(item_empty + (n & 1));
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        }
        if (!ok) fail();
    } else {
        // ------------------------------------------------------------ paged K/V write of the item's rows
        // The item's rows qa0 .. qlast are the keys of its last key tiles (qa0 / BN .. nkv - 1).  This
        // warp follows every K tile and every V tile of the rings in order and holds each stage until
        // it is done with it (a stage frees after the MMAs that read it and this warp).  Whole blocks
        // leave shared memory as tiled TMA stores into their (block, K|V, head) tile of the pool (one
        // lane per block, one box of bs rows x 64 dims per half of D); the rows of a partly filled last
        // block go out as 16-byte stores, so no slot past the sequence is touched.  Only items of the
        // first query head of each KV group write, so every (token, KV head) is written once.
        constexpr int CPR = D / 8;    // 16-byte chunks per row
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
            const bool writes = it.h % G == 0;
            const int kvh = it.h / G, lb0 = it.qa0 >> a.lg_bs;
            // lane l: table entry of logical block lb0 + l (the item's 256 rows span at most 32 blocks)
            int blkv = -1;
            {
                const int lb = lb0 + lane;
                if (writes && (lb << a.lg_bs) <= it.qlast && lb < a.max_blocks)
                    blkv = a.tables[(int64_t)it.seq * a.max_blocks + lb];
            }
            // the item's rows of key tile j, from `src` (a K or a V stage) into the K (kv = 0) or V half
            auto write_tile = [&](int j, const uint8_t *src, int kv) {
                const int lo = max(j * BN, it.qa0), hi = min(j * BN + BN - 1, it.qlast);
                if (lo > hi) return;
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
                    const int rr = p - j * BN;
                    const int sw = c2 * BN * 128 + (rr >> 3) * 1024 + (rr & 7) * 128 + ((u ^ (rr & 7)) << 4);
                    const uint4 x = *reinterpret_cast<const uint4 *>(src + sw);
                    const int64_t dst = ((int64_t)(blk * 2 + kv) * a.hkv + kvh) * a.tile_elems +
                                        (int64_t)(p - (lb << a.lg_bs)) * D + cc * 8;
                    *reinterpret_cast<uint4 *>(a.pool + dst * 2) = x;
                }
                tc::bulk_wait_read_all(); // the stores have read the stage; it may be released
            };
            for (int j = 0; j < it.nkv && ok; ++j) {
                const int64_t gg = g + j;
                const bool mine = writes && j >= it.qa0 / BN;
                const int sk = (int)(gg % NKS), sv = (int)(gg % NVS);
                ok = __all_sync(0xffffffffu, mbar_wait_sleep(k_full + sk, (gg / NKS) & 1));
                if (!ok) break;
                if (mine) write_tile(j, smem + L::K0 + sk * L::KV_BYTES, 0);
                __syncwarp();
                if (lane == 0) mbar_arrive(k_empty + sk);
                ok = __all_sync(0xffffffffu, mbar_wait_sleep(v_full + sv, (gg / NVS) & 1));
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
}

template <int D>
cudaError_t launch_kernel(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &tp,
                          const Args &a, int64_t items, int num_sms, cudaStream_t st) {
    auto kern = prefill_pair_kernel<D>;
    const int smem = Layout<D>::TOTAL;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    const int64_t grid = std::min<int64_t>(items, num_sms);
    return pdl_launch(kern, dim3((unsigned)grid), dim3(kThreads), smem, st, tq, tk, tv, tp, a);
}

} // namespace pkv_prefill_pair

bool pkv_prefill_pair_eligible(const pkv_cache *c, const PrefillLaunch &p) {
    if (p.ctx != nullptr || c->model_dtype != PKV_F16) return false;
    if (c->head_dim != 64 && c->head_dim != 128) return false;
    const char *v = std::getenv("PAGEDKV_PREFILL_PAIRS");
    return !(v && v[0] == '0');
}

cudaError_t launch_prefill_pair(pkv_cache *c, const PrefillLaunch &p, cudaStream_t st) {
    using namespace pkv_prefill_pair;
    if (p.total_tokens <= 0) return cudaSuccess;
    const int D = c->head_dim;
    Args a;
    a.k = static_cast<const char *>(p.k);
    a.v = static_cast<const char *>(p.v);
    a.out = p.out;
    a.cu = p.cu;
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
    a.npr_max = ((p.max_seqlen + BM - 1) / BM + 1) / 2;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    // (sequence, pair) items: sum_i ceil(ceil(n_i / BM) / 2) <= T / (2 BM) + num_seqs
    const int64_t items = std::min<int64_t>((int64_t)a.npr_max * p.num_seqs, p.total_tokens / (2 * BM) + p.num_seqs);
    if (items == 0) return cudaSuccess;
    if (items * p.num_q_heads > 0x7FFFFFFF) return cudaErrorNotSupported;
    if ((2 * ((int64_t)a.npr_max + 1) + 32) * (int64_t)sizeof(int) > 200 * 1024) return cudaErrorNotSupported;
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
    const int64_t pool_rows = c->num_blocks * 2 * c->num_kv_heads * c->block_size;
    if (pool_rows > 0x7FFFFFFFLL) return cudaErrorNotSupported;
    CUtensorMap tq, tk, tv, tp;
    if (!pkv_tmap_2d(&tq, p.q, PKV_F16, p.total_tokens, (int64_t)p.num_q_heads * D, BM) ||
        !pkv_tmap_2d(&tk, p.k, PKV_F16, p.total_tokens, (int64_t)c->num_kv_heads * D, BN) ||
        !pkv_tmap_2d(&tv, p.v, PKV_F16, p.total_tokens, (int64_t)c->num_kv_heads * D, BN) ||
        !pkv_tmap_2d(&tp, c->pool, PKV_F16, pool_rows, D, c->block_size))
        return cudaErrorInvalidValue;
    PkvTimer timer(c, PKV_KIND_PREFILL, st);
    const int plan_smem = (2 * (a.npr_max + 1) + 32) * (int)sizeof(int);
    cudaError_t e = cudaFuncSetAttribute(plan_pairs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, plan_smem);
    if (e != cudaSuccess) return e;
    e = pdl_launch(plan_pairs_kernel, dim3(1), dim3(kPlanThreads), plan_smem, st, a);
    g_pkv_launches++;
    if (e != cudaSuccess) return e;
    const int64_t total_items = items * p.num_q_heads;
    e = D == 128 ? launch_kernel<128>(tq, tk, tv, tp, a, total_items, c->num_sms, st)
                 : launch_kernel<64>(tq, tk, tv, tp, a, total_items, c->num_sms, st);
    g_pkv_launches++;
    return e;
}
