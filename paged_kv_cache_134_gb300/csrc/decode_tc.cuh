// Paged decode attention for grouped-query heads on the 5th-generation tensor cores.
//
// What it computes is the decode of "PagedAttention 与前缀缓存" (2kiu.com, section 2.3), the same
// as decode_impl.cuh: for sequence s and query head h, softmax(scale q.K_t) weighted sum of V_t
// over the L_s tokens of the sequence, token t in physical block block_table[s][t / bs] at offset
// t % bs, query head h reading KV head h / G.  With G query heads per KV head every K/V element
// meets G queries, so the CUDA-core kernel runs out of issue slots long before HBM runs out of
// bandwidth; here the two contractions go to tcgen05 instead, transposed so that the token axis
// fills the MMA's M = 128 rows:
//   S^T [128 tokens x 16] = K [128 tokens x D] . Q^T [D x 16]      (heads padded from G to 16)
//   O^T [D x 16]         += V^T [D x 128 tokens] . P^T [128 tokens x 16]
// K and V come straight from the paged pool by tiled TMA (16-bit caches: one box of bs rows x 64
// dims per block and half of D, 128-byte swizzle), landing in the K-major layout the first MMA
// reads as A and the MN-major layout the second MMA reads as A.  E4M3 caches: one box per block
// brings its K and its V codes together (the SM issues copies one after another, so a step's copy
// count, not its bytes, set the pace); K is read by the MMA as it lands and V is widened to fp16 by
// converter warps.  Q sits in shared memory K-major, P is written there by the softmax threads.
// Accumulators live in tensor memory.
//
// Work unit = (sequence, KV head, split of up to split_blocks blocks), the same unit list as the
// CUDA-core kernel (full splits first), round-robin over one persistent CTA per SM.  A unit is
// processed in steps of 128 tokens.  Roles:
//   warp 0     loads: block-table entries (read a unit ahead into registers, one lane per block of
//              the step), Q of the unit, and the K boxes of every block into a ring of 3 K stages
//              (E4M3: the K + V boxes into a ring of 4 code stages);
//   warp 6     the same walk for the V boxes (ring of 3 V stages); each ring has a second loader
//              taking the odd steps: warps 11 (K) and 12 (V), or for E4M3 caches warp 6 (codes);
//   warps 11-14 (E4M3) q to three E4M3 terms, V codes widened into a ring of 2 fp16 V stages;
//   warp 1     tensor-memory owner and MMA issuer (one thread);
//   warps 2-5  one thread per token row of S^T (a TMEM lane): mask, scale, tile max over the 128
//              rows (shuffles + shared memory), online softmax with a lazily moved base (the base
//              changes only when a head's max grows by more than 2^8, exact algebra), P written to
//              shared memory (fp16; bf16 models as hi + lo so that P keeps ~16 bits); rows that are
//              masked get their V row zeroed so that no NaN from an unused slot reaches the MMA;
//              at the end of a unit one thread per dimension reads O^T and writes the output row
//              (one split) or the fp32 partial (m, l, o) for the split merge.
// Every mbarrier wait is bounded; a timeout sets PKV_DEVERR_TIMEOUT and the CTA winds down.
#pragma once

#include "decode_impl.cuh"
#include "tcgen05.cuh"

namespace pkv_decode_tc {

using pkv_decode::Args;
using pkv_decode::Unit;

constexpr int D = 128;
constexpr int TOK = 128;             // tokens per step: MMA M of S^T, MMA K of O^T
constexpr int NQ = 16;               // MMA N: the group's query heads, padded
// warp 0 Q and K loads, 1 MMA, 2-5 softmax, 6 V loads, 7-10 epilogue; 16-bit caches: 11 and 12
// second K and V loaders (odd steps); FP8 caches: 11-14 converters
template <bool F8>
__host__ __device__ constexpr int threads_for() {
    return F8 ? 480 : 416;
}
constexpr uint32_t kTmemCols = 128;  // two S^T buffers, then O^T of even and odd units (see NSC, OB)
constexpr float kRescale = 8.0f;     // log2 units
constexpr int kUnitRing = 16;        // unit records published by the K loader (see UnitRec)

// One work unit as the K loader publishes it for the other roles, which would otherwise each
// repeat the (sequence, head, split) lookup at every unit boundary on their critical paths.  The
// loader publishes unit n once it has issued the K loads of unit n - 1; the last of those waited
// for the S^T four steps back, which waited for the softmax to release the scores six steps back,
// so the softmax warps are within six units and the other roles within a few more (the epilogue
// two units behind the softmax): a ring of 16 is never overwritten before it is read.
struct UnitRec {
    int s, kvh, j, blk0, ntiles, nsplit;
    int tok_end; // first token past the unit: min(sequence length, end of its last block)
    float ksc;   // the KV head's K scale (FP8 caches)
    int tag;     // the unit's index in this CTA's order, written last
    int pad[7];
};

template <int MT, bool F8 = false>
struct Layout {
    // K stages and V stages.  16-bit caches: three of each, K and V loaded by their own copies.  E4M3
    // caches: four code stages, each holding the K and the V codes of a step as they land (one copy per
    // block brings both), and two stages of V widened to fp16 for the P V MMA
    static constexpr int NS = F8 ? 4 : 3;
    static constexpr int NSV = F8 ? 2 : 3;
    static constexpr int NP = MT == PKV_BF16 ? 2 : 1;      // P parts (hi, lo for bf16)
    // rows of the P^T operand: the group's heads (padded to NQ), and for bf16 the lo parts as rows
    // NQ.. 2 NQ - 1, so that one N = 2 NQ MMA per K step covers both parts (the two O^T column
    // groups are added in the epilogue)
    static constexpr int NPR = NQ * NP;
    static constexpr int STAGE = TOK * D * 2;              // V (and 16-bit K): [half][128 rows][128 B] = 32 KB
    static constexpr int KSTAGE = STAGE;                   // E4M3: [row group][K, V][8 rows][128 B] = 32 KB
    static constexpr int K0 = 0;
    static constexpr int V0 = K0 + NS * KSTAGE;
    static constexpr int Q = V0 + NSV * STAGE;             // [2 buffers][half][16 rows][128 B]
    static constexpr int Q_BYTES = NQ * D * 2;
    static constexpr int P = Q + 2 * Q_BYTES;                  // [buffer][part][64-token chunk][16 rows][128 B]
    static constexpr int P_BYTES = NPR * TOK * 2;          // one buffer
    static constexpr int RED = P + 2 * P_BYTES;            // [2][4 warps][NQ] maxima, [2][4 warps][NQ] sums,
    static constexpr int BAR = RED + (4 * 4 * NQ + 2 * NQ) * 4; // [2][NQ] bases (sums and bases per unit parity)
    static constexpr int UNITS = BAR + 640;                // ring of kUnitRing unit records
    static constexpr int FIXED = UNITS + kUnitRing * 64;   // + unit tables, 3 (S + 1) ints
};

inline size_t smem_bytes(int mt, bool f8, int num_seqs) {
    const size_t fixed = f8 ? Layout<PKV_F16, true>::FIXED
                            : (mt == PKV_BF16 ? Layout<PKV_BF16>::FIXED : Layout<PKV_F16>::FIXED);
    return fixed + (size_t)3 * (num_seqs + 1) * sizeof(int);
}

// one packed pair of the model dtype from two floats (round-to-nearest-even), `lo` in the low half
template <int MT>
PKV_DEV uint32_t pack2(float lo, float hi) {
    uint32_t r;
    if constexpr (MT == PKV_BF16)
        asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    else
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// The unit lookup of the CUDA-core kernel, done by a whole warp: each search round tests 32 rows
// at once and keeps the bracket of the last row whose prefix is <= k, so a few hundred sequences
// take two rounds of independent shared-memory reads instead of a chain of dependent ones.  All
// 32 lanes call it with the same arguments.
PKV_DEV int find_row_warp(const int *pref, int n, int k, int lane) {
    // largest i in [0, n) with pref[i] <= k (pref non-decreasing, pref[0] = 0 <= k)
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) >> 5;
        const int i = lo + lane * step;
        const unsigned le = __ballot_sync(0xffffffffu, i < hi && pref[i] <= k);
        lo += (31 - __clz(le)) * step; // lane 0 always passes: pref[lo] <= k
        hi = min(hi, lo + step);
    }
    return lo;
}

static __device__ __noinline__ Unit unit_info_warp(int u, const int *pf, const int *pp, const int *nb, int S, int hkv, int bps, int sb,
                            int lane) {
    Unit r;
    const int nfull_units = pf[S] * hkv;
    if (u < nfull_units) {
        const int k = u / hkv;
        r.kvh = u - k * hkv;
        r.s = find_row_warp(pf, S, k, lane);
        r.j = k - pf[r.s];
        r.blk0 = sb + r.j * bps;
        r.ntiles = bps;
    } else {
        const int k = (u - nfull_units) / hkv;
        r.kvh = (u - nfull_units) - k * hkv;
        r.s = find_row_warp(pp, S, k, lane);
        r.j = pf[r.s + 1] - pf[r.s];
        r.blk0 = sb + r.j * bps;
        r.ntiles = nb[r.s] - r.blk0;
    }
    r.nsplit = (pf[r.s + 1] - pf[r.s]) + (pp[r.s + 1] - pp[r.s]);
    return r;
}

// wait (bounded) until a unit record's tag reads n
static __device__ __noinline__ bool wait_tag(const volatile int *tag, int n) {
    const uint64_t t0 = global_timer_ns();
    while (*tag != n)
        if (global_timer_ns() - t0 > PKV_WAIT_LIMIT_NS) return false;
    return true;
}

// byte offset of element (row g, token t) in a P buffer of NPR rows: K-major, 128-byte swizzle,
// 64-token chunks
template <int NPR>
PKV_DEV int p_offset(int g, int t) {
    const int e = t & 63;
    return (t >> 6) * (NPR * 128) + (g >> 3) * 1024 + (g & 7) * 128 + ((((e >> 3) ^ (g & 7))) << 4) + ((e & 7) << 1);
}

template <int G, int MT, int KVT>
__global__ void __launch_bounds__(threads_for<KVT == PKV_FP8_E4M3>(), 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tkv, const __grid_constant__ CUtensorMap tq, const Args a) {
    // FP8 caches: S^T = K q^T is an E4M3 x E4M3 MMA (K as stored, q as three E4M3 terms with a
    // power-of-two scale); P V runs on fp16 operands (V widened exactly from E4M3, P in fp16); the
    // per-head K and V scales fold into the softmax scale and the epilogue
    constexpr bool F8 = KVT == PKV_FP8_E4M3;
    constexpr int OT = F8 ? (int)PKV_F16 : MT; // operand dtype of the MMAs
    constexpr int kThreads = threads_for<F8>();
    using LY = Layout<OT, F8>;
    constexpr int NS = LY::NS;
    // tensor-memory columns: two S^T buffers of NSC columns (FP8: q as three E4M3 terms of 8 heads
    // each, N = 32), then O^T of even units at OB and of odd units at OB + 32
    constexpr int NSC = F8 ? 32 : NQ;
    constexpr uint32_t OB = 2 * NSC;
    using M = ModelT<MT>;
    using T = typename M::T;
    extern __shared__ __align__(1024) uint8_t smem[];

    const int S = a.num_seqs;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + LY::BAR);
    uint64_t *k_full = bars, *k_empty = bars + NS, *v_full = bars + 2 * NS, *v_empty = bars + 3 * NS;
    uint64_t *s_full = bars + 4 * NS, *s_free = s_full + 2, *p_full = s_full + 4, *t_full = s_full + 6;
    uint64_t *q_full = s_full + 8, *q_empty = s_full + 10;
    // per unit parity: O^T complete / read out of tensor memory; row sums and bases published / read
    uint64_t *o_full = s_full + 12, *o_free = s_full + 14, *l_ready = s_full + 16, *l_free = s_full + 18;
    uint64_t *fin = s_full + 20;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(fin + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(fin + 2);
    // FP8 caches: the exponent of unit nu's q scale in slot nu % 8, published with "Q converted"
    // (q_ready, a ring of 8: unit nu + 8's Q cannot be loaded before the softmax has read the scores
    // of unit nu + 4, so the MMA and the softmax, which wait for unit nu, never see a later phase),
    // and the converters' partial maxima
    volatile int *qexp = reinterpret_cast<volatile int *>(fin + 5);              // [8]
    volatile float *qred = reinterpret_cast<volatile float *>(fin + 9);          // [2 unit parities][4 warps]
    uint64_t *q_ready = fin + 13 + 2 * NS; // [8]
    float *red_max = reinterpret_cast<float *>(smem + LY::RED);                  // [2][4][NQ]
    float *red_sum = red_max + 2 * 4 * NQ;                                      // [2][4][NQ]
    float *m_base = red_sum + 2 * 4 * NQ;                                       // [2][NQ]
    int *pf = reinterpret_cast<int *>(smem + LY::FIXED);
    int *pp = pf + (S + 1);
    int *nb = pp + (S + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(k_full + i, 1); // the TMA arrival (E4M3 K is read by the MMA as is)
            // free once the four softmax warps have read the S^T its K gave (so the MMA has read K) and,
            // E4M3, the four converter warps its V codes: arrivals instead of a commit per step (the
            // MMA warp issues every MMA and commit of a step in a row, and a commit costs about as
            // much as two MMAs)
            mbar_init(k_empty + i, F8 ? 8 : 4);
        }
        for (int i = 0; i < LY::NSV; ++i) {
            mbar_init(v_full + i, F8 ? 128 : 1);  // the converters' rows (E4M3) or the TMA arrival
            mbar_init(v_empty + i, 1);
        }
        if constexpr (F8)
            for (int b = 0; b < 8; ++b) mbar_init(q_ready + b, 128);
        for (int b = 0; b < 2; ++b) {
            mbar_init(s_full + b, 1);
            mbar_init(s_free + b, 128);
            mbar_init(p_full + b, 128);
            mbar_init(t_full + b, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(q_full + b, 1);
            mbar_init(q_empty + b, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(o_full + b, 1);
            mbar_init(o_free + b, 128);
            mbar_init(l_ready + b, 128);
            mbar_init(l_free + b, 128);
        }
        mbar_init(fin, 1);
        *abort_flag = 0;
        fence_mbarrier_init();
    }
    UnitRec *ring = reinterpret_cast<UnitRec *>(smem + LY::UNITS);
    for (int k = threadIdx.x; k < kUnitRing; k += kThreads) ring[k].tag = -1;
    // Q rows past the group stay zero (the MMA's padding heads)
    for (int i = threadIdx.x; i < 2 * LY::Q_BYTES / 16; i += kThreads)
        reinterpret_cast<uint4 *>(smem + LY::Q)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    pdl_wait(); // the previous kernel (e.g. the append of this step) has finished
    const int bps = a.split_blocks;
    pkv_decode::build_unit_list(a, pf, pp, nb, warp, lane);
    const int U = (pf[S] + pp[S]) * a.hkv;
    const int bpstep = TOK / a.bs; // blocks per step
    auto fail = [&]() {
        set_error(a.err, PKV_DEVERR_TIMEOUT);
        *abort_flag = 1;
    };
    // (sequence, KV head, split) of unit u; every lane of the calling warp takes part
    auto unit_at = [&](int u) { return unit_info_warp(u, pf, pp, nb, S, a.hkv, bps, a.start_block, lane); };
    // publish this CTA's n-th unit (one thread of the K loader)
    auto write_rec = [&](int n, const Unit &x, int L, float ks) {
        UnitRec *r = ring + (n % kUnitRing);
        r->s = x.s;
        r->kvh = x.kvh;
        r->j = x.j;
        r->blk0 = x.blk0;
        r->ntiles = x.ntiles;
        r->nsplit = x.nsplit;
        r->tok_end = min(L, (x.blk0 + x.ntiles) * a.bs);
        r->ksc = ks;
        __threadfence_block();
        *reinterpret_cast<volatile int *>(&r->tag) = n;
    };
    // read this CTA's n-th unit once published (every lane waits for the tag itself); false after
    // the wait limit, agreed over the warp
    auto read_rec = [&](int n, Unit &x, int &tok_end, float &ks) -> bool {
        const UnitRec *r = ring + (n % kUnitRing);
        const volatile int *tag = &r->tag;
        const bool okr = __all_sync(0xffffffffu, *tag == n || wait_tag(tag, n));
        __threadfence_block();
        x.s = r->s;
        x.kvh = r->kvh;
        x.j = r->j;
        x.blk0 = r->blk0;
        x.ntiles = r->ntiles;
        x.nsplit = r->nsplit;
        tok_end = r->tok_end;
        ks = r->ksc;
        return okr;
    };

    if (warp == 0 || warp == 6 || (!F8 && (warp == 11 || warp == 12))) {
        // ---------------------------------------------------------------- loads
        // Every ring is filled by two warps taking alternate steps, the first of each pair the even
        // ones: a step's walk (table entries, waits, copy issue, one copy per lane after another)
        // takes about as long as the step's bytes take to arrive, so one warp alone would set the
        // pace.  16-bit caches: warps 0 and 11 the K boxes, 6 and 12 the V boxes; E4M3 caches: a
        // block's box brings its K and its V codes (one copy, not two), warps 0 and 6.  Warp 0 also
        // loads Q of each unit and publishes the unit records the other roles read.  All walk this
        // CTA's steps in the same order, one lane per block of a step.
        const bool boss = warp == 0;                             // Q loads, unit records, look-ahead
        const bool kring = F8 || warp == 0 || warp == 11;        // the K ring (E4M3: code stages) or V
        const int parity = (warp == 0 || (!F8 && warp == 6)) ? 0 : 1; // its steps: even or odd
        const uint64_t policy = l2_policy_evict_first();
        if (lane == 0) tc::prefetch_tmap(&tkv);
        if (lane == 0 && boss) tc::prefetch_tmap(&tq);
        // A unit's block-table entries are read once, a unit ahead, into registers: lane l holds the
        // entries of the unit's blocks l, l + 32, l + 64, l + 96 (a step picks its own with shuffles).
        // A per-step read would leave the loader waiting for it at every step.  Units of more blocks
        // (longer splits set through the tuning variables) read the rest directly.
        constexpr int kER = 4;
        int ecur[kER], enx[kER];
        auto load_entries = [&](const Unit &x, int (&e)[kER]) {
#pragma unroll
            for (int k = 0; k < kER; ++k) {
                const int idx = k * 32 + lane;
                e[k] = idx < x.ntiles ? a.tables[(int64_t)x.s * a.max_blocks + x.blk0 + idx] : 0;
            }
        };
        // table entry of this lane's block in step i of unit `x` (0 for lanes past the step's blocks)
        auto entry = [&](const Unit &x, const int (&e)[kER], int i) -> int {
            const int idx = i * bpstep + lane;
            int v = 0;
#pragma unroll
            for (int k = 0; k < kER; ++k) {
                const int t = __shfl_sync(0xffffffffu, e[k], idx & 31);
                if ((idx >> 5) == k) v = t;
            }
            if (idx >= kER * 32 && idx < x.ntiles) v = a.tables[(int64_t)x.s * a.max_blocks + x.blk0 + idx];
            return lane < min(bpstep, x.ntiles - i * bpstep) ? v : 0;
        };
        int64_t gs = 0; // steps issued so far, all units
        int nu = 0, q_next = 0; // q_next: this CTA's next unit (in its order) whose Q is still to load
        // Q of this CTA's k-th unit `uq` into buffer k % 2 (free once the last S^T of unit k - 2 is issued)
        auto issue_q = [&](int k, const Unit &uq) {
            const int qb = k & 1;
            mbar_arrive_expect_tx(q_full + qb, (uint32_t)(G * D * 2));
#pragma unroll
            for (int c = 0; c < D / 64; ++c)
                tc::tma_load_2d(smem + LY::Q + qb * LY::Q_BYTES + c * NQ * 128, &tq, c * 64, uq.s * a.hq + uq.kvh * G,
                                q_full + qb);
        };
        bool ok = true;
        int u = blockIdx.x, i = 0, nsteps = 0;
        // un: the current unit; nx (K loader): the one after it, looked up when `un` starts, with its
        // length and K scale, which are published a unit later (their loads have landed by then)
        Unit un{}, nx{};
        int nx_len = 0;
        float nx_ks = 1.f;
        auto look_ahead = [&](int uu) {
            if (uu < U) {
                nx = unit_at(uu);
                nx_len = a.lens[nx.s];
                if constexpr (F8) nx_ks = a.k_scale[nx.kvh];
            }
        };
        if (u < U) {
            if (boss) {
                un = unit_at(u);
                if (lane == 0) write_rec(0, un, a.lens[un.s], F8 ? a.k_scale[un.kvh] : 1.f);
                look_ahead(u + (int)gridDim.x);
                if (u + (int)gridDim.x < U) load_entries(nx, enx);
            } else {
                int te;
                float ks;
                ok = read_rec(0, un, te, ks);
            }
            nsteps = (un.ntiles + bpstep - 1) / bpstep;
            if (ok) load_entries(un, ecur);
        }
        while (u < U && ok) {
            if (boss) {
                // this unit's Q is loaded by its first step at the latest (waiting for its buffer); the
                // next unit's goes as soon as its buffer is free, tested at every step without waiting
                const bool first = i == 0 && q_next == nu;
                const bool early = q_next == nu + 1 && u + (int)gridDim.x < U;
                if (lane == 0) {
                    if (first) {
                        if (nu >= 2 && !mbar_wait_sleep(q_empty + (nu & 1), ((nu >> 1) - 1) & 1)) ok = false;
                        if (ok) issue_q(q_next++, un);
                    } else if (early &&
                               (q_next < 2 || mbar_test_wait(q_empty + (q_next & 1), ((q_next >> 1) - 1) & 1))) {
                        issue_q(q_next++, nx);
                    }
                }
                q_next = __shfl_sync(0xffffffffu, q_next, 0);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            // the next step (maybe of the next unit) and its table entries, read ahead
            int u2 = u, i2 = i + 1, nsteps2 = nsteps;
            Unit un2 = un;
            if (i2 >= nsteps) {
                u2 = u + gridDim.x;
                i2 = 0;
                if (u2 < U) {
                    if (boss) {
                        un2 = nx;
                    } else {
                        int te;
                        float ks;
                        if (!read_rec(nu + 1, un2, te, ks)) {
                            ok = false;
                            break;
                        }
                        load_entries(un2, enx); // used from the next step on
                    }
                    nsteps2 = (un2.ntiles + bpstep - 1) / bpstep;
                }
            }
            // this step (E4M3: only every other one is this warp's)
            const bool my_step = (int)(gs & 1) == parity;
            const int st = (int)(gs % NS);
            const int64_t round = gs / NS;
            const int nblk = min(bpstep, un.ntiles - i * bpstep);
            if (my_step) {
                const int b = entry(un, ecur, i);
                const bool good = lane < nblk && b >= 0 && b < a.num_blocks;
                const unsigned goodmask = __ballot_sync(0xffffffffu, good);
                const unsigned bad = __ballot_sync(0xffffffffu, lane < nblk && !good);
                // bs rows of 2 D bytes a block: a 16-bit K or V tile, or an E4M3 K tile and its V tile
                const uint32_t bytes = (uint32_t)__popc(goodmask) * (uint32_t)a.bs * (uint32_t)(2 * D);
                // E4M3: the K codes are read by the MMA as they land; the converters widen the V codes into
                // a V stage of their own
                uint64_t *full = kring ? k_full + st : v_full + st;
                uint64_t *empty = kring ? k_empty + st : v_empty + st;
                if (lane == 0) {
                    if (round >= 1 && !mbar_wait_sleep(empty, (round - 1) & 1)) ok = false;
                    if (ok) {
                        // bad block ids: reported by the V loader (16-bit) or by the step's loader (E4M3)
                        if ((F8 || !kring) && bad) set_error(a.err, PKV_DEVERR_BLOCK_ID);
                        mbar_arrive_expect_tx(full, bytes);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok || *abort_flag) break;
                // 16-bit stage layout: [row group of 8][half][8 rows][128 bytes]; E4M3 code stage:
                // [row group of 8][K, V][8 rows][128 bytes]; a block's bs rows at lane * bs * 256
                uint8_t *dst0 = smem + (kring ? LY::K0 + st * LY::KSTAGE : LY::V0 + st * LY::STAGE) + lane * a.bs * 256;
                if (good) {
                    if constexpr (F8) {
                        // the K and V codes of (block b, KV head), 128-byte swizzled: K in the MMA's K-major layout
                        tc::tma_load_5d_hint(dst0, &tkv, 0, 0, 0, un.kvh * (a.bs >> 3), b, full, policy);
                    } else {
                        // row group of (block b, K or V, KV head) in the pool's [rows][D] view
                        const int row = ((b * 2 + (kring ? 0 : 1)) * a.hkv + un.kvh) * a.bs;
                        tc::tma_load_4d_hint(dst0, &tkv, 0, 0, 0, row / 8, full, policy);
                    }
                }
            }
            ++gs;
            if (i2 == 0) {
                ++nu;
#pragma unroll
                for (int k = 0; k < kER; ++k) ecur[k] = enx[k]; // read a unit ago (warp 0) or a step ago
                if (boss && u2 < U) {
                    // entering unit nu (its Q may still be loading): publish it, look up the next one
                    if (lane == 0) write_rec(nu, un2, nx_len, nx_ks);
                    look_ahead(u2 + (int)gridDim.x);
                    if (u2 + (int)gridDim.x < U) load_entries(nx, enx);
                }
            }
            u = u2;
            i = i2;
            un = un2;
            nsteps = nsteps2;
        }
        if (!ok && lane == 0) fail();
        // the next kernel (the split merge) may start launching once every CTA has issued its last load
        if (boss) pdl_trigger();
        // the copies of the last stages must land before this CTA's shared memory goes away
        if (lane == 0) {
            for (int64_t g = gs > NS ? gs - NS : 0; g < gs; ++g)
                if (!mbar_wait_sleep((kring ? k_full : v_full) + g % NS, (g / NS) & 1))
                    set_error(a.err, PKV_DEVERR_TIMEOUT);
            const int last_q = q_next - 1;
            if (boss)
                for (int n = last_q > 0 ? last_q - 1 : 0; n <= last_q; ++n)
                    if (!mbar_wait_sleep(q_full + (n & 1), (n >> 1) & 1)) set_error(a.err, PKV_DEVERR_TIMEOUT);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------------- MMA issuer
        // the whole warp runs the issue loop in step (waits agreed with __all_sync); one elected lane
        // issues each MMA and commit
        {
            constexpr uint32_t ab = OT == PKV_BF16 ? 1u : 0u;
            // A = K (K-major), B = Q (K-major); FP8: E4M3 x E4M3 (type fields 0) with N = 32
            constexpr uint32_t ISK = tc::idesc_f16_ab(F8 ? 0u : ab, 0u, 0u, TOK, NSC);
            constexpr uint32_t IPV = tc::idesc_f16_ab(ab, 1u, 0u, D, LY::NPR); // A = V^T (MN-major), B = P (K-major)
            // one descriptor per operand layout; the address field counts 16-byte units, so a tile at
            // byte offset `off` from the base is the base descriptor plus off / 16 (shared memory stays
            // below the field's 256 KB): each MMA adds a constant instead of rebuilding its descriptors
            // K: groups of 8 token rows 2048 bytes apart (16-bit: the second 64-dim half of a group sits
            // 1024 bytes after the first; E4M3: the group's V codes do)
            const uint64_t dK = tc::smem_desc(smem_u32(smem + LY::K0), 16, 2048);
            const uint64_t dQ = tc::smem_desc(smem_u32(smem + LY::Q), 16, 1024);
            // V^T (MN-major): the two 64-dim halves LBO apart, groups of 8 tokens SBO apart
            const uint64_t dV = F8 ? tc::smem_desc(smem_u32(smem + LY::V0), TOK * 128, 1024)
                                   : tc::smem_desc(smem_u32(smem + LY::V0), 1024, 2048);
            constexpr int kVStep = F8 ? 2048 : 4096; // bytes per 16 tokens of V
            const uint64_t dP = tc::smem_desc(smem_u32(smem + LY::P), 16, 1024);
            bool any_mma = false;
            // S^T of step g (Q buffer qb) into S buffer g % 2; the K stage is released as soon as S^T is done
            auto issue_s = [&](int64_t g, int qb) -> bool {
                const int st = (int)(g % NS), b = (int)(g & 1);
                if (!__all_sync(0xffffffffu, mbar_wait_sleep(k_full + st, (g / NS) & 1))) return false;
                if (g >= 2 && !__all_sync(0xffffffffu, mbar_wait_sleep(s_free + b, ((g >> 1) - 1) & 1))) return false;
                tc::fence_after_sync();
                any_mma = true;
                const uint64_t a0 = dK + (uint64_t)((st * LY::KSTAGE) >> 4), b0 = dQ + (uint64_t)((qb * LY::Q_BYTES) >> 4);
                if constexpr (F8) {
                    // E4M3 K rows of 128 codes (one swizzle row each) against the q terms, 32 codes a step
#pragma unroll
                    for (int k = 0; k < D / 32; ++k)
                        tc::mma_f8_warp(tmem + b * NSC, a0 + (uint64_t)((k * 32) >> 4), b0 + (uint64_t)((k * 32) >> 4), ISK,
                                        k > 0 ? 1u : 0u);
                } else {
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const int c = k >> 2, kk = k & 3;
                        tc::mma_f16_warp(tmem + b * NSC, a0 + (uint64_t)((c * 1024 + kk * 32) >> 4),
                                         b0 + (uint64_t)((c * (NQ * 128) + kk * 32) >> 4), ISK, k > 0 ? 1u : 0u);
                    }
                }
                tc::commit_warp(s_full + b);
                return true;
            };
            // Q of unit n in place: loaded (q_full), or for FP8 caches converted (q_ready, ring of 8)
            auto q_bar = [&](int n) { return F8 ? q_ready + (n & 7) : q_full + (n & 1); };
            auto q_par = [&](int n) -> uint32_t { return F8 ? (uint32_t)(n >> 3) & 1u : (uint32_t)(n >> 1) & 1u; };
            bool ok = true, ahead = false; // ahead: the unit's first S^T went out during the previous unit
            int64_t gs = 0;
            int nu = 0;
            for (int u = blockIdx.x; u < U && ok; u += gridDim.x, ++nu) {
                Unit un;
                int te;
                float ks;
                if (!read_rec(nu, un, te, ks)) {
                    ok = false;
                    break;
                }
                const int nsteps = (un.ntiles + bpstep - 1) / bpstep;
                const int qb = nu & 1;
                if (!ahead) ok = __all_sync(0xffffffffu, mbar_wait_sleep(q_bar(nu), q_par(nu))) && issue_s(gs, qb);
                ahead = false;
                for (int i = 0; i < nsteps && ok; ++i) {
                    const int64_t g = gs + i;
                    // the next S^T (Q buffer qn) goes out before this step's P V
                    int qn = qb;
                    if (i + 1 == nsteps) {
                        tc::commit_warp(q_empty + qb); // the unit's last S^T has been issued: its Q buffer may be refilled
                        // the next unit's first S^T goes ahead of this P V when its Q is already in place, so
                        // the softmax warps find it ready when they start that unit
                        qn = -1;
                        if (u + (int)gridDim.x < U && __all_sync(0xffffffffu, mbar_test_wait(q_bar(nu + 1), q_par(nu + 1)))) {
                            qn = (nu + 1) & 1;
                            ahead = true;
                        }
                    }
                    if (qn >= 0) {
                        ok = issue_s(g + 1, qn);
                        if (!ok) break;
                    }
                    const int sv = (int)(g % LY::NSV), b = (int)(g & 1);
                    ok = __all_sync(0xffffffffu, mbar_wait_sleep(p_full + b, (g >> 1) & 1) &&
                                                     mbar_wait_sleep(v_full + sv, (g / LY::NSV) & 1));
                    // O^T of this unit's parity was read out by the epilogue warps for unit nu - 2
                    if (ok && i == 0 && nu >= 2)
                        ok = __all_sync(0xffffffffu, mbar_wait_sleep(o_free + (nu & 1), ((nu >> 1) - 1) & 1));
                    if (!ok) break;
                    const uint32_t tO = tmem + OB + (uint32_t)((nu & 1) * 32);
                    tc::fence_after_sync();
                    const uint64_t a0 = dV + (uint64_t)((sv * LY::STAGE) >> 4), b0 = dP + (uint64_t)((b * LY::P_BYTES) >> 4);
#pragma unroll
                    for (int k = 0; k < TOK / 16; ++k)
                        tc::mma_f16_warp(tO, a0 + (uint64_t)((k * kVStep) >> 4),
                                         b0 + (uint64_t)(((k >> 2) * (LY::NPR * 128) + (k & 3) * 32) >> 4), IPV,
                                         (i > 0 || k > 0) ? 1u : 0u);
                    tc::commit_warp(t_full + b);
                    // 16-bit: the V stage's release for the V loader (E4M3: the converters wait for
                    // t_full, the same event with two V stages)
                    if constexpr (!F8) tc::commit_warp(v_empty + sv);
                    if (i + 1 == nsteps) tc::commit_warp(o_full + (nu & 1));
                }
                gs += nsteps;
                if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
            }
            if (!ok && lane == 0) fail();
            // every MMA issued by the elected lane has completed before tensor memory is released
            if (any_mma) {
                tc::commit_warp(fin);
                if (!__all_sync(0xffffffffu, mbar_wait_sleep(fin, 0)) && lane == 0) set_error(a.err, PKV_DEVERR_TIMEOUT);
            }
        }
    } else if (warp < 6) {
        // ---------------------------------------------------------------- softmax
        const int lw = warp & 3;
        const int r = lw * 32 + lane;                      // token row of S^T, then dimension of O^T
        const uint32_t lane_off = static_cast<uint32_t>(lw * 32) << 16;
        bool ok = true;
        int64_t gs = 0;
        int nu = 0;
        // table entry of this thread's block (row r of the step) in step i of a unit, and whether that
        // block belongs to the unit
        const int jb = r / a.bs;
        // (the read is always made, from an index kept inside the table row, and whether the block
        // belongs to the unit is kept apart: a select between the loaded value and -1 would wait for
        // the load on the spot, while here the value is first used a step later)
        auto blk_read = [&](const Unit &x, int i) -> int {
            const int idx = min(x.blk0 + i * bpstep + jb, a.max_blocks - 1);
            return a.tables[(int64_t)x.s * a.max_blocks + max(idx, 0)];
        };
        auto blk_in = [&](const Unit &x, int i) -> bool { return i * bpstep + jb < x.ntiles; };
        // the units come from the K loader's records: the next one is read at the last step of the
        // current one, with the table entry of its first step; entries are read a step ahead
        int u = blockIdx.x;
        Unit un{};
        int tok_end = 0, ent = -1;
        bool ent_in = false;
        float ksc = 1.f;
        if (u < U) {
            ok = read_rec(0, un, tok_end, ksc);
            if (ok) {
                ent = blk_read(un, 0);
                ent_in = blk_in(un, 0);
            }
        }
        for (; u < U && ok; u += gridDim.x, ++nu) {
            const int nsteps = (un.ntiles + bpstep - 1) / bpstep;
            const int u2 = u + (int)gridDim.x;
            Unit un2{};
            int tok_end2 = 0;
            float ksc2 = 1.f;
            const int tok0 = un.blk0 * a.bs;
            // scores in log2 units: scale * log2(e), times the K scale of the head and the power of two
            // taken out of q by the converters (FP8 caches)
            float qsc = a.qk_scale_log2;
            float m[G], lp[G]; // base (uniform over the CTA) and this thread's partial row sums
#pragma unroll
            for (int g = 0; g < G; ++g) {
                m[g] = -INFINITY;
                lp[g] = 0.f;
            }
            // `ok` agreement: the four warps stop together, at a barrier (see named_barrier_and)
            for (int i = 0; i < nsteps; ++i) {
                const int64_t g0 = gs + i;
                const int b = (int)(g0 & 1);
                // the next step's table entry (the next unit's first one after the last step)
                bool rec_ok = true;
                if (i + 1 == nsteps && u2 < U) rec_ok = read_rec(nu + 1, un2, tok_end2, ksc2);
                const bool last = i + 1 == nsteps;
                const int ent_nx = blk_read(last ? un2 : un, last ? 0 : i + 1);
                const bool ent_nx_in = last ? u2 < U && rec_ok && blk_in(un2, 0) : blk_in(un, i + 1);
                bool mine = ok && rec_ok && *abort_flag == 0;
                if constexpr (F8) {
                    // the unit's q exponent, published with its "Q converted" barrier
                    if (mine && i == 0) {
                        mine = __all_sync(0xffffffffu, mbar_wait_sleep(q_ready + (nu & 7), (uint32_t)(nu >> 3) & 1u));
                        qsc = a.qk_scale_log2 * ksc * exp2f((float)qexp[nu & 7]);
                    }
                }
                if (mine) mine = __all_sync(0xffffffffu, mbar_wait_sleep(s_full + b, (g0 >> 1) & 1));
                const int step0 = tok0 + i * TOK;
                // a row holds a token of the unit if it lies before the unit's end and in a block whose
                // table entry names a block of the pool (the loaders skip the others)
                const bool valid = step0 + r < tok_end && ent_in && ent >= 0 && ent < a.num_blocks;
                ent = ent_nx;
                ent_in = ent_nx_in;
                float sc[G];
                bool need = !mine; // a failed wait takes the exchange path, where `ok` is agreed
                if (mine) {
                    tc::fence_after_sync();
                    uint32_t sr[G];
                    tc::ldn<G>(tmem + lane_off + b * NSC, sr);
                    if constexpr (F8) {
                        // S^T of the three E4M3 terms of q (columns 0, 8, 16 of the buffer)
                        uint32_t s1[G], s2[G];
                        tc::ldn<G>(tmem + lane_off + b * NSC + 8, s1);
                        tc::ldn<G>(tmem + lane_off + b * NSC + 16, s2);
                        tc::wait_ld();
#pragma unroll
                        for (int g = 0; g < G; ++g)
                            sr[g] = __float_as_uint((__uint_as_float(sr[g]) + __uint_as_float(s1[g])) + __uint_as_float(s2[g]));
                    }
                    tc::wait_ld();
                    tc::fence_before_sync();
                    mbar_arrive(s_free + b);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(k_empty + (int)(g0 % NS)); // S^T is done: the MMA has read the step's K
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        sc[g] = valid ? __uint_as_float(sr[g]) * qsc : -INFINITY;
                        need |= sc[g] > m[g] + kRescale; // false while sc = -inf
                    }
                }
                // The base moves only where a score passes it by more than kRescale.  The four warps
                // first agree whether any score does (one barrier); only then do they exchange the tile
                // maxima per head (warp shuffles, shared memory, a second barrier).  After a unit's
                // first step that is rare, so most steps pay one barrier.
                bool moved = false;
                float alpha[G], p[G];
#pragma unroll
                for (int g = 0; g < G; ++g) alpha[g] = 1.f;
                // (a unit's first step always sets the base: its scores are the first, so the exchange runs
                // without asking)
                if (i == 0 || named_barrier_or(1, 128, need)) {
                    if (mine) {
                        float tmx[G];
#pragma unroll
                        for (int g = 0; g < G; ++g) {
                            float v = sc[g];
#pragma unroll
                            for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
                            tmx[g] = v;
                        }
                        if (lane < G) {
                            float v = tmx[0];
#pragma unroll
                            for (int g = 1; g < G; ++g)
                                if (lane == g) v = tmx[g];
                            red_max[(int)(g0 & 1) * 4 * NQ + lw * NQ + lane] = v;
                        }
                    }
                    ok = named_barrier_and(1, 128, mine);
                    if (!ok) break;
                    const float *rm = red_max + (int)(g0 & 1) * 4 * NQ;
#pragma unroll
                    for (int g = 0; g < G; ++g) {
                        const float t = fmaxf(fmaxf(rm[g], rm[NQ + g]), fmaxf(rm[2 * NQ + g], rm[3 * NQ + g]));
                        const bool up = t > m[g] + kRescale; // false while t = -inf
                        alpha[g] = up ? fast_exp2(m[g] - t) : 1.f;
                        if (up) m[g] = t;
                        moved |= up;
                    }
                }
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    p[g] = valid ? fast_exp2(sc[g] - m[g]) : 0.f;
                    lp[g] = lp[g] * alpha[g] + p[g];
                }
                // P buffer b is free once P V of step g0 - 2 is done; O^T is stable once P V of g0 - 1 is
                if (g0 >= 2) ok = __all_sync(0xffffffffu, mbar_wait_sleep(t_full + b, ((g0 >> 1) - 1) & 1));
                if (ok && moved && i > 0) {
                    ok = __all_sync(0xffffffffu, mbar_wait_sleep(t_full + (b ^ 1), ((g0 - 1) >> 1) & 1));
                    if (ok) {
                        tc::fence_after_sync();
#pragma unroll
                        for (int part = 0; part < LY::NP; ++part) {
                            uint32_t o[G];
                            tc::ldn<G>(tmem + lane_off + OB + (nu & 1) * 32 + part * NQ, o);
                            tc::wait_ld();
#pragma unroll
                            for (int g = 0; g < G; ++g) o[g] = __float_as_uint(__uint_as_float(o[g]) * alpha[g]);
                            tc::stn<G>(tmem + lane_off + OB + (nu & 1) * 32 + part * NQ, o);
                        }
                        tc::wait_st();
                    }
                }
                // a warp that failed here carries ok = false to the next barrier
                if (!ok) continue;
                uint8_t *pb = smem + LY::P + b * LY::P_BYTES;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const int off = p_offset<LY::NPR>(g, r);
                    if constexpr (LY::NP == 2) {
                        const uint32_t hi = pack2<OT>(p[g], 0.f) & 0xFFFFu;
                        const float rest = p[g] - __uint_as_float(hi << 16);
                        *reinterpret_cast<uint16_t *>(pb + off) = (uint16_t)hi;
                        *reinterpret_cast<uint16_t *>(pb + p_offset<LY::NPR>(NQ + g, r)) =
                            (uint16_t)(pack2<OT>(rest, 0.f) & 0xFFFFu);
                    } else {
                        *reinterpret_cast<uint16_t *>(pb + off) = (uint16_t)(pack2<OT>(p[g], 0.f) & 0xFFFFu);
                    }
                }
                if (__any_sync(0xffffffffu, !valid)) {
                    // a row without a token holds an unused slot, a skipped block's stale row or (FP8)
                    // widened garbage: zero its V once the stage has landed, so that no NaN reaches the
                    // MMA (only these steps wait for V here; P V waits for it in the MMA warp)
                    const int sv = (int)(g0 % LY::NSV);
                    if (!__all_sync(0xffffffffu, mbar_wait_sleep(v_full + sv, (g0 / LY::NSV) & 1))) {
                        ok = false;
                        continue; // carried to the next barrier
                    }
                    if (!valid) {
#pragma unroll
                        for (int c = 0; c < D / 64; ++c) {
                            uint4 *vr = reinterpret_cast<uint4 *>(
                                smem + LY::V0 + sv * LY::STAGE +
                                (F8 ? c * (TOK * 128) + r * 128 : (r >> 3) * 2048 + c * 1024 + (r & 7) * 128));
#pragma unroll
                            for (int e = 0; e < 8; ++e) vr[e] = make_uint4(0u, 0u, 0u, 0u);
                        }
                    }
                }
                fence_proxy_async_smem();
                tc::fence_before_sync();
                mbar_arrive(p_full + b);
            }
            gs += nsteps;
            // ---- hand the unit's row sums and bases to the epilogue warps (buffer nu % 2)
            const int eb = nu & 1;
            if (ok && nu >= 2) ok = __all_sync(0xffffffffu, mbar_wait_sleep(l_free + eb, ((nu >> 1) - 1) & 1));
            if (ok) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float v = lp[g];
#pragma unroll
                    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
                    if (lane == g) red_sum[(eb * 4 + lw) * NQ + g] = v;
                    if (r == 0) m_base[eb * NQ + g] = m[g];
                }
                mbar_arrive(l_ready + eb);
            }
            // the four warps leave the unit loop together or not at all (a warp that left alone would
            // leave the others waiting at the next named barrier)
            ok = named_barrier_and(1, 128, ok);
            if (!ok) break;
            un = un2;
            tok_end = tok_end2;
            ksc = ksc2;
        }
        if (!ok) fail();
    } else if (warp < 11) {
        // ---------------------------------------------------------------- epilogue (warps 7-10)
        // Thread r holds dimension r of the unit's G output rows: O^T from tensor memory (its lane
        // quadrant), the row sums of the four softmax warps and the bases from shared memory.  The
        // softmax warps go on with the next unit meanwhile; O^T and the sums are double-buffered.
        const int lw = warp & 3;
        const int r = lw * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(lw * 32) << 16;
        bool ok = true;
        int nu = 0;
        for (int u = blockIdx.x; u < U && ok; u += gridDim.x, ++nu) {
            Unit un;
            int te;
            float ks;
            if (!read_rec(nu, un, te, ks)) {
                ok = false;
                break;
            }
            const int eb = nu & 1;
            ok = __all_sync(0xffffffffu, mbar_wait_sleep(o_full + eb, (nu >> 1) & 1) && mbar_wait_sleep(l_ready + eb, (nu >> 1) & 1));
            if (!ok) break;
            tc::fence_after_sync();
            uint32_t o[G];
            tc::ldn<G>(tmem + lane_off + OB + eb * 32, o);
            if constexpr (LY::NP == 2) {
                uint32_t o2[G];
                tc::ldn<G>(tmem + lane_off + OB + NQ + eb * 32, o2);
                tc::wait_ld();
#pragma unroll
                for (int g = 0; g < G; ++g) o[g] = __float_as_uint(__uint_as_float(o[g]) + __uint_as_float(o2[g]));
            }
            tc::wait_ld();
            tc::fence_before_sync();
            mbar_arrive(o_free + eb); // unit nu + 2's first P V may overwrite this O^T
            float lt[G], mb[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float *rs = red_sum + eb * 4 * NQ + g;
                lt[g] = (rs[0] + rs[NQ]) + (rs[2 * NQ] + rs[3 * NQ]);
                mb[g] = m_base[eb * NQ + g];
            }
            mbar_arrive(l_free + eb); // the softmax may publish unit nu + 2's sums here
            const int h0 = un.kvh * G;
            if constexpr (F8) {
                const float vs = a.v_scale[un.kvh]; // V codes were widened without their scale
#pragma unroll
                for (int g = 0; g < G; ++g) o[g] = __float_as_uint(__uint_as_float(o[g]) * vs);
            }
            if (un.nsplit == 1 && a.slot0 == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float y = lt[g] > 0.f ? __uint_as_float(o[g]) / lt[g] : 0.f;
                    static_cast<T *>(a.out)[((int64_t)un.s * a.hq + h0 + g) * D + r] = M::from_f(y);
                }
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const int64_t idx = ((int64_t)un.s * a.hq + h0 + g) * a.max_splits + a.slot0 + un.j;
                    a.ws_o[idx * D + r] = __uint_as_float(o[g]);
                    if (r == 0) reinterpret_cast<float2 *>(a.ws_ml)[idx] = make_float2(mb[g], lt[g]);
                }
            }
            if (__any_sync(0xffffffffu, *abort_flag != 0)) break;
        }
        if (!ok && lane == 0) fail();
    } else if constexpr (F8) {
        // ---------------------------------------------------------------- E4M3 V -> fp16, q -> E4M3 (warps 11-14)
        // Thread r owns token r of every step and dimension r of q.  Token r's V codes sit in the code
        // stage as row r & 7 of the V half of row group r >> 3, 128-byte swizzled as they landed; they
        // are widened into row r of a V stage (fp16, the P V MMA's MN-major layout).  E4M3 values are
        // exact in fp16.  K stays E4M3: the S^T MMA reads it as it landed.
        const int cw = warp - 11, r = cw * 32 + lane;
        auto widen_row = [&](const uint8_t *codes, uint8_t *stage) {
            const uint8_t *src = codes + (r >> 3) * 2048 + 1024 + (r & 7) * 128;
            uint4 w[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) w[c] = *reinterpret_cast<const uint4 *>(src + (((c + lane) & 7) << 4));
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int ch = ((c + lane) & 7) ^ (r & 7); // 16 dims: 16 ch .. 16 ch + 15 (the swizzled chunk read)
                const uint32_t in[4] = {w[c].x, w[c].y, w[c].z, w[c].w};
                uint32_t o[8];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const unsigned short lo = (unsigned short)(in[e] & 0xFFFFu), hi = (unsigned short)(in[e] >> 16);
                    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o[2 * e]) : "h"(lo));
                    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(o[2 * e + 1]) : "h"(hi));
                }
                uint8_t *row = stage + (ch >> 2) * (TOK * 128) + r * 128;
                const int u0 = (ch & 3) * 2;
                *reinterpret_cast<uint4 *>(row + ((u0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                *reinterpret_cast<uint4 *>(row + (((u0 + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
            }
        };
        // byte offset of (head g, dimension r) in the loaded Q tile (model dtype, K-major, 128-byte swizzle)
        auto qoff = [&](int g) {
            const int e = r & 63;
            return (r >> 6) * (NQ * 128) + g * 128 + (((e >> 3) ^ (g & 7)) << 4) + (e & 7) * 2;
        };
        auto e4m3_value = [](uint32_t code) -> float {
            uint32_t h2;
            asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)code));
            return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
        };
        // q of this CTA's n-th unit as three E4M3 terms, q = 2^e (t0 + t1 + t2): the largest |q| is
        // scaled into [2^7, 2^8), each term codes what the earlier ones left (about 4 more significant
        // bits a term, so ~12 in all, like fp16's 11).  The MMA operand is 32 rows of 128 codes, K-major
        // and 128-byte swizzled, written over the loaded tile (same 4 KB, every thread has read its
        // values before the barrier): row 8 t + g holds term t of head g, other rows are zero.  False,
        // agreed by the four warps at their barrier, after a failed wait.
        auto convert_q = [&](int n, bool mine) -> bool {
            const int qb = n & 1;
            if (mine) mine = __all_sync(0xffffffffu, mbar_wait_sleep(q_full + qb, (n >> 1) & 1));
            uint8_t *qt = smem + LY::Q + qb * LY::Q_BYTES;
            float x[G], mx = 0.f;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                x[g] = 0.f;
                if (mine) {
                    const uint16_t bits = *reinterpret_cast<const uint16_t *>(qt + qoff(g));
                    x[g] = MT == PKV_BF16 ? __uint_as_float((uint32_t)bits << 16) : __half2float(__ushort_as_half(bits));
                    mx = fmaxf(mx, fabsf(x[g]));
                }
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            if (lane == 0) qred[qb * 4 + cw] = mx;
            if (!named_barrier_and(2, 128, mine)) return false;
            const float qm = fmaxf(fmaxf(qred[qb * 4], qred[qb * 4 + 1]), fmaxf(qred[qb * 4 + 2], qred[qb * 4 + 3]));
            int e = 0;
            if (qm > 0.f) {
                int ex;
                frexpf(qm, &ex);
                e = min(max(ex - 8, -100), 100);
            }
            uint32_t code[3][G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float y = ldexpf(x[g], -e);
#pragma unroll
                for (int t = 0; t < 3; ++t) {
                    code[t][g] = e4m3x2_from_f32(y, 0.f) & 0xFFu;
                    y -= e4m3_value(code[t][g]);
                }
            }
#pragma unroll
            for (int row = 0; row < 32; ++row) {
                const int t = row >> 3, g = row & 7;
                uint32_t v = 0u;
#pragma unroll
                for (int tt = 0; tt < 3; ++tt)
#pragma unroll
                    for (int gg = 0; gg < G; ++gg)
                        if (tt == t && gg == g) v = code[tt][gg];
                qt[row * 128 + (((r >> 4) ^ (row & 7)) << 4) + (r & 15)] = (uint8_t)v;
            }
            if (r == 0) qexp[n & 7] = e; // read by the softmax after q_ready
            fence_proxy_async_smem();   // Q is read by the MMA
            mbar_arrive(q_ready + (n & 7));
            return true;
        };
        // unit 0's q first; each later unit's once the previous unit's V tile of step max(0, n - 4) is
        // widened (its first step for units of up to four steps), so that it is ready when the softmax
        // starts that unit
        bool ok = (int)blockIdx.x < U ? convert_q(0, *abort_flag == 0) : true;
        int64_t gs = 0;
        int nu = 0;
        for (int u = blockIdx.x; u < U && ok; u += gridDim.x, ++nu) {
            Unit un;
            int te;
            float ks;
            if (!read_rec(nu, un, te, ks)) {
                ok = false;
                break;
            }
            const int nsteps = (un.ntiles + bpstep - 1) / bpstep;
            // ---- the unit's V stages
            for (int i = 0; i < nsteps && ok; ++i) {
                const int64_t g = gs + i;
                const int st = (int)(g % NS), sv = (int)(g % LY::NSV);
                // the step's codes have landed, and P V of the step that used this V stage before is done
                ok = __all_sync(0xffffffffu, mbar_wait_sleep(k_full + st, (g / NS) & 1));
                static_assert(!F8 || LY::NSV == 2, "V stage g % 2 frees with P V of step g - 2 (t_full)");
                if (ok && g >= 2) ok = __all_sync(0xffffffffu, mbar_wait_sleep(t_full + (g & 1), ((g >> 1) - 1) & 1));
                if (!ok) break;
                widen_row(smem + LY::K0 + st * LY::KSTAGE, smem + LY::V0 + sv * LY::STAGE);
                fence_proxy_async_smem();
                mbar_arrive(v_full + sv);
                __syncwarp();
                if (lane == 0) mbar_arrive(k_empty + st); // this warp's V codes are read
                // not before step nsteps - 4: convert_q waits for the next unit's Q, which warp 0 issues at
                // the latest with the next unit's first step, and warp 0 gets there only if it is at most
                // NS = 4 steps ahead of the code stages this warp has released (releases come first)
                static_assert(NS == 4, "the conversion point assumes four code stages");
                if (i == (nsteps > NS ? nsteps - NS : 0) && u + (int)gridDim.x < U) {
                    ok = convert_q(nu + 1, *abort_flag == 0);
                    if (!ok) break;
                }
            }
            gs += nsteps;
            // the four warps leave together (the next unit's barrier would wait for a warp gone)
            ok = named_barrier_and(2, 128, ok && *abort_flag == 0);
            if (!ok) break;
        }
        if (!ok && lane == 0) fail();
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <int G, int MT, int KVT>
cudaError_t launch(const CUtensorMap &tkv, const CUtensorMap &tq, const Args &a, int grid, size_t smem,
                   cudaStream_t st) {
    auto kern = decode_tc_kernel<G, MT, KVT>;
    constexpr int kThreads = threads_for<KVT == PKV_FP8_E4M3>();
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return pdl_launch(kern, dim3(grid), dim3(kThreads), smem, st, tkv, tq, a);
}

} // namespace pkv_decode_tc
