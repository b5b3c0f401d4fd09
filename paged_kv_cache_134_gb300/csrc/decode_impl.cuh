// Paged decode attention: split-K flash-decoding over block-table entries.
//
// What it computes ("PagedAttention 与前缀缓存", 2kiu.com, section 2.3): for every sequence
// s and query head h, softmax(scale * q . K_t) weighted sum of V_t over the sequence's
// L_s tokens, where token t lives in physical block block_table[s][t / bs] at offset
// t % bs; slots of the tail block at or beyond L_s are never used (the page's tail-block
// warning).  Grouped-query heads: query head h reads KV head h / G, and one pass over a KV
// head's tiles serves all G query heads that share it, so every K/V byte is read once.
//
// Design (GB300, HBM-bound, ~1 flop per byte for G = 1):
//  * Work unit = (sequence, KV head, split), a split being up to `split_blocks` consecutive
//    logical blocks.  Splits are block-aligned and depend only on L_s, so the arithmetic
//    order of every output is fixed by the lengths alone (placement of physical blocks,
//    sharing of prefix blocks and the batch composition never change a bit).
//  * Persistent CTAs (a whole number of CTAs per SM) walk a unit list that puts full splits
//    first and partial tail splits last; units go round-robin over CTAs.
//  * One producer warp per CTA reads block-table entries (32 at a time, coalesced) and issues
//    one 1-D bulk async copy (cp.async.bulk, the TMA's linear mode) per (block, K|V, head)
//    tile into a ring of shared-memory stages, completion tracked by mbarrier transaction
//    counts.  The pool layout [block][K|V][head][offset][dim] makes each tile one contiguous
//    bs*D*elt-byte run (4 KB for bs=16, D=128, fp16), so one table lookup yields two large
//    aligned copies.  Blocks whose K plus V tile would exceed a stage's bytes (bs=32 at fp16,
//    D=128) go in equal parts of consecutive tokens, one part per stage, so that a stage stays
//    small and more CTAs fit an SM; parts wholly past the sequence's end are not loaded.  The
//    copies carry an L2 evict-first hint: KV is streamed once.
//  * Four consumer warps take the tiles round-robin by their index in the CTA's tile stream.  In a warp, D/8 lanes share a
//    token (16-byte vector loads from shared memory, conflict-free), partial dot products are
//    reduced with xor-shuffles, and an online softmax (running max m, sum l, rescaled
//    accumulator) runs per 16-token chunk with exp2 on prescaled scores.
//  * At the end of a unit each warp hands its (m, l, acc) to one of two merge slots in shared
//    memory (by the parity of the CTA's unit count) and goes on to its next unit's tiles; the
//    warp that hands in last merges the four in warp order and writes the result, so no warp
//    waits for the others at a unit boundary while its next tiles land.  A sequence with one
//    split writes its output row directly; otherwise the unit writes an fp32 partial (m, l,
//    unnormalised o) and a merge kernel combines the splits in split order.
//  * Every mbarrier wait is bounded (PKV_WAIT_LIMIT_NS); a timeout sets PKV_DEVERR_TIMEOUT
//    and the CTA winds down without further waiting on work that will not arrive.
#pragma once

#include "device_common.cuh"
#include "pkv_internal.h"

namespace pkv_decode {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxSeqs = 1024;

struct Args {
    const void *q;
    void *out;
    const char *pool;
    const float *k_scale, *v_scale;
    const int32_t *tables, *lens;
    float *ws_o, *ws_ml;
    unsigned int *err;
    int64_t num_blocks;
    int64_t blk_stride;  // bytes between consecutive physical blocks
    int64_t kv_stride;   // bytes between the K and V halves of a block
    int tile_bytes;      // one (block, K|V, head) tile
    // one stage of the CUDA-core kernel's ring: sub_tokens consecutive tokens of a block (the
    // whole block, or an equal part of it) of one head, K then V, sub_bytes each
    int sub_tokens, sub_bytes;
    int max_blocks, num_seqs, hq, hkv, bs;
    int split_blocks, max_splits, nstages;
    float qk_scale_log2; // scale * log2(e)
    // cascade decode: the first start_block blocks of every table are a shared prefix whose
    // attention another kernel computed into workspace slots [0, slot0); this kernel then covers the
    // blocks from start_block on and writes its splits from slot slot0 on (both 0 otherwise)
    int start_block = 0, slot0 = 0;
};

template <int KVT>
PKV_DEV void load8(const char *p, float *f) {
    if constexpr (KVT == PKV_FP8_E4M3) {
        cvt8_e4m3(*reinterpret_cast<const uint2 *>(p), f);
    } else {
        cvt8<KVT>(*reinterpret_cast<const uint4 *>(p), f);
    }
}

// Which unit is u: (sequence, KV head, split index, first logical block, tiles).
struct Unit {
    int s, kvh, j, blk0, ntiles, nsplit;
};

PKV_DEV int find_row(const int *pref, int n, int k) {
    // largest i in [0, n) with pref[i] <= k (pref non-decreasing, pref[0] = 0)
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (pref[mid] <= k)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

PKV_DEV Unit unit_info(int u, const int *pf, const int *pp, const int *nb, int S, int hkv, int bps, int sb = 0) {
    Unit r;
    const int nfull_units = pf[S] * hkv;
    if (u < nfull_units) {
        const int k = u / hkv;
        r.kvh = u - k * hkv;
        r.s = find_row(pf, S, k);
        r.j = k - pf[r.s];
        r.blk0 = sb + r.j * bps;
        r.ntiles = bps;
    } else {
        const int u2 = u - nfull_units;
        const int k = u2 / hkv;
        r.kvh = u2 - k * hkv;
        r.s = find_row(pp, S, k);
        r.j = pf[r.s + 1] - pf[r.s];
        r.blk0 = sb + r.j * bps;
        r.ntiles = nb[r.s] - r.blk0;
    }
    r.nsplit = (pf[r.s + 1] - pf[r.s]) + (pp[r.s + 1] - pp[r.s]);
    return r;
}

// Lane layout of a consumer warp for head_dim D and G query heads per KV head.  A token's row is
// covered by LT = LH * G lanes: each of the G query heads gets LH lanes, each lane DL consecutive
// dims of that head (so it keeps q, the accumulator and the scores of one head only).  Lanes of
// different heads read the same K/V chunk (a shared-memory broadcast).  TPP tokens go in one pass.
//   G=1, D=128: DL=8,  LH=16, 2 tokens/pass     G=4, D=128: DL=16, LH=8, 1 token/pass
//   G=1, D=64:  DL=8,  LH=8,  4 tokens/pass     G=8, D=128: DL=32, LH=4, 1 token/pass
template <int D, int G>
struct Lanes {
    static constexpr int DL = (D * G / 32) > 8 ? (D * G / 32) : 8; // dims per lane
    static constexpr int LH = D / DL;                               // lanes per (token, head)
    static constexpr int LT = LH * G;                               // lanes per token
    static constexpr int TPP = 32 / LT;                             // tokens per pass
    static constexpr int MAXP = 16 / TPP;                           // passes per 16-token chunk
    static_assert(LT <= 32 && 32 % LT == 0 && D % DL == 0 && DL % 8 == 0, "lane layout");
};

template <int KVT, int N>
PKV_DEV void loadN(const char *p, float *f) {
    constexpr int EB = (KVT == PKV_FP8_E4M3) ? 1 : 2;
#pragma unroll
    for (int c = 0; c < N / 8; ++c) load8<KVT>(p + c * 8 * EB, f + 8 * c);
}

// One tile of `bs` tokens, `valid` of them real, for this lane's query head.
template <int D, int G, int KVT>
PKV_DEV void process_tile(const char *ks, const char *vs, int bs, int valid,
                          const float (&qf)[Lanes<D, G>::DL], float &m, float &l, float (&acc)[Lanes<D, G>::DL],
                          int lane) {
    using LY = Lanes<D, G>;
    constexpr int DL = LY::DL, LH = LY::LH, LT = LY::LT, TPP = LY::TPP, MAXP = LY::MAXP;
    constexpr int EB = (KVT == PKV_FP8_E4M3) ? 1 : 2;
    const int sub = lane % LH, tg = lane / LT;
    const int ch = bs < 16 ? bs : 16;
    const int npc = ch / TPP;
    for (int c0 = 0; c0 < bs; c0 += ch) {
        if (c0 >= valid) break;
        float sc[MAXP];
#pragma unroll
        for (int p = 0; p < MAXP; ++p) {
            if (p < npc) {
                const int t = c0 + p * TPP + tg;
                float kf[DL];
                loadN<KVT, DL>(ks + (t * D + sub * DL) * EB, kf);
                float d0 = 0.f, d1 = 0.f;
#pragma unroll
                for (int e = 0; e < DL; e += 2) {
                    d0 = fmaf(qf[e], kf[e], d0);
                    d1 = fmaf(qf[e + 1], kf[e + 1], d1);
                }
                sc[p] = d0 + d1;
            }
        }
#pragma unroll
        for (int p = 0; p < MAXP; ++p) {
            if (p < npc) {
                float v = sc[p];
#pragma unroll
                for (int o = LH / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                sc[p] = (c0 + p * TPP + tg) < valid ? v : -INFINITY;
            }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int p = 0; p < MAXP; ++p)
            if (p < npc) mx = fmaxf(mx, sc[p]);
#pragma unroll
        for (int o = LT; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float mn = fmaxf(m, mx); // finite: the chunk holds at least one live token
        const float alpha = fast_exp2(m - mn);
        m = mn;
        l *= alpha;
#pragma unroll
        for (int e = 0; e < DL; ++e) acc[e] *= alpha;
#pragma unroll
        for (int p = 0; p < MAXP; ++p) {
            if (p < npc) {
                const float pr = fast_exp2(sc[p] - mn);
                sc[p] = pr;
                l += pr;
            }
        }
#pragma unroll
        for (int p = 0; p < MAXP; ++p) {
            if (p < npc) {
                const int t = c0 + p * TPP + tg;
                if (t < valid) {
                    float vf[DL];
                    loadN<KVT, DL>(vs + (t * D + sub * DL) * EB, vf);
#pragma unroll
                    for (int e = 0; e < DL; ++e) acc[e] = fmaf(sc[p], vf[e], acc[e]);
                }
            }
        }
    }
}

// Grouped-query heads (G >= 2): token-parallel lanes.  D/8 lanes share a token (8 dims each) and
// every lane works for all G query heads, so each K/V element is loaded and widened once and
// feeds G products.  Products and the P.V accumulation use packed fp32 FMAs (two lanes of an
// IEEE fma each).  The partial dot products of the chunk's passes are summed across the token's
// lanes by a reduce-scatter: after log2 steps every lane holds the full score of one pass, so the
// softmax of a head costs one exp2 per lane, and each pass's weight is then fetched back by a
// shuffle from the lane that owns it.
template <int D, int G, int KVT>
PKV_DEV void process_tile_tp(const char *ks, const char *vs, int bs, int valid, const float (&qf)[G][8],
                             float (&m)[G], float (&l)[G], float (&acc)[G][8], int lane) {
    constexpr int LPT = D / 8;     // lanes per token
    constexpr int TPP = 32 / LPT;  // tokens per pass
    constexpr int MAXP = 16 / TPP; // passes per 16-token chunk (8 for D=128, 4 for D=64)
    constexpr int EB = (KVT == PKV_FP8_E4M3) ? 1 : 2;
    // after the reduce-scatter the lane with sub-lane bits s holds pass (s >> DUP) of its token group;
    // the DUP lowest sub-lane bits only duplicate it
    constexpr int LOG_LPT = LPT == 16 ? 4 : 3;
    constexpr int LOG_P = MAXP == 8 ? 3 : (MAXP == 4 ? 2 : 1);
    constexpr int DUP = LOG_LPT - LOG_P;
    const int sub = lane % LPT, grp = lane / LPT;
    const int mypass = sub >> DUP;
    const bool owner = (sub & ((1 << DUP) - 1)) == 0;
    const int ch = bs < 16 ? bs : 16;
    const int npc = ch / TPP;
    for (int c0 = 0; c0 < bs; c0 += ch) {
        if (c0 >= valid) break;
        float part[G][MAXP];
#pragma unroll
        for (int p = 0; p < MAXP; ++p) {
            if (p < npc) {
                const int t = c0 + p * TPP + grp;
                float kf[8];
                load8<KVT>(ks + (t * D + sub * 8) * EB, kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float d0 = 0.f, d1 = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; e += 2) ffma2(d0, d1, qf[g][e], qf[g][e + 1], kf[e], kf[e + 1]);
                    part[g][p] = d0 + d1;
                }
            } else {
#pragma unroll
                for (int g = 0; g < G; ++g) part[g][p] = 0.f;
            }
        }
        // reduce-scatter over the LPT lanes of a token
        float sc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int lv = 0; lv < LOG_P; ++lv) {
                const int S = LPT >> (lv + 1); // partner distance
                const int C = MAXP >> lv;      // values still held
                const bool upper = (sub & S) != 0;
#pragma unroll
                for (int i = 0; i < C / 2; ++i) {
                    const float a = part[g][i], b = part[g][i + C / 2];
                    const float recv = __shfl_xor_sync(0xffffffffu, upper ? a : b, S);
                    part[g][i] = (upper ? b : a) + recv;
                }
            }
            float v = part[g][0];
#pragma unroll
            for (int o = (1 << DUP) >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            sc[g] = (c0 + mypass * TPP + grp) < valid ? v : -INFINITY;
        }
        // online softmax per head; the chunk's scores are spread one per lane
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mx = sc[g];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mn = fmaxf(m[g], mx); // finite: the chunk holds at least one live token
            const float alpha = fast_exp2(m[g] - mn);
            m[g] = mn;
            const float pr = fast_exp2(sc[g] - mn);
            sc[g] = pr;
            l[g] = l[g] * alpha + (owner ? pr : 0.f);
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] *= alpha;
        }
#pragma unroll
        for (int p = 0; p < MAXP; ++p) {
            if (p < npc) {
                const int t = c0 + p * TPP + grp;
                const int src = grp * LPT + (p << DUP);
                float w[G];
#pragma unroll
                for (int g = 0; g < G; ++g) w[g] = __shfl_sync(0xffffffffu, sc[g], src);
                if (t < valid) {
                    float vf[8];
                    load8<KVT>(vs + (t * D + sub * 8) * EB, vf);
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int e = 0; e < 8; e += 2) ffma2(acc[g][e], acc[g][e + 1], w[g], w[g], vf[e], vf[e + 1]);
                }
            }
        }
    }
}

// Unit list, built by the whole CTA into shared memory: per sequence its block count nb[s], and
// prefix counts of full splits (pf) and of partial tail splits (pp, 0 or 1 per sequence), so that
// unit u resolves to (sequence, KV head, split) with two binary searches (unit_info).  Sequences
// longer than the table allows are clamped and reported.
PKV_DEV void build_unit_list(const Args &a, int *pf, int *pp, int *nb, int warp, int lane) {
    const int S = a.num_seqs, bps = a.split_blocks;
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const int L = a.lens[s];
        int n = L > 0 ? (L + a.bs - 1) / a.bs : 0;
        if (n > a.max_blocks) {
            if (blockIdx.x == 0) set_error(a.err, PKV_DEVERR_LENGTH);
            n = a.max_blocks;
        }
        nb[s] = n;
        const int m = n > a.start_block ? n - a.start_block : 0; // blocks this kernel covers
        pf[s + 1] = m / bps;
        pp[s + 1] = (m % bps) ? 1 : 0;
    }
    __syncthreads();
    if (warp == 0) {
        int cf = 0, cp = 0;
        for (int base = 0; base < S; base += 32) {
            const int i = base + lane;
            int vf = i < S ? pf[i + 1] : 0, vp = i < S ? pp[i + 1] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int tf = __shfl_up_sync(0xffffffffu, vf, o), tp = __shfl_up_sync(0xffffffffu, vp, o);
                if (lane >= o) {
                    vf += tf;
                    vp += tp;
                }
            }
            if (i < S) {
                pf[i + 1] = vf + cf;
                pp[i + 1] = vp + cp;
            }
            cf += __shfl_sync(0xffffffffu, vf, 31);
            cp += __shfl_sync(0xffffffffu, vp, 31);
        }
        if (lane == 0) {
            pf[0] = 0;
            pp[0] = 0;
        }
    }
    __syncthreads();
}

// wait (bounded) until a shared-memory counter reaches n or the CTA aborts; false after the limit
PKV_DEV bool wait_at_least(const int *x, int n, const int *abort_flag) {
    const volatile int *v = x;
    if (*v >= n) return true;
    const uint64_t t0 = global_timer_ns();
    while (*v < n && !*reinterpret_cast<const volatile int *>(abort_flag)) {
        if (global_timer_ns() - t0 > PKV_WAIT_LIMIT_NS) return false;
        __nanosleep(32);
    }
    return true;
}

template <int D, int G, int MT, int KVT>
__global__ void __launch_bounds__(kThreads) decode_kernel(const Args a) {
    using M = ModelT<MT>;
    using T = typename M::T;
    constexpr int NCW = kConsumerWarps;
    extern __shared__ __align__(128) unsigned char smem[];
    const int NST = a.nstages;
    const int S = a.num_seqs;
    char *ring = reinterpret_cast<char *>(smem);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)NST * 2 * a.sub_bytes);
    uint64_t *empty = full + NST;
    int *flags = reinterpret_cast<int *>(empty + NST);
    int *abort_flag = flags + NST;
    int *mcount = abort_flag + 1;                               // [2] warps handed in to merge slot p
    int *mdone = abort_flag + 3;                                // [2] merges of slot p completed
    float *mrg = reinterpret_cast<float *>(abort_flag + 8);     // [2 slots][NCW warps][G][D + 2]
    int *pf = reinterpret_cast<int *>(mrg + 2 * NCW * G * (D + 2));
    int *pp = pf + (S + 1);
    int *nb = pp + (S + 1);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NST; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 8; ++i) abort_flag[i] = 0;
        fence_mbarrier_init();
    }
    pdl_wait(); // the previous kernel (e.g. the append of this step) has finished
    // cascade decode: the next kernel is the prefix phase, which reads nothing this kernel writes;
    // it may launch now and take the SMs this grid's CTAs leave
    if (a.slot0 > 0) pdl_trigger();
    const int bps = a.split_blocks;
    build_unit_list(a, pf, pp, nb, warp, lane);
    const int U = (pf[S] + pp[S]) * a.hkv;
    const int ST = a.sub_tokens, spb = a.bs / a.sub_tokens; // stage tokens, stages per block

    if (warp == NCW) {
        // ---------------------------------------------------------------- producer warp
        const uint64_t policy = l2_policy_evict_first();
        uint32_t tau = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < U && ok; u += gridDim.x) {
            const Unit un = unit_info(u, pf, pp, nb, S, a.hkv, bps, a.start_block);
            const int32_t *trow = a.tables + (int64_t)un.s * a.max_blocks + un.blk0;
            const char *head_base = a.pool + (int64_t)un.kvh * a.tile_bytes;
            // stages of this unit: spb per block, less the parts wholly past the sequence's end
            const int nt = spb > 1 ? min(un.ntiles * spb, (a.lens[un.s] - un.blk0 * a.bs + ST - 1) / ST) : un.ntiles;
            for (int i0 = 0; i0 < un.ntiles && ok; i0 += 32) {
                const int cnt = min(32, un.ntiles - i0);
                const int myb = lane < cnt ? trow[i0 + lane] : 0;
                for (int i = 0; i < cnt && ok; ++i) {
                    const int b = __shfl_sync(0xffffffffu, myb, i);
                    for (int h = 0, k = (i0 + i) * spb; h < spb && k < nt; ++h, ++k) {
                        if (lane == 0) {
                            const uint32_t stage = tau % NST, round = tau / NST;
                            if (round > 0 && !mbar_wait(&empty[stage], (round - 1) & 1)) {
                                // stop issuing; the consumers time out on the stages that never fill
                                set_error(a.err, PKV_DEVERR_TIMEOUT);
                                ok = false;
                            } else if (b >= 0 && b < a.num_blocks) {
                                flags[stage] = 0;
                                char *dst = ring + (size_t)stage * 2 * a.sub_bytes;
                                const char *src = head_base + (int64_t)b * a.blk_stride + (int64_t)h * a.sub_bytes;
                                mbar_arrive_expect_tx(&full[stage], 2u * a.sub_bytes);
                                bulk_g2s_hint(dst, src, a.sub_bytes, &full[stage], policy);
                                bulk_g2s_hint(dst + a.sub_bytes, src + a.kv_stride, a.sub_bytes, &full[stage], policy);
                            } else {
                                flags[stage] = 1;
                                set_error(a.err, PKV_DEVERR_BLOCK_ID);
                                mbar_arrive(&full[stage]);
                            }
                        }
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        if (!ok) break;
                        ++tau;
                    }
                }
            }
        }
        // the next kernel (the split merge) may start launching once every CTA has issued its last load
        pdl_trigger();
        // drain: the copies of the last stages must land before this CTA's shared memory goes away
        if (lane == 0) {
            const uint32_t first = tau > (uint32_t)NST ? tau - NST : 0;
            for (uint32_t t = first; t < tau; ++t)
                if (!mbar_wait(&full[t % NST], (t / NST) & 1)) set_error(a.err, PKV_DEVERR_TIMEOUT);
        }
        return;
    }

    // -------------------------------------------------------------------- consumer warps
    // G == 1: Lanes<D, 1> layout (D/8 lanes per token, 8 dims each); G >= 2: token-parallel lanes
    // (process_tile_tp), each lane carrying all G heads.
    using LY = Lanes<D, G>;
    constexpr int DL = (G == 1) ? LY::DL : 8;
    constexpr int LH = (G == 1) ? LY::LH : D / 8;
    constexpr int LT = (G == 1) ? LY::LT : D / 8;
    constexpr int GS = (G == 1) ? 1 : G; // heads a lane carries
    const int sub = lane % LH, gl = (G == 1) ? 0 : 0, tg = lane / LT;
    uint32_t tau = 0;
    int nu = 0; // this CTA's units so far
    for (int u = blockIdx.x; u < U; u += gridDim.x, ++nu) {
        const Unit un = unit_info(u, pf, pp, nb, S, a.hkv, bps, a.start_block);
        const int L = a.lens[un.s];
        float qs = a.qk_scale_log2;
        if constexpr (KVT == PKV_FP8_E4M3) qs *= a.k_scale[un.kvh];
        float qf[GS][DL];
#pragma unroll
        for (int g = 0; g < GS; ++g) {
            const T *qp = static_cast<const T *>(a.q) + ((int64_t)un.s * a.hq + un.kvh * G + g + gl) * D + sub * DL;
#pragma unroll
            for (int c = 0; c < DL / 8; ++c) cvt8<MT>(reinterpret_cast<const uint4 *>(qp)[c], qf[g] + 8 * c);
#pragma unroll
            for (int e = 0; e < DL; ++e) qf[g][e] *= qs;
        }
        float m[GS], l[GS], acc[GS][DL];
#pragma unroll
        for (int g = 0; g < GS; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int e = 0; e < DL; ++e) acc[g][e] = 0.f;
        }
        // Tile t of the CTA's stream (t counted over all its units) belongs to warp t % NCW and
        // sits in stage t % NST with NST a multiple of NCW, so a warp's previous tile in any stage
        // is its own: when it waits for phase k of a stage, phase k-1 has completed, which keeps
        // the parity wait unambiguous.
        int i0 = warp - static_cast<int>(tau % NCW);
        if (i0 < 0) i0 += NCW;
        const int nt = spb > 1 ? min(un.ntiles * spb, (L - un.blk0 * a.bs + ST - 1) / ST) : un.ntiles;
        for (int i = i0; i < nt; i += NCW) {
            const uint32_t t = tau + i;
            const uint32_t stage = t % NST;
            if (!mbar_wait(&full[stage], (t / NST) & 1)) {
                set_error(a.err, PKV_DEVERR_TIMEOUT);
                *reinterpret_cast<volatile int *>(abort_flag) = 1;
            }
            if (*reinterpret_cast<volatile int *>(abort_flag)) break;
            if (!flags[stage]) {
                const char *ks = ring + (size_t)stage * 2 * a.sub_bytes;
                const int valid = min(ST, L - un.blk0 * a.bs - i * ST);
                if constexpr (G == 1)
                    process_tile<D, 1, KVT>(ks, ks + a.sub_bytes, ST, valid, qf[0], m[0], l[0], acc[0], lane);
                else
                    process_tile_tp<D, G, KVT>(ks, ks + a.sub_bytes, ST, valid, qf, m, l, acc, lane);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
        }
        tau += nt;
        // combine the token groups of this warp (same heads, same dims); for G >= 2 the row sums are
        // spread over all lanes
#pragma unroll
        for (int g = 0; g < GS; ++g) {
            if constexpr (G == 1) {
#pragma unroll
                for (int o = LT; o < 32; o <<= 1) l[g] += __shfl_xor_sync(0xffffffffu, l[g], o);
            } else {
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) l[g] += __shfl_xor_sync(0xffffffffu, l[g], o);
            }
#pragma unroll
            for (int o = LT; o < 32; o <<= 1)
#pragma unroll
                for (int e = 0; e < DL; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], o);
        }
        // merge slot nu % 2 is free once the merge of this CTA's unit nu - 2 is done
        const int sp = nu & 1;
        float *slot = mrg + sp * (NCW * G * (D + 2));
        bool ok = true;
        if (lane == 0) {
            ok = wait_at_least(mdone + sp, nu >> 1, abort_flag);
            __threadfence_block(); // the merger's reads of the slot come before this warp's writes
        }
        __syncwarp();
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) {
            set_error(a.err, PKV_DEVERR_TIMEOUT);
            *reinterpret_cast<volatile int *>(abort_flag) = 1;
        }
        if (*reinterpret_cast<volatile int *>(abort_flag)) break;
        if (tg == 0) {
#pragma unroll
            for (int g = 0; g < GS; ++g) {
                float *r = slot + (warp * G + g + gl) * (D + 2);
#pragma unroll
                for (int e = 0; e < DL; ++e) r[sub * DL + e] = acc[g][e];
                if (sub == 0) {
                    r[D] = m[g];
                    r[D + 1] = l[g];
                }
            }
        }
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block(); // this warp's partial, then its hand-in
            last = atomicAdd(mcount + sp, 1) == NCW - 1;
            __threadfence_block(); // the last hand-in, then the other warps' partials
        }
        __syncwarp();
        if (!__shfl_sync(0xffffffffu, last, 0)) continue;
        // the last warp to hand in: merge the four warps' partials in warp order
        if (lane == 0) mcount[sp] = 0; // no warp hands in to this slot before mdone[sp] moves on
        const float vs = (KVT == PKV_FP8_E4M3) ? a.v_scale[un.kvh] : 1.f;
        for (int o = lane; o < G * D; o += 32) {
            const int g = o / D, d = o - g * D;
            float Mx = -INFINITY;
#pragma unroll
            for (int w = 0; w < NCW; ++w) {
                const float *r = slot + (w * G + g) * (D + 2);
                if (r[D + 1] > 0.f) Mx = fmaxf(Mx, r[D]);
            }
            float num = 0.f, den = 0.f;
#pragma unroll
            for (int w = 0; w < NCW; ++w) {
                const float *r = slot + (w * G + g) * (D + 2);
                if (r[D + 1] > 0.f) {
                    const float wt = fast_exp2(r[D] - Mx);
                    num = fmaf(wt, r[d], num);
                    den = fmaf(wt, r[D + 1], den);
                }
            }
            const int h = un.kvh * G + g;
            if (un.nsplit == 1 && a.slot0 == 0) {
                const float y = den > 0.f ? (num / den) * vs : 0.f;
                static_cast<T *>(a.out)[((int64_t)un.s * a.hq + h) * D + d] = M::from_f(y);
            } else {
                const int64_t idx = ((int64_t)un.s * a.hq + h) * a.max_splits + a.slot0 + un.j;
                a.ws_o[idx * D + d] = num * vs;
                if (d == 0) reinterpret_cast<float2 *>(a.ws_ml)[idx] = make_float2(Mx, den);
            }
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            *reinterpret_cast<volatile int *>(mdone + sp) = mdone[sp] + 1;
        }
    }
}

// Merge of the per-split partials of sequences with more than one split; zero rows for
// L_s == 0.  One CTA of four warps per (sequence, query head) row: every warp forms the common
// max M from all splits' (m, l), then accumulates the splits j = warp, warp + 4, ... (lane = D/32
// dims, vector loads; the first 16 splits' loads go out with those of the maxima); the four warp
// sums are added in warp order through shared memory, so the result is deterministic.
template <int D, int MT>
__global__ void __launch_bounds__(128) merge_kernel(const Args a) {
    using M = ModelT<MT>;
    using T = typename M::T;
    constexpr int PER = D / 32;
    __shared__ float s_num[4][D];
    __shared__ float s_den[4];
    // No early trigger: the kernel after the merge (typically the next decode step's append, then
    // its decode kernel, whose persistent CTAs fill the SMs) launches when the merge has finished,
    // rather than taking SM room from the merge's own CTAs while it runs.
    pdl_wait();
    const int row = blockIdx.x, warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int s = row / a.hq;
    const int L = a.lens[s];
    int n = L > 0 ? (L + a.bs - 1) / a.bs : 0;
    if (n > a.max_blocks) n = a.max_blocks;
    if (a.slot0 > 0 && L < a.start_block * a.bs) {
        // cascade: a sequence shorter than the shared prefix it claims
        if (threadIdx.x == 0 && row % a.hq == 0) set_error(a.err, PKV_DEVERR_LENGTH);
    }
    const int m = n > a.start_block ? n - a.start_block : 0;
    const int nsplit = a.slot0 + m / a.split_blocks + ((m % a.split_blocks) ? 1 : 0);
    if (nsplit == 1 && a.slot0 == 0) return;
    T *o = static_cast<T *>(a.out) + (int64_t)row * D;
    if (nsplit == 0) {
        for (int e = threadIdx.x; e < D; e += blockDim.x) o[e] = M::from_f(0.f);
        return;
    }
    const int64_t base = (int64_t)row * a.max_splits;
    const float2 *ml = reinterpret_cast<const float2 *>(a.ws_ml) + base;
    // this warp's splits j0, j0 + 4, ... (U of them): (m, l) and its lane's dims of o
    constexpr int U = 4;
    float2 mlj[U];
    float vj[U][PER];
    auto load_group = [&](int j0) {
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int j = j0 + 4 * k;
            if (j < nsplit) {
                mlj[k] = ml[j];
                const float *src = a.ws_o + (base + j) * D + lane * PER;
                if constexpr (PER == 4) {
                    const float4 v = *reinterpret_cast<const float4 *>(src);
                    vj[k][0] = v.x;
                    vj[k][1] = v.y;
                    vj[k][2] = v.z;
                    vj[k][3] = v.w;
                } else {
                    const float2 v = *reinterpret_cast<const float2 *>(src);
                    vj[k][0] = v.x;
                    vj[k][1] = v.y;
                }
            } else {
                mlj[k] = make_float2(0.f, 0.f);
            }
        }
    };
    // the first group (all splits of a row with up to 16) is loaded with the maxima's (m, l), so the
    // row takes one round trip to memory instead of two
    load_group(warp);
    float Mx = -INFINITY;
    for (int j = lane; j < nsplit; j += 32) {
        const float2 v = ml[j];
        if (v.y > 0.f) Mx = fmaxf(Mx, v.x);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, off));
    float num[PER], den = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) num[e] = 0.f;
    for (int j0 = warp; j0 < nsplit; j0 += 4 * U) {
        if (j0 != warp) load_group(j0);
#pragma unroll
        for (int k = 0; k < U; ++k) {
            if (mlj[k].y > 0.f) {
                const float w = fast_exp2(mlj[k].x - Mx);
                den = fmaf(w, mlj[k].y, den);
#pragma unroll
                for (int e = 0; e < PER; ++e) num[e] = fmaf(w, vj[k][e], num[e]);
            }
        }
    }
#pragma unroll
    for (int e = 0; e < PER; ++e) s_num[warp][lane * PER + e] = num[e];
    if (lane == 0) s_den[warp] = den;
    __syncthreads();
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        const float tn = ((s_num[0][d] + s_num[1][d]) + s_num[2][d]) + s_num[3][d];
        const float td = ((s_den[0] + s_den[1]) + s_den[2]) + s_den[3];
        o[d] = M::from_f(td > 0.f ? tn / td : 0.f);
    }
}

inline size_t smem_bytes(int D, int G, int nst, int stage_part_bytes, int S) {
    return (size_t)nst * 2 * stage_part_bytes + (size_t)nst * (8 + 8 + 4) + 32 + (size_t)2 * kConsumerWarps * G * (D + 2) * 4 +
           (size_t)(3 * S + 2) * 4;
}

template <int D, int G, int MT, int KVT>
cudaError_t launch_t(const Args &a, int grid, size_t smem, cudaStream_t st) {
    auto kern = decode_kernel<D, G, MT, KVT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return pdl_launch(kern, dim3(grid), dim3(kThreads), smem, st, a);
}

template <int D, int MT>
cudaError_t launch_merge_t(const Args &a, cudaStream_t st) {
    const int rows = a.num_seqs * a.hq;
    if (rows == 0) return cudaSuccess;
    return pdl_launch(merge_kernel<D, MT>, dim3(rows), dim3(128), 0, st, a);
}

// Dispatch over head_dim and group size for one (model dtype, KV dtype) pair.
template <int MT, int KVT>
cudaError_t dispatch(const Args &a, int D, int G, int grid, size_t smem, cudaStream_t st, bool merge) {
#define PKV_CASE(DD, GG)                                                                                               \
    if (D == DD && G == GG) return merge ? launch_merge_t<DD, MT>(a, st) : launch_t<DD, GG, MT, KVT>(a, grid, smem, st);
    PKV_CASE(64, 1)
    PKV_CASE(64, 2)
    PKV_CASE(64, 4)
    PKV_CASE(64, 8)
    PKV_CASE(128, 1)
    PKV_CASE(128, 2)
    PKV_CASE(128, 4)
    PKV_CASE(128, 8)
#undef PKV_CASE
    return cudaErrorInvalidValue;
}

template <int D, int G, int MT, int KVT>
int occupancy(size_t smem) {
    int n = 0;
    cudaFuncSetAttribute(decode_kernel<D, G, MT, KVT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<D, G, MT, KVT>, kThreads, smem);
    return n;
}

template <int MT, int KVT>
int occupancy_dispatch(int D, int G, size_t smem) {
#define PKV_CASE(DD, GG)                                                                                               \
    if (D == DD && G == GG) return occupancy<DD, GG, MT, KVT>(smem);
    PKV_CASE(64, 1)
    PKV_CASE(64, 2)
    PKV_CASE(64, 4)
    PKV_CASE(64, 8)
    PKV_CASE(128, 1)
    PKV_CASE(128, 2)
    PKV_CASE(128, 4)
    PKV_CASE(128, 8)
#undef PKV_CASE
    return 0;
}

} // namespace pkv_decode

// Per (model dtype, KV dtype) entry points, each compiled in its own translation unit.
cudaError_t pkv_decode_f16(const pkv_decode::Args &, int D, int G, int grid, size_t smem, cudaStream_t, bool merge);
cudaError_t pkv_decode_bf16(const pkv_decode::Args &, int D, int G, int grid, size_t smem, cudaStream_t, bool merge);
cudaError_t pkv_decode_fp8_f16(const pkv_decode::Args &, int D, int G, int grid, size_t smem, cudaStream_t,
                               bool merge);
cudaError_t pkv_decode_fp8_bf16(const pkv_decode::Args &, int D, int G, int grid, size_t smem, cudaStream_t,
                                bool merge);
int pkv_decode_occupancy_f16(int D, int G, size_t smem);
int pkv_decode_occupancy_bf16(int D, int G, size_t smem);
int pkv_decode_occupancy_fp8_f16(int D, int G, size_t smem);
int pkv_decode_occupancy_fp8_bf16(int D, int G, size_t smem);
