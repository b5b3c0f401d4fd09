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
//  * Work unit = (sequence, KV head, split), a split being up to `split_blocks` (<= 32)
//    consecutive logical blocks.  Splits are block-aligned and depend only on L_s, so the
//    arithmetic order of every output is fixed by the lengths alone (placement of physical
//    blocks, sharing of prefix blocks and the batch composition never change a bit).
//  * Persistent CTAs (as many as fit per SM); every warp is an independent worker.  Units are
//    listed full splits first, partial tail splits last, and go round-robin over all warps of
//    the grid.
//  * A warp owns a ring of `nstages` shared-memory stages.  Its lane 0 issues one 1-D bulk async
//    copy (cp.async.bulk, the TMA's linear mode) per (block, K|V, head) tile, completion tracked by
//    an mbarrier transaction count; it refills a stage right after the warp has consumed it, so the
//    ring runs `nstages` tiles ahead across unit boundaries and needs no "empty" barrier.  The pool
//    layout [block][K|V][head][offset][dim] makes each tile one contiguous bs*D*elt-byte run (4 KB
//    for bs=16, D=128, fp16): one table lookup yields two large aligned copies, issued with an L2
//    evict-first hint because KV is streamed once.  Block ids for a unit are read once, one per
//    lane, and moved to lane 0 with a shuffle.
//  * In a warp, D/8 lanes share a token (16-byte vector loads from shared memory, conflict-free),
//    partial dot products are reduced with xor-shuffles, and an online softmax (running max m, sum l,
//    rescaled accumulator) runs per 16-token chunk with exp2 on prescaled scores.
//  * A sequence with one split writes its output row at the end of its unit.  Otherwise the warp
//    writes an fp32 partial (m, l, unnormalised o), and its lane 0 fences and bumps a per-(sequence,
//    KV head) counter; the warp that finishes the last split combines all partials in split order
//    and resets the counter (so the merge order, and every output bit, does not depend on which warp
//    is last).  A warp's unit-end work never blocks the other warps.
//  * Every mbarrier wait is bounded (PKV_WAIT_LIMIT_NS); a timeout sets PKV_DEVERR_TIMEOUT, the warp
//    waits (bounded) for its own copies in flight and stops.
#pragma once

#include "device_common.cuh"
#include "pkv_internal.h"

namespace pkv_decode {

constexpr int kMaxWarps = 4;
constexpr int kMaxSeqs = 1024;

struct Args {
    const void *q;
    void *out;
    const char *pool;
    const float *k_scale, *v_scale;
    const int32_t *tables, *lens;
    float *ws_o, *ws_ml; // split partials: o [rows][D], (m, l) [rows][2], rows = S * Hq * max_splits
    int *counters;       // [S * Hkv] finished split units per (sequence, KV head); zero between launches
    unsigned int *err;
    int64_t num_blocks;
    int64_t blk_stride;  // bytes between consecutive physical blocks
    int64_t kv_stride;   // bytes between the K and V halves of a block
    int tile_bytes;      // one (block, K|V, head) tile
    int max_blocks, num_seqs, hq, hkv, bs;
    int split_blocks, max_splits, nstages;
    float qk_scale_log2; // scale * log2(e)
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

PKV_DEV Unit unit_info(int u, const int *pf, const int *pp, const int *nb, int S, int hkv, int bps) {
    Unit r;
    const int nfull_units = pf[S] * hkv;
    if (u < nfull_units) {
        const int k = u / hkv;
        r.kvh = u - k * hkv;
        r.s = find_row(pf, S, k);
        r.j = k - pf[r.s];
        r.blk0 = r.j * bps;
        r.ntiles = bps;
    } else {
        const int u2 = u - nfull_units;
        const int k = u2 / hkv;
        r.kvh = u2 - k * hkv;
        r.s = find_row(pp, S, k);
        r.j = pf[r.s + 1] - pf[r.s];
        r.blk0 = r.j * bps;
        r.ntiles = nb[r.s] - r.blk0;
    }
    r.nsplit = (pf[r.s + 1] - pf[r.s]) + (pp[r.s + 1] - pp[r.s]);
    return r;
}

// One tile of `bs` tokens, `valid` of them real, for the G query heads of one KV head.
template <int D, int G, int KVT>
PKV_DEV void process_tile(const char *ks, const char *vs, int bs, int valid, const float (&qf)[G][8], float (&m)[G],
                          float (&l)[G], float (&acc)[G][8], int lane) {
    constexpr int LPT = D / 8;        // lanes per token
    constexpr int TPP = 32 / LPT;     // tokens per pass
    constexpr int MAXP = 16 / TPP;    // passes per 16-token chunk
    constexpr int EB = (KVT == PKV_FP8_E4M3) ? 1 : 2;
    const int sub = lane % LPT, grp = lane / LPT;
    const int ch = bs < 16 ? bs : 16;
    const int npc = ch / TPP;
    for (int c0 = 0; c0 < bs; c0 += ch) {
        if (c0 >= valid) break;
        float sc[G][MAXP];
#pragma unroll
        for (int p = 0; p < MAXP; ++p) {
            if (p < npc) {
                const int t = c0 + p * TPP + grp;
                float kf[8];
                load8<KVT>(ks + (t * D + sub * 8) * EB, kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float d0 = 0.f;
#pragma unroll
                    for (int e = 0; e < 8; ++e) d0 = fmaf(qf[g][e], kf[e], d0);
                    sc[g][p] = d0;
                }
            }
        }
#pragma unroll
        for (int p = 0; p < MAXP; ++p) {
            if (p < npc) {
                const bool live = (c0 + p * TPP + grp) < valid;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float v = sc[g][p];
#pragma unroll
                    for (int o = LPT / 2; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    sc[g][p] = live ? v : -INFINITY;
                }
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mx = -INFINITY;
#pragma unroll
            for (int p = 0; p < MAXP; ++p)
                if (p < npc) mx = fmaxf(mx, sc[g][p]);
#pragma unroll
            for (int o = LPT; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            const float mn = fmaxf(m[g], mx); // finite: the chunk holds at least one live token
            const float alpha = fast_exp2(m[g] - mn);
            m[g] = mn;
            l[g] *= alpha;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] *= alpha;
#pragma unroll
            for (int p = 0; p < MAXP; ++p) {
                if (p < npc) {
                    const float pr = fast_exp2(sc[g][p] - mn);
                    sc[g][p] = pr;
                    l[g] += pr;
                }
            }
        }
#pragma unroll
        for (int p = 0; p < MAXP; ++p) {
            if (p < npc) {
                const int t = c0 + p * TPP + grp;
                if (t < valid) {
                    float vf[8];
                    load8<KVT>(vs + (t * D + sub * 8) * EB, vf);
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int e = 0; e < 8; ++e) acc[g][e] = fmaf(sc[g][p], vf[e], acc[g][e]);
                }
            }
        }
    }
}

PKV_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
PKV_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Combine the split partials of (sequence s, KV head kvh) and write the rows of its G query heads,
// one warp.  The weights exp2(m_j - M) are formed per split; the sums run in a fixed order.
// Partials written by other warps are read through L2 (ld.global.cg).
template <int D, int G, int MT>
PKV_DEV void merge_splits_warp(const Args &a, int s, int kvh, int nsplit, int lane) {
    using M = ModelT<MT>;
    using T = typename M::T;
    constexpr int PER = D / 32;
#pragma unroll 1
    for (int g = 0; g < G; ++g) {
        const int h = kvh * G + g;
        const int64_t base = ((int64_t)s * a.hq + h) * a.max_splits;
        float Mx = -INFINITY;
        for (int j = lane; j < nsplit; j += 32) {
            const float lj = __ldcg(a.ws_ml + 2 * (base + j) + 1);
            if (lj > 0.f) Mx = fmaxf(Mx, __ldcg(a.ws_ml + 2 * (base + j)));
        }
        Mx = warp_max(Mx);
        float num[PER], den = 0.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) num[e] = 0.f;
        for (int j0 = 0; j0 < nsplit; j0 += 32) {
            const int j = j0 + lane;
            float wj = 0.f, lj = 0.f;
            if (j < nsplit) {
                lj = __ldcg(a.ws_ml + 2 * (base + j) + 1);
                if (lj > 0.f) wj = fast_exp2(__ldcg(a.ws_ml + 2 * (base + j)) - Mx);
            }
            den += warp_sum(wj * lj);
            const int cnt = min(32, nsplit - j0);
            for (int jj = 0; jj < cnt; ++jj) {
                const float w = __shfl_sync(0xffffffffu, wj, jj);
                const float *src = a.ws_o + (base + j0 + jj) * D + lane * PER;
                if constexpr (PER == 4) {
                    const float4 o4 = __ldcg(reinterpret_cast<const float4 *>(src));
                    num[0] = fmaf(w, o4.x, num[0]);
                    num[1] = fmaf(w, o4.y, num[1]);
                    num[2] = fmaf(w, o4.z, num[2]);
                    num[3] = fmaf(w, o4.w, num[3]);
                } else {
                    const float2 o2 = __ldcg(reinterpret_cast<const float2 *>(src));
                    num[0] = fmaf(w, o2.x, num[0]);
                    num[1] = fmaf(w, o2.y, num[1]);
                }
            }
        }
        T *orow = static_cast<T *>(a.out) + ((int64_t)s * a.hq + h) * D + lane * PER;
#pragma unroll
        for (int e = 0; e < PER; ++e) orow[e] = M::from_f(den > 0.f ? num[e] / den : 0.f);
    }
}

template <int D, int G, int MT, int KVT>
__global__ void __launch_bounds__(kMaxWarps * 32) decode_kernel(const Args a) {
    using M = ModelT<MT>;
    using T = typename M::T;
    constexpr int LPT = D / 8;
    extern __shared__ __align__(128) unsigned char smem[];
    const int NW = blockDim.x >> 5;
    const int NST = a.nstages;
    const int S = a.num_seqs;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const size_t stage_bytes = 2 * (size_t)a.tile_bytes;
    char *ring = reinterpret_cast<char *>(smem) + (size_t)warp * NST * stage_bytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)NW * NST * stage_bytes) + warp * NST;
    int *flags = reinterpret_cast<int *>(reinterpret_cast<uint64_t *>(smem + (size_t)NW * NST * stage_bytes) +
                                         NW * NST) + warp * NST;
    int *pf = reinterpret_cast<int *>(reinterpret_cast<uint64_t *>(smem + (size_t)NW * NST * stage_bytes) + NW * NST) +
              NW * NST;
    int *pp = pf + (S + 1);
    int *nb = pp + (S + 1);

    if (lane == 0) {
        for (int i = 0; i < NST; ++i) mbar_init(&full[i], 1);
        fence_mbarrier_init();
    }
    // unit list: per sequence, full splits and (0 or 1) partial split
    const int bps = a.split_blocks;
    for (int s = threadIdx.x; s < S; s += blockDim.x) {
        const int L = a.lens[s];
        int n = L > 0 ? (L + a.bs - 1) / a.bs : 0;
        if (n > a.max_blocks) {
            if (blockIdx.x == 0) set_error(a.err, PKV_DEVERR_LENGTH);
            n = a.max_blocks;
        }
        nb[s] = n;
        pf[s + 1] = n / bps;
        pp[s + 1] = (n % bps) ? 1 : 0;
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
    const int U = (pf[S] + pp[S]) * a.hkv;
    // rows of sequences with no tokens are zero (no unit covers them)
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < (int64_t)S * a.hq * D;
         e += (int64_t)gridDim.x * blockDim.x)
        if (nb[e / ((int64_t)a.hq * D)] == 0) static_cast<T *>(a.out)[e] = M::from_f(0.f);

    const int gw = blockIdx.x * NW + warp, TW = gridDim.x * NW;
    const uint64_t policy = l2_policy_evict_first();

    // ---- issue side: runs `NST` tiles ahead of consumption over this warp's unit sequence
    int iu = gw, it = 0;
    Unit iun{};
    int irow = 0; // block id of tile `lane` of unit iu
    if (iu < U) {
        iun = unit_info(iu, pf, pp, nb, S, a.hkv, bps);
        irow = lane < iun.ntiles ? a.tables[(int64_t)iun.s * a.max_blocks + iun.blk0 + lane] : 0;
    }
    uint32_t issued = 0, consumed = 0;
    auto issue_one = [&]() {
        while (iu < U && it >= iun.ntiles) {
            iu += TW;
            it = 0;
            if (iu < U) {
                iun = unit_info(iu, pf, pp, nb, S, a.hkv, bps);
                irow = lane < iun.ntiles ? a.tables[(int64_t)iun.s * a.max_blocks + iun.blk0 + lane] : 0;
            }
        }
        if (iu >= U) return;
        const int b = __shfl_sync(0xffffffffu, irow, it);
        if (lane == 0) {
            const uint32_t st = issued % NST;
            char *dst = ring + st * stage_bytes;
            if (b >= 0 && b < a.num_blocks) {
                flags[st] = 0;
                const char *src = a.pool + (int64_t)iun.kvh * a.tile_bytes + (int64_t)b * a.blk_stride;
                mbar_arrive_expect_tx(&full[st], 2u * a.tile_bytes);
                bulk_g2s_hint(dst, src, a.tile_bytes, &full[st], policy);
                bulk_g2s_hint(dst + a.tile_bytes, src + a.kv_stride, a.tile_bytes, &full[st], policy);
            } else {
                flags[st] = 1;
                set_error(a.err, PKV_DEVERR_BLOCK_ID);
                mbar_arrive(&full[st]);
            }
        }
        ++it;
        ++issued;
    };
    for (int k = 0; k < NST; ++k) issue_one();

    // ---- consume side
    const int sub = lane % LPT, grp = lane / LPT;
    bool ok = true;
    for (int u = gw; u < U && ok; u += TW) {
        const Unit un = unit_info(u, pf, pp, nb, S, a.hkv, bps);
        const int L = a.lens[un.s];
        float qs = a.qk_scale_log2;
        if constexpr (KVT == PKV_FP8_E4M3) qs *= a.k_scale[un.kvh];
        float qf[G][8];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const T *qp = static_cast<const T *>(a.q) + ((int64_t)un.s * a.hq + un.kvh * G + g) * D + sub * 8;
            cvt8<MT>(*reinterpret_cast<const uint4 *>(qp), qf[g]);
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[g][e] *= qs;
        }
        float m[G], l[G], acc[G][8];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            m[g] = -INFINITY;
            l[g] = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[g][e] = 0.f;
        }
        for (int i = 0; i < un.ntiles; ++i) {
            const uint32_t st = consumed % NST;
            if (!mbar_wait(&full[st], (consumed / NST) & 1)) ok = false;
            if (!__all_sync(0xffffffffu, ok)) {
                ok = false;
                break;
            }
            if (!flags[st]) {
                const char *ks = ring + st * stage_bytes;
                const int valid = min(a.bs, L - (un.blk0 + i) * a.bs);
                process_tile<D, G, KVT>(ks, ks + a.tile_bytes, a.bs, valid, qf, m, l, acc, lane);
            }
            __syncwarp();
            ++consumed;
            issue_one(); // refills the stage just consumed
        }
        if (!ok) break;
        // combine the token groups of this warp
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int o = LPT; o < 32; o <<= 1) {
                l[g] += __shfl_xor_sync(0xffffffffu, l[g], o);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], o);
            }
        }
        const float vs = (KVT == PKV_FP8_E4M3) ? a.v_scale[un.kvh] : 1.f;
        if (un.nsplit == 1) {
            if (grp == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float r = l[g] > 0.f ? vs / l[g] : 0.f;
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) w[e] = M::pack(acc[g][2 * e] * r, acc[g][2 * e + 1] * r);
                    T *orow = static_cast<T *>(a.out) + ((int64_t)un.s * a.hq + un.kvh * G + g) * D + sub * 8;
                    *reinterpret_cast<uint4 *>(orow) = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        } else {
            if (grp == 0) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const int64_t idx = ((int64_t)un.s * a.hq + un.kvh * G + g) * a.max_splits + un.j;
                    float *dst = a.ws_o + idx * D + sub * 8;
                    reinterpret_cast<float4 *>(dst)[0] =
                        make_float4(acc[g][0] * vs, acc[g][1] * vs, acc[g][2] * vs, acc[g][3] * vs);
                    reinterpret_cast<float4 *>(dst)[1] =
                        make_float4(acc[g][4] * vs, acc[g][5] * vs, acc[g][6] * vs, acc[g][7] * vs);
                    if (sub == 0) reinterpret_cast<float2 *>(a.ws_ml)[idx] = make_float2(m[g], l[g]);
                }
            }
            __syncwarp();
            int last = 0;
            int *cnt = a.counters + (int64_t)un.s * a.hkv + un.kvh;
            if (lane == 0) {
                __threadfence();
                last = (atomicAdd(cnt, 1) == un.nsplit - 1) ? 1 : 0;
            }
            last = __shfl_sync(0xffffffffu, last, 0);
            if (last) {
                __threadfence();
                merge_splits_warp<D, G, MT>(a, un.s, un.kvh, un.nsplit, lane);
                if (lane == 0) *cnt = 0;
            }
        }
    }
    if (!ok) {
        // a wait gave up: record it, let this warp's copies in flight land (bounded), stop
        if (lane == 0) {
            set_error(a.err, PKV_DEVERR_TIMEOUT);
            for (uint32_t t = consumed; t < issued; ++t) mbar_wait(&full[t % NST], (t / NST) & 1);
        }
    }
}

// Shared memory of one CTA of `nw` warps with `nst` stages each.
inline size_t smem_bytes(int nw, int nst, int tile_bytes, int S) {
    return (size_t)nw * nst * (2 * (size_t)tile_bytes + 8 + 4) + (size_t)(3 * S + 2) * 4;
}

template <int D, int G, int MT, int KVT>
cudaError_t launch_t(const Args &a, int grid, int threads, size_t smem, cudaStream_t st) {
    auto kern = decode_kernel<D, G, MT, KVT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, threads, smem, st>>>(a);
    return cudaGetLastError();
}

template <int D, int G, int MT, int KVT>
int occupancy(int threads, size_t smem) {
    int n = 0;
    cudaFuncSetAttribute(decode_kernel<D, G, MT, KVT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<D, G, MT, KVT>, threads, smem);
    return n;
}

// Dispatch over head_dim and group size for one (model dtype, KV dtype) pair: occupancy query
// when grid == 0, launch otherwise.
template <int MT, int KVT>
cudaError_t dispatch(const Args &a, int D, int G, int grid, int threads, size_t smem, cudaStream_t st, int *occ) {
#define PKV_CASE(DD, GG)                                                                                               \
    if (D == DD && G == GG) {                                                                                          \
        if (occ) {                                                                                                     \
            *occ = occupancy<DD, GG, MT, KVT>(threads, smem);                                                          \
            return cudaSuccess;                                                                                        \
        }                                                                                                              \
        return launch_t<DD, GG, MT, KVT>(a, grid, threads, smem, st);                                                  \
    }
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

} // namespace pkv_decode

// Per (model dtype, KV dtype) entry points, each compiled in its own translation unit.
using PkvDecodeFn = cudaError_t (*)(const pkv_decode::Args &, int D, int G, int grid, int threads, size_t smem,
                                    cudaStream_t, int *occ);
cudaError_t pkv_decode_f16(const pkv_decode::Args &, int, int, int, int, size_t, cudaStream_t, int *);
cudaError_t pkv_decode_bf16(const pkv_decode::Args &, int, int, int, int, size_t, cudaStream_t, int *);
cudaError_t pkv_decode_fp8_f16(const pkv_decode::Args &, int, int, int, int, size_t, cudaStream_t, int *);
cudaError_t pkv_decode_fp8_bf16(const pkv_decode::Args &, int, int, int, int, size_t, cudaStream_t, int *);
