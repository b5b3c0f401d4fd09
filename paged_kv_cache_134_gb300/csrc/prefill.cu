// Packed causal prefill on the 5th-generation tensor cores, with the paged K/V write fused in.
//
// What it computes ("Paged KV Cache 与 Packed Sequence", discosf.com, sections 3.1-3.3, 4.2):
// sequences packed back to back, sequence i owning rows [cu[i], cu[i+1]); a query at in-sequence
// position r attends to the keys of its own sequence at positions c <= r (block-diagonal causal
// mask), out = softmax(scale q.k) v.  Every token's k/v is also written into the paged cache at
// block_table[i][r / bs], offset r % bs (the prompt-phase write of section 4.2, bounded by the
// sequence length so a partly filled tail block is never overrun).
//
// One CTA = (sequence, 128-query tile, query head).  Warp roles:
//   warp 0     TMA producers: lane 0 loads the Q tile once and K tiles of 64 keys into a 2-stage ring,
//              lane 1 V tiles into another (tiled TMA, 128-byte swizzle, out-of-range rows zero-filled);
//              a K stage frees when S = Q K^T of its tile is done, a V stage when P V is done;
//   warp 1     tensor-memory owner and MMA issuer (one thread): S = Q K^T into one of two TMEM S
//              buffers (M=128, N=64, fp32), then O += P V into the TMEM O accumulator (M=128, N=D);
//   warps 2-5  softmax, one thread per query row (TMEM lane = row): mask, exp2, row sums, P written
//              to shared memory in the 128-byte-swizzled K-major layout the MMA reads (fp16 P for
//              fp16 models; for bf16 models P = hi + lo, two bf16 tiles and two accumulating MMAs); O in TMEM is rescaled only when a row's running max grows by
//              more than 2^8 (the exponent base stays fixed otherwise, which is exact algebra);
//   warps 6-7  paged K/V writer for the tile's rows, straight from the K/V tiles already in shared
//              memory (only the CTA of the first query head of each KV group writes, so every
//              (token, KV head) is written once).
// The diagonal tiles are masked per element; tiles entirely above the diagonal are never issued.
// Every mbarrier wait is bounded; a timeout sets PKV_DEVERR_TIMEOUT and the CTA winds down.
#include <algorithm>
#include <mutex>

#include "tcgen05.cuh"
#include "pkv_internal.h"

namespace pkv_prefill {

constexpr int BM = 128;          // query rows per tile (MMA M)
constexpr int BN = 64;           // keys per tile (MMA N of Q K^T, K of P V)
constexpr int kThreads = 256;
constexpr uint32_t kTmemCols = 256; // S0 [0,64) S1 [64,128) O [128, 128+D)
constexpr float kRescale = 8.0f; // log2 units

struct Args {
    const char *k, *v;  // packed [T][Hkv][D]
    void *out;          // packed [T][Hq][D]
    const int32_t *cu, *tables;
    char *pool;
    unsigned int *err;
    int64_t total_tokens, num_blocks, tile_elems;
    int num_seqs, max_seqlen, max_blocks, hq, hkv, bs, nqt_max;
    float scale_log2;
};

// Shared memory.  bf16 models keep P as a hi + lo pair of bf16 tiles (P = hi + lo to ~2^-16
// relative), because one bf16 rounding of P (2^-9 relative) alone would exceed the accuracy the
// outputs are held to; fp16 P (2^-12) is used as a single tile.
template <int D, int MT>
struct Layout {
    static constexpr int NP = MT == PKV_BF16 ? 2 : 1;
    static constexpr int Q = 0;
    static constexpr int Q_BYTES = BM * D * 2;
    static constexpr int KV_BYTES = BN * D * 2; // one K or V tile
    static constexpr int K0 = Q + Q_BYTES;
    static constexpr int V0 = K0 + 2 * KV_BYTES;
    static constexpr int P = V0 + 2 * KV_BYTES;
    static constexpr int P_BYTES = BM * BN * 2;
    static constexpr int BAR = P + NP * P_BYTES;
    static constexpr int TOTAL = BAR + 256;
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

template <int D, int MT>
__global__ void __launch_bounds__(kThreads, min_blocks<D, MT>())
    prefill_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, const Args a) {
    using L = Layout<D, MT>;
    extern __shared__ __align__(1024) uint8_t smem[];

    pdl_trigger();
    pdl_wait();
    // ---- work item.  Items are (sequence, query tile) pairs, hq CTAs (one per query head) each, in
    // rank order: rank r holds every sequence's r-th heaviest query tile (its (nq-1-r)-th), so the
    // longest tiles start first.  The grid is sized from the packed token count (at most
    // T/BM + num_seqs items), and each CTA finds its item from a histogram of per-sequence tile
    // counts kept, for this prologue only, in the P buffer's shared memory.
    int *nq = reinterpret_cast<int *>(smem + L::P);
    int *hist = nq + a.num_seqs;          // [nqt_max + 1]
    int *pick = hist + a.nqt_max + 1;     // seq, qt
    for (int x = threadIdx.x; x <= a.nqt_max; x += blockDim.x) hist[x] = 0;
    __syncthreads();
    for (int i = threadIdx.x; i < a.num_seqs; i += blockDim.x) {
        const int st = a.cu[i], en = a.cu[i + 1];
        int c = 0;
        if (st < 0 || en < st || en > a.total_tokens || en - st > a.max_seqlen) {
            if (blockIdx.x == 0) set_error(a.err, PKV_DEVERR_CU_SEQLENS);
        } else {
            c = (en - st + BM - 1) / BM;
        }
        nq[i] = c;
        atomicAdd(&hist[c], 1);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        int k = blockIdx.x / a.hq, r = 0, above = a.num_seqs - hist[0]; // above = #{i : nq_i > r}
        while (r < a.nqt_max && k >= above) {
            k -= above;
            ++r;
            above -= hist[r];
        }
        int seq_found = -1;
        if (r < a.nqt_max) {
            for (int base = 0; base < a.num_seqs; base += 32) {
                const int i = base + (int)threadIdx.x;
                const unsigned bal = __ballot_sync(0xffffffffu, i < a.num_seqs && nq[i] > r);
                const int cnt = __popc(bal);
                if (k < cnt) {
                    seq_found = base + (int)__fns(bal, 0, k + 1);
                    break;
                }
                k -= cnt;
            }
        }
        if (threadIdx.x == 0) {
            pick[0] = seq_found;
            pick[1] = seq_found >= 0 ? nq[seq_found] - 1 - r : -1;
        }
    }
    __syncthreads();
    const int seq = pick[0], qt = pick[1];
    const int h = blockIdx.x % a.hq;
    if (seq < 0) return;
    const int start = a.cu[seq];
    const int n = a.cu[seq + 1] - start;
    if (smem_u32(smem) & 1023u) return; // the swizzled tiles need 1024-byte alignment (always true)
    const int G = a.hq / a.hkv;
    const int kvh = h / G;
    const int q0 = qt * BM;
    const int qlast = min(q0 + BM, n) - 1;
    const int nkv = qlast / BN + 1;

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::BAR);
    uint64_t *q_full = bars + 0, *k_full = bars + 1, *v_full = bars + 3, *k_empty = bars + 5, *v_empty = bars + 7;
    uint64_t *s_full = bars + 9, *s_free = bars + 11, *p_full = bars + 13, *t_full = bars + 14, *fin = bars + 15;
    uint64_t *loaded = bars + 16;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 17);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(bars + 18);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(k_full + s, 1);
            mbar_init(v_full + s, 1);
            mbar_init(k_empty + s, 1);
            mbar_init(v_empty + s, 1);
            mbar_init(s_full + s, 1);
            mbar_init(s_free + s, 128);
        }
        mbar_init(p_full, 128);
        mbar_init(t_full, 1);
        mbar_init(fin, 1);
        mbar_init(loaded, 1);
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

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producers
        // K and V have rings of their own: a K stage is free once S = Q K^T of its tile is done, so
        // K loads run about two tiles ahead of the softmax; a V stage is free once P V is done.
        // Lane 0 streams Q and K, lane 1 streams V.
        if (lane < 2) {
            const bool is_k = lane == 0;
            const CUtensorMap *map = is_k ? &tk : &tv;
            uint64_t *full = is_k ? k_full : v_full, *empty = is_k ? k_empty : v_empty;
            uint8_t *ring = smem + (is_k ? L::K0 : L::V0);
            tc::prefetch_tmap(map);
            if (is_k) {
                tc::prefetch_tmap(&tq);
                mbar_arrive_expect_tx(q_full, L::Q_BYTES);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tc::tma_load_2d(smem + L::Q + c * BM * 128, &tq, h * D + c * 64, start + q0, q_full);
            }
            int issued = 0;
            for (int j = 0; j < nkv; ++j) {
                const int st = j & 1;
                if (j >= 2 && !mbar_wait(empty + st, ((j >> 1) - 1) & 1)) {
                    set_error(a.err, PKV_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                mbar_arrive_expect_tx(full + st, L::KV_BYTES);
#pragma unroll
                for (int c = 0; c < D / 64; ++c)
                    tc::tma_load_2d(ring + st * L::KV_BYTES + c * BN * 128, map, kvh * D + c * 64, start + j * BN,
                                    full + st);
                issued = j + 1;
            }
            // the loads of the last stages must land before this CTA's shared memory goes away
            for (int j = issued > 2 ? issued - 2 : 0; j < issued; ++j)
                if (!mbar_wait(full + (j & 1), (j >> 1) & 1)) set_error(a.err, PKV_DEVERR_TIMEOUT);
            if (is_k && !mbar_wait(q_full, 0)) set_error(a.err, PKV_DEVERR_TIMEOUT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IQK = tc::idesc_f16(MT == PKV_BF16 ? 1u : 0u, 0u, BM, BN);
            constexpr uint32_t IPV = tc::idesc_f16(MT == PKV_BF16 ? 1u : 0u, 1u, BM, D);
            const uint32_t sQ = smem_u32(smem + L::Q), sK = smem_u32(smem + L::K0), sV = smem_u32(smem + L::V0);
            const uint32_t sP = smem_u32(smem + L::P);
            const uint32_t tO = tmem + 128;
            // S_j = Q K_j^T into S buffer j % 2; its K stage is released as soon as S_j is done
            auto issue_s = [&](int j) {
                const int st = j & 1;
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const int c = k >> 2, kk = k & 3;
                    const uint64_t ad = tc::smem_desc(sQ + c * BM * 128 + kk * 32, 16, 1024);
                    const uint64_t bd = tc::smem_desc(sK + st * L::KV_BYTES + c * BN * 128 + kk * 32, 16, 1024);
                    tc::mma_f16(tmem + st * BN, ad, bd, IQK, k > 0 ? 1u : 0u);
                }
                tc::commit(s_full + st);
                tc::commit(k_empty + st);
            };
            bool ok = mbar_wait(q_full, 0) && mbar_wait(k_full, 0);
            if (ok) {
                tc::fence_after_sync();
                issue_s(0);
            }
            for (int j = 0; j < nkv && ok; ++j) {
                if (j + 1 < nkv) {
                    const int b = (j + 1) & 1;
                    ok = mbar_wait(k_full + b, ((j + 1) >> 1) & 1);
                    if (ok && j + 1 >= 2) ok = mbar_wait(s_free + b, ((j - 1) >> 1) & 1);
                    if (!ok) break;
                    tc::fence_after_sync();
                    issue_s(j + 1);
                }
                const int st = j & 1;
                ok = mbar_wait(p_full, j & 1) && mbar_wait(v_full + st, (j >> 1) & 1);
                if (!ok) break;
                if (j == nkv - 1) mbar_arrive(loaded); // every K and V tile of this CTA has landed
                tc::fence_after_sync();
#pragma unroll
                for (int part = 0; part < L::NP; ++part)
#pragma unroll
                    for (int k = 0; k < BN / 16; ++k) {
                        const uint64_t ad = tc::smem_desc(sP + part * L::P_BYTES + k * 32, 16, 1024);
                        const uint64_t bd = tc::smem_desc(sV + st * L::KV_BYTES + k * 2048, BN * 128, 1024);
                        tc::mma_f16(tO, ad, bd, IPV, (j > 0 || k > 0 || part > 0) ? 1u : 0u);
                    }
                tc::commit(t_full);
                tc::commit(v_empty + st);
            }
            if (!ok) {
                set_error(a.err, PKV_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            // every MMA issued by this thread has completed before TMEM is released
            tc::commit(fin);
            if (!mbar_wait(fin, 0)) set_error(a.err, PKV_DEVERR_TIMEOUT);
        }
    } else if (warp < 6) {
        // ------------------------------------------------------------ softmax, one thread per row
        const int lw = warp & 3;
        const int r = lw * 32 + lane;
        const int qpos = q0 + r;
        const uint32_t lane_off = static_cast<uint32_t>(lw * 32) << 16;
        float m_use = -INFINITY, l = 0.f;
        bool ok = true;
        uint8_t *prow = smem + L::P + (r >> 3) * 1024 + (r & 7) * 128;
        for (int j = 0; j < nkv && ok; ++j) {
            const int b = j & 1;
            ok = __all_sync(0xffffffffu, mbar_wait(s_full + b, (j >> 1) & 1));
            if (!ok) break;
            tc::fence_after_sync();
            uint32_t sr[64];
            {
                uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[0]);
                uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sr[32]);
                tc::ld32(tmem + lane_off + b * BN, lo);
                tc::ld32(tmem + lane_off + b * BN + 32, hi);
            }
            tc::wait_ld();
            tc::fence_before_sync();
            mbar_arrive(s_free + b);
            // causal mask, only on tiles that reach past this tile's first query row
            const int kbase = j * BN;
            if (kbase + BN - 1 > q0) {
                const int lim = qpos - kbase + 1; // keys c < lim are at or before this row
#pragma unroll
                for (int c = 0; c < BN; ++c)
                    if (c >= lim) sr[c] = 0xFF800000u; // -inf
            }
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int c = 0; c < BN; c += 2) {
                mx0 = fmaxf(mx0, __uint_as_float(sr[c]));
                mx1 = fmaxf(mx1, __uint_as_float(sr[c + 1]));
            }
            const float mx = fmaxf(mx0, mx1) * a.scale_log2; // scale > 0 keeps the order
            const bool up = mx > m_use + kRescale;
            const float m_new = up ? mx : m_use;
            const float alpha = up ? fast_exp2(m_use - m_new) : 1.f;
            m_use = m_new;
            const float nbase = m_use == -INFINITY ? 0.f : -m_use; // a row with no live key yet keeps p = 0
            float rs0 = 0.f, rs1 = 0.f;
            uint32_t phi[BN / 2], plo[L::NP == 2 ? BN / 2 : 1];
#pragma unroll
            for (int c = 0; c < BN / 2; ++c) {
                const float p0 = fast_exp2(fmaf(__uint_as_float(sr[2 * c]), a.scale_log2, nbase));
                const float p1 = fast_exp2(fmaf(__uint_as_float(sr[2 * c + 1]), a.scale_log2, nbase));
                rs0 += p0;
                rs1 += p1;
                phi[c] = pack2(p0, p1, MT);
                if constexpr (L::NP == 2) // remainders after bf16 rounding, themselves rounded to bf16
                    plo[c] = pack2(p0 - __uint_as_float(phi[c] << 16), p1 - __uint_as_float(phi[c] & 0xFFFF0000u), MT);
            }
            const float rs = rs0 + rs1;
            l = l * alpha + rs;
            if (j > 0) {
                // P V of the previous tile has finished: P's buffer is free and O is stable
                ok = __all_sync(0xffffffffu, mbar_wait(t_full, (j - 1) & 1));
                if (!ok) break;
                tc::fence_after_sync();
                if (__any_sync(0xffffffffu, up)) {
#pragma unroll
                    for (int cc = 0; cc < D / 16; ++cc) {
                        uint32_t o[16];
                        tc::ld16(tmem + lane_off + 128 + cc * 16, o);
                        tc::wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                        tc::st16(tmem + lane_off + 128 + cc * 16, o);
                    }
                    tc::wait_st();
                }
            }
#pragma unroll
            for (int c = 0; c < BN / 8; ++c) {
                const int off = (c ^ (r & 7)) << 4;
                *reinterpret_cast<uint4 *>(prow + off) =
                    make_uint4(phi[4 * c], phi[4 * c + 1], phi[4 * c + 2], phi[4 * c + 3]);
                if constexpr (L::NP == 2)
                    *reinterpret_cast<uint4 *>(prow + L::P_BYTES + off) =
                        make_uint4(plo[4 * c], plo[4 * c + 1], plo[4 * c + 2], plo[4 * c + 3]);
            }
            fence_proxy_async_smem();
            tc::fence_before_sync();
            mbar_arrive(p_full);
        }
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(t_full, (nkv - 1) & 1));
        if (!ok) {
            set_error(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
        } else {
            tc::fence_after_sync();
            const float inv = 1.f / l;
            using T = typename ModelT<MT>::T;
            T *orow = static_cast<T *>(a.out) + ((int64_t)(start + qpos) * a.hq + h) * D;
#pragma unroll
            for (int cc = 0; cc < D / 16; ++cc) {
                uint32_t o[16];
                tc::ld16(tmem + lane_off + 128 + cc * 16, o);
                tc::wait_ld();
                uint32_t w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    w[e] = pack2(__uint_as_float(o[2 * e]) * inv, __uint_as_float(o[2 * e + 1]) * inv, MT);
                if (qpos < n) {
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + cc * 16);
                    dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                    dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                }
            }
        }
    } else if (h % G == 0) {
        // ------------------------------------------------------------ paged K/V write of this tile's rows
        // The tile's own rows q0..qlast are the keys of K/V tiles q0/BN .. nkv-1, the last ones the
        // producer loads; no later tile recycles their stages, so they are copied straight from
        // shared memory (undoing the 128-byte swizzle) to their slots: no global reads, and each
        // row leaves as one contiguous D*2-byte store from D/8 lanes.
        constexpr int CPR = D / 8;   // 16-byte chunks per row
        constexpr int RPI = 32 / CPR; // rows per warp instruction
        const int wl = warp - 6;
        const int cc = lane % CPR, rsub = lane / CPR;
        const int c2 = cc >> 3, u = cc & 7;
        // `loaded` has a single phase (the MMA thread arrives once it has seen the last K/V tile land);
        // waiting on k_full/v_full here could target a phase two or more ahead, which a parity wait cannot tell
        // from an already completed one
        const bool landed = __all_sync(0xffffffffu, mbar_wait(loaded, 0));
        if (!landed && lane == 0) {
            set_error(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
        for (int j = q0 / BN; j < nkv && landed; ++j) {
            const int st = j & 1;
            const int lo = max(j * BN, q0), hi = min(j * BN + BN - 1, qlast);
            for (int p0 = lo + wl * RPI; p0 <= hi; p0 += 2 * RPI) {
                const int p = p0 + rsub;
                if (p > hi) continue;
                const int lb = p / a.bs;
                const int blk = lb < a.max_blocks ? a.tables[(int64_t)seq * a.max_blocks + lb] : -1;
                if (blk < 0 || blk >= a.num_blocks) {
                    if (cc == 0) set_error(a.err, PKV_DEVERR_BLOCK_ID);
                    continue;
                }
                const int r = p - j * BN;
                const int sw = c2 * BN * 128 + (r >> 3) * 1024 + (r & 7) * 128 + ((u ^ (r & 7)) << 4);
                const uint4 kx = *reinterpret_cast<const uint4 *>(smem + L::K0 + st * L::KV_BYTES + sw);
                const uint4 vx = *reinterpret_cast<const uint4 *>(smem + L::V0 + st * L::KV_BYTES + sw);
                const int64_t dst = ((int64_t)blk * 2 * a.hkv + kvh) * a.tile_elems + (int64_t)(p - lb * a.bs) * D + cc * 8;
                *reinterpret_cast<uint4 *>(a.pool + dst * 2) = kx;
                *reinterpret_cast<uint4 *>(a.pool + (dst + (int64_t)a.hkv * a.tile_elems) * 2) = vx;
            }
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
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
bool make_map(CUtensorMap *m, const void *base, int mt, int64_t rows, int64_t cols, int box_rows) {
    EncodeFn enc = encode_fn();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, mt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                           const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D, int MT>
cudaError_t launch_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const Args &a, int grid,
                     cudaStream_t st) {
    auto kern = prefill_kernel<D, MT>;
    const int smem = Layout<D, MT>::TOTAL;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return pdl_launch(kern, dim3(grid), dim3(kThreads), smem, st, tq, tk, tv, a);
}

} // namespace pkv_prefill

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
    a.nqt_max = (p.max_seqlen + BM - 1) / BM;
    a.scale_log2 = p.scale * 1.4426950408889634f;
    // the work-item prologue keeps num_seqs + nqt_max + 3 ints in the P buffer
    if ((int64_t)p.num_seqs + a.nqt_max + 3 > (int64_t)BM * BN * 2 / 4) return cudaErrorNotSupported;
    CUtensorMap tq, tk, tv;
    if (!make_map(&tq, p.q, mt, p.total_tokens, (int64_t)p.num_q_heads * D, BM) ||
        !make_map(&tk, p.k, mt, p.total_tokens, (int64_t)c->num_kv_heads * D, BN) ||
        !make_map(&tv, p.v, mt, p.total_tokens, (int64_t)c->num_kv_heads * D, BN))
        return cudaErrorInvalidValue;
    // (sequence, query tile) items: sum_i ceil(n_i / BM) <= T / BM + num_seqs
    const int64_t items = std::min<int64_t>((int64_t)a.nqt_max * p.num_seqs, p.total_tokens / BM + p.num_seqs);
    const int64_t grid = items * p.num_q_heads;
    if (grid == 0) return cudaSuccess;
    if (grid > 0x7FFFFFFF) return cudaErrorNotSupported;
    PkvTimer timer(c, PKV_KIND_PREFILL, st);
    cudaError_t e;
    if (D == 128)
        e = mt == PKV_BF16 ? launch_t<128, PKV_BF16>(tq, tk, tv, a, (int)grid, st)
                           : launch_t<128, PKV_F16>(tq, tk, tv, a, (int)grid, st);
    else
        e = mt == PKV_BF16 ? launch_t<64, PKV_BF16>(tq, tk, tv, a, (int)grid, st)
                           : launch_t<64, PKV_F16>(tq, tk, tv, a, (int)grid, st);
    g_pkv_launches++;
    return e;
}
