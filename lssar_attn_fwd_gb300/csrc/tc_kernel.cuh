// Tensor-core causal LSSAR / LSSA / softmax attention forward for sm_103a.
//
// What is computed (notes on "Softplus Attention with Re-weighting Boosts
// Length Extrapolation in Large Language Models", Key designs 1-3, and the
// scaled dot-product formula in its Background section), for row i (1-based)
// and keys j <= i of one head:
//   LSSA/LSSAR scores  z_ij = log2(e) * ln d * ln i * qh_i . kh_j, with qh, kh
//                      the L2-normalised rows (prepared in fp16 by a prologue)
//   softmax scores     z_ij = log2(e) / sqrt(d) * q_i . k_j (raw bf16 rows)
//   sp2(z) = max(z, 0) + log2(1 + 2^-|z|)  = softplus(x) / ln 2  for z = x log2 e
//   pass 1 (LSSAR):    S1_i = sum_j sp2(z_ij),  m_i = max_j z_ij
//   pass 1 (softmax):  m_i = max_j z_ij
//   pass 2 weights:    LSSA     w = sp2(z)
//                      LSSAR    w = max(sp2(z) kappa_i + beta_i, 0)^p with
//                               theta_i = O_i S1_i / i, kappa_i = 1/(sp2(m_i) - theta_i),
//                               beta_i = -theta_i kappa_i, i.e. the re-weighted row
//                               ReLU^p(i A - O) divided by its (positive) row maximum,
//                               which the final L1 normalisation cancels; an all-zero
//                               row (sp2(m_i) <= theta_i) gets w = 1 (prefix mean)
//                      softmax  w = 2^(z - m_i)
//   out_i = (sum_j w_ij v_j) / (sum_j w_ij)
//
// Structure (one persistent CTA per SM, 384 threads):
//   warp 0      TMA producer: Q tiles once per work item, then K (pass 1) and
//               K, V (pass 2) tiles through an NS-stage shared-memory ring.
//   warp 1      TMEM owner and single-thread tcgen05.mma issuer.
//   warps 4-7   score warpgroup 0, warps 8-11 score warpgroup 1: thread t owns
//               query row t of its Q tile (TMEM lane t), reads S from TMEM,
//               computes statistics / weights, writes P (bf16) back into TMEM
//               over its own S columns, and runs the epilogue.
// A work item is a pair of consecutive 128-row Q tiles of one head (2m, 2m+1)
// sharing every K/V tile load; the two warpgroups ping-pong so that the MMA
// of one tile overlaps the elementwise work of the other.
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+D), O1 [256+D,256+2D).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lssar_internal.cuh"
#include "tc_ptx.cuh"

namespace lssar {
namespace tc {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kThreads = 384;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a stuck wait gives up after 2 s

// Error codes written to the device error word (first failure wins).
enum : unsigned { kErrQFull = 1, kErrQEmpty, kErrKvFull, kErrKvEmpty, kErrSFull, kErrSFree,
                  kErrOFull, kErrOFree };

// Shared-memory descriptor strides.  K-major tiles (Q, K): rows of 128 bytes,
// 8-row groups 1024 bytes apart.  MN-major V tiles: 16 keys per MMA = 2048
// bytes, 8-key groups 1024 bytes apart, 64-column blocks 16384 bytes apart.
constexpr uint32_t kKmajorLbo = 16;
constexpr uint32_t kKmajorSbo = 1024;
constexpr uint32_t kVLbo = 16384;
constexpr uint32_t kVSbo = 1024;

struct Params {
    int BH;          // B * H
    int L;
    int n_qtiles;    // ceil(L / 128)
    int n_pairs;     // ceil(n_qtiles / 2)
    int n_items;     // BH * n_pairs
    float ln_d;      // ln(d)
    int p;           // LSSAR exponent (used by the generic power path)
    __nv_bfloat16 *out;
    unsigned *err;   // device error word
};

template <int D>
struct Cfg {
    static constexpr int kTileBytes = kBM * D * 2;       // one Q, K or V tile
    static constexpr int kStages = D == 64 ? 8 : 4;      // ring stages
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = 2 * kTileBytes;
    static constexpr int kBarOff = kRingOff + kStages * kTileBytes;
    static constexpr int kBarBytes = 1024;
    static constexpr int kSmemBytes = kBarOff + kBarBytes + 1024;  // + alignment slack
};

struct __align__(8) Barriers {
    uint64_t q_full, q_empty;
    uint64_t s_full[2], s_free[2], o_full[2], o_free[2];
    uint64_t kv_full[8], kv_empty[8];
    uint32_t tmem_base;
    int abort_flag;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Barriers *b, unsigned *err,
                                         unsigned code) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((spin & 63u) == 0) {
            if (*(volatile int *)&b->abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
                atomicCAS(err, 0u, code);
                *(volatile int *)&b->abort_flag = 1;
                return false;
            }
        }
    }
}

// softplus(x)/ln 2 for z = x log2 e: max(z, 0) + log2(1 + 2^-|z|).
__device__ __forceinline__ float sp2(float z) {
    return fmaxf(z, 0.f) + ptx::lg2(1.f + ptx::ex2(-fabsf(z)));
}

template <int PK>
__device__ __forceinline__ float powk(float r, int p) {
    if constexpr (PK == 1) {
        return r;
    } else if constexpr (PK == 2) {
        return r * r;
    } else if constexpr (PK == 3) {
        return r * r * r;
    } else if constexpr (PK == 15) {
        const float r2 = r * r, r3 = r2 * r, r6 = r3 * r3, r12 = r6 * r6;
        return r12 * r3;
    } else {
        float acc = 1.f;
        while (p) {
            if (p & 1) acc *= r;
            r *= r;
            p >>= 1;
        }
        return acc;
    }
}

struct RowConst {
    float a;       // score scale: z = a * s
    float kappa;   // LSSAR slope
    float beta;    // LSSAR offset
    float m;       // softmax: row maximum of z
};

template <int MODE, int PK>
__device__ __forceinline__ float weight(float z, const RowConst &rc, int p) {
    if constexpr (MODE == kSoftmax) {
        return ptx::ex2(z - rc.m);
    } else if constexpr (MODE == kLssa) {
        return sp2(z);
    } else {
        return powk<PK>(fmaxf(fmaf(sp2(z), rc.kappa, rc.beta), 0.f), p);
    }
}

// One 32-column chunk of pass-1 statistics.
template <int MODE, bool MASK>
__device__ __forceinline__ void stats_chunk(const uint32_t (&r)[32], int col0, int trow, float a,
                                            float &s1, float &m) {
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float z = __uint_as_float(r[j]) * a;
        const bool keep = !MASK || (col0 + j <= trow);
        if (keep) {
            m = fmaxf(m, z);
            if constexpr (MODE == kLssar) {
                if (j & 1) acc1 += sp2(z); else acc0 += sp2(z);
            }
        }
    }
    s1 += acc0 + acc1;
}

// One 32-column chunk of pass-2 weights, packed to 16 bf16x2 words.
template <int MODE, int PK, bool MASK>
__device__ __forceinline__ void weight_chunk(const uint32_t (&r)[32], int col0, int trow,
                                             const RowConst &rc, int p, float &s2, uint32_t *pk) {
    float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        float w0 = weight<MODE, PK>(__uint_as_float(r[j]) * rc.a, rc, p);
        float w1 = weight<MODE, PK>(__uint_as_float(r[j + 1]) * rc.a, rc, p);
        if (MASK) {
            if (col0 + j > trow) w0 = 0.f;
            if (col0 + j + 1 > trow) w1 = 0.f;
        }
        acc0 += w0;
        acc1 += w1;
        pk[j / 2] = ptx::pack_bf16x2(w0, w1);
    }
    s2 += acc0 + acc1;
}

template <int D, int MODE, int PK>
__global__ void __launch_bounds__(kThreads, 1)
lssar_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, const Params prm) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *sQ = smem + C::kQOff;
    uint8_t *ring = smem + C::kRingOff;
    Barriers *bars = reinterpret_cast<Barriers *>(smem + C::kBarOff);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    constexpr int NS = C::kStages;
    constexpr int TB = C::kTileBytes;
    constexpr bool kTwoPass = MODE != kLssa;
    // S = Q K^T: fp16 (normalised) operands for LSSA/LSSAR, raw bf16 for softmax.
    constexpr uint32_t kIdescS = ptx::idesc_f16(MODE == kSoftmax, kBM, kBN, false, false);
    // O += P V: P bf16 from TMEM (K-major), V bf16 MN-major.
    constexpr uint32_t kIdescPV = ptx::idesc_f16(true, kBM, D, false, true);

    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bars->q_full), 1);
        ptx::mbar_init(ptx::smem_u32(&bars->q_empty), 1);
        for (int w = 0; w < 2; ++w) {
            ptx::mbar_init(ptx::smem_u32(&bars->s_full[w]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->s_free[w]), kBM);
            ptx::mbar_init(ptx::smem_u32(&bars->o_full[w]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->o_free[w]), kBM);
        }
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(ptx::smem_u32(&bars->kv_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->kv_empty[s]), 1);
        }
        bars->abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&bars->tmem_base), 512);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = bars->tmem_base;

    const int BH = prm.BH;
    auto decode = [&](int item, int &bh, int &m) {
        m = prm.n_pairs - 1 - item / BH;   // longest pairs first
        bh = item % BH;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::prefetch_tensormap(&tmQ);
            ptx::prefetch_tensormap(&tmK);
            ptx::prefetch_tensormap(&tmV);
            uint32_t ring_idx = 0, q_cnt = 0;
            bool ok = true;
            auto push = [&](const CUtensorMap *map, int tile, int bh) -> bool {
                const uint32_t s = ring_idx % NS, use = ring_idx / NS;
                if (use > 0 && !wait_bar(ptx::smem_u32(&bars->kv_empty[s]), (use - 1) & 1, bars,
                                         prm.err, kErrKvEmpty))
                    return false;
                const uint32_t full = ptx::smem_u32(&bars->kv_full[s]);
                ptx::mbar_arrive_expect_tx(full, TB);
#pragma unroll
                for (int b = 0; b < D / 64; ++b)
                    ptx::tma_load_3d(ptx::smem_u32(ring + s * TB + b * 16384), map, full, b * 64,
                                     tile * kBN, bh);
                ++ring_idx;
                return true;
            };
            for (int item = blockIdx.x; ok && item < prm.n_items; item += gridDim.x) {
                int bh, m;
                decode(item, bh, m);
                const int qa = 2 * m, qb = 2 * m + 1;
                const bool vb = qb < prm.n_qtiles;
                const int nk = vb ? qb + 1 : qa + 1;
                if (q_cnt > 0 && !wait_bar(ptx::smem_u32(&bars->q_empty), (q_cnt - 1) & 1, bars,
                                           prm.err, kErrQEmpty)) {
                    ok = false;
                    break;
                }
                const uint32_t qf = ptx::smem_u32(&bars->q_full);
                ptx::mbar_arrive_expect_tx(qf, (vb ? 2 : 1) * TB);
#pragma unroll
                for (int b = 0; b < D / 64; ++b) {
                    ptx::tma_load_3d(ptx::smem_u32(sQ + b * 16384), &tmQ, qf, b * 64, qa * kBM, bh);
                    if (vb)
                        ptx::tma_load_3d(ptx::smem_u32(sQ + TB + b * 16384), &tmQ, qf, b * 64,
                                         qb * kBM, bh);
                }
                ++q_cnt;
                if (kTwoPass)
                    for (int kt = 0; ok && kt < nk; ++kt) ok = push(&tmK, kt, bh);
                if (ok) ok = push(&tmK, 0, bh);
                for (int kt = 0; ok && kt < nk; ++kt) {
                    if (kt + 1 < nk) ok = push(&tmK, kt + 1, bh);
                    if (ok) ok = push(&tmV, kt, bh);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            uint32_t ring_idx = 0, q_cnt = 0;
            uint32_t sf_phase[2] = {0, 0}, of_phase[2] = {0, 0};
            bool s_pending[2] = {false, false}, o_pending[2] = {false, false};
            bool ok = true;
            auto acquire = [&](uint32_t &slot) -> bool {
                slot = ring_idx % NS;
                const uint32_t use = ring_idx / NS;
                ++ring_idx;
                if (!wait_bar(ptx::smem_u32(&bars->kv_full[slot]), use & 1, bars, prm.err,
                              kErrKvFull))
                    return false;
                ptx::tc_fence_after();
                return true;
            };
            auto touch_s = [&](int w) -> bool {
                if (!s_pending[w]) return true;
                if (!wait_bar(ptx::smem_u32(&bars->s_free[w]), sf_phase[w], bars, prm.err, kErrSFree))
                    return false;
                sf_phase[w] ^= 1;
                s_pending[w] = false;
                ptx::tc_fence_after();
                return true;
            };
            auto issue_s = [&](int w, uint32_t kslot) {
                const uint32_t qb = ptx::smem_u32(sQ + w * TB), kb = ptx::smem_u32(ring + kslot * TB);
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = (k / 4) * 16384 + (k % 4) * 32;
                    ptx::mma_ss(tmem + w * kBN, ptx::smem_desc_sw128(qb + off, kKmajorLbo, kKmajorSbo),
                                ptx::smem_desc_sw128(kb + off, kKmajorLbo, kKmajorSbo), kIdescS, k > 0);
                }
                ptx::mma_commit(ptx::smem_u32(&bars->s_full[w]));
                s_pending[w] = true;
            };
            auto issue_pv = [&](int w, uint32_t vslot, bool accumulate) {
                const uint32_t vb = ptx::smem_u32(ring + vslot * TB);
#pragma unroll
                for (int k = 0; k < kBN / 16; ++k)
                    ptx::mma_ts(tmem + 2 * kBN + w * D, tmem + w * kBN + k * 8,
                                ptx::smem_desc_sw128(vb + k * 2048, kVLbo, kVSbo), kIdescPV,
                                (accumulate || k > 0) ? 1u : 0u);
            };
            for (int item = blockIdx.x; ok && item < prm.n_items; item += gridDim.x) {
                int bh, m;
                decode(item, bh, m);
                const int qa = 2 * m, qb = 2 * m + 1;
                const bool vb = qb < prm.n_qtiles;
                const int n_w[2] = {qa + 1, vb ? qb + 1 : 0};
                const int nk = vb ? qb + 1 : qa + 1;
                if (!wait_bar(ptx::smem_u32(&bars->q_full), q_cnt & 1, bars, prm.err, kErrQFull)) {
                    ok = false;
                    break;
                }
                ++q_cnt;
                ptx::tc_fence_after();
                uint32_t slot;
                if (kTwoPass) {
                    for (int kt = 0; ok && kt < nk; ++kt) {
                        if (!(ok = acquire(slot))) break;
                        for (int w = 0; w < 2 && ok; ++w)
                            if (kt < n_w[w]) {
                                if (!(ok = touch_s(w))) break;
                                issue_s(w, slot);
                            }
                        ptx::mma_commit(ptx::smem_u32(&bars->kv_empty[slot]));
                    }
                }
                if (!ok || !(ok = acquire(slot))) break;
                for (int w = 0; w < 2 && ok; ++w)
                    if (n_w[w] > 0) {
                        if (!(ok = touch_s(w))) break;
                        issue_s(w, slot);
                    }
                ptx::mma_commit(ptx::smem_u32(&bars->kv_empty[slot]));
                for (int kt = 0; ok && kt < nk; ++kt) {
                    const bool has_next = kt + 1 < nk;
                    uint32_t kslot = 0, vslot;
                    if (has_next && !(ok = acquire(kslot))) break;
                    if (!(ok = acquire(vslot))) break;
                    for (int w = 0; w < 2 && ok; ++w) {
                        if (kt >= n_w[w]) continue;
                        if (!(ok = touch_s(w))) break;   // P_w(kt) is in TMEM
                        if (kt == 0 && o_pending[w]) {
                            if (!(ok = wait_bar(ptx::smem_u32(&bars->o_free[w]), of_phase[w], bars,
                                                prm.err, kErrOFree)))
                                break;
                            of_phase[w] ^= 1;
                            o_pending[w] = false;
                            ptx::tc_fence_after();
                        }
                        issue_pv(w, vslot, kt > 0);
                        if (kt + 1 < n_w[w]) {
                            issue_s(w, kslot);
                        } else {
                            ptx::mma_commit(ptx::smem_u32(&bars->o_full[w]));
                            o_pending[w] = true;
                        }
                    }
                    ptx::mma_commit(ptx::smem_u32(&bars->kv_empty[vslot]));
                    if (has_next) ptx::mma_commit(ptx::smem_u32(&bars->kv_empty[kslot]));
                }
                ptx::mma_commit(ptx::smem_u32(&bars->q_empty));
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ score warpgroups
        const int w = (warp - 4) >> 2;              // warpgroup 0 or 1
        const int t = threadIdx.x - 128 - 128 * w;  // row within the Q tile = TMEM lane
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_col = tmem + lane_addr + w * kBN;
        const uint32_t o_col = tmem + lane_addr + 2 * kBN + w * D;
        const uint32_t s_full = ptx::smem_u32(&bars->s_full[w]);
        const uint32_t s_free = ptx::smem_u32(&bars->s_free[w]);
        const uint32_t o_full = ptx::smem_u32(&bars->o_full[w]);
        const uint32_t o_free = ptx::smem_u32(&bars->o_free[w]);
        uint32_t sf_phase = 0, of_phase = 0;
        const float log2e = 1.4426950408889634f;
        auto wait_warp = [&](uint32_t bar, uint32_t parity, unsigned code) -> bool {
            const bool mine = wait_bar(bar, parity, bars, prm.err, code);
            return __all_sync(0xffffffffu, mine);
        };
        bool ok = true;
        for (int item = blockIdx.x; ok && item < prm.n_items; item += gridDim.x) {
            int bh, m;
            decode(item, bh, m);
            const int qt = 2 * m + w;
            if (qt >= prm.n_qtiles) continue;
            const int n = qt + 1;
            const int row = qt * kBM + t;
            const float fi = (float)(row + 1);
            RowConst rc;
            if constexpr (MODE == kSoftmax)
                rc.a = log2e * rsqrtf((float)D);
            else
                rc.a = log2e * prm.ln_d * logf(fi);
            rc.kappa = 0.f;
            rc.beta = 0.f;
            rc.m = 0.f;
            if constexpr (kTwoPass) {
                float s1 = 0.f, mx = -INFINITY;
                for (int kt = 0; kt < n; ++kt) {
                    if (!(ok = wait_warp(s_full, sf_phase, kErrSFull))) break;
                    sf_phase ^= 1;
                    ptx::tc_fence_after();
                    uint32_t r0[32], r1[32], r2[32], r3[32];
                    ptx::tmem_ld32(s_col + 0, r0);
                    ptx::tmem_ld32(s_col + 32, r1);
                    ptx::tmem_ld32(s_col + 64, r2);
                    ptx::tmem_ld32(s_col + 96, r3);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence(r0);
                    ptx::reg_fence(r1);
                    ptx::reg_fence(r2);
                    ptx::reg_fence(r3);
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(s_free);   // S may be overwritten: values are in registers
                    if (kt == qt) {
                        stats_chunk<MODE, true>(r0, 0, t, rc.a, s1, mx);
                        stats_chunk<MODE, true>(r1, 32, t, rc.a, s1, mx);
                        stats_chunk<MODE, true>(r2, 64, t, rc.a, s1, mx);
                        stats_chunk<MODE, true>(r3, 96, t, rc.a, s1, mx);
                    } else {
                        stats_chunk<MODE, false>(r0, 0, t, rc.a, s1, mx);
                        stats_chunk<MODE, false>(r1, 32, t, rc.a, s1, mx);
                        stats_chunk<MODE, false>(r2, 64, t, rc.a, s1, mx);
                        stats_chunk<MODE, false>(r3, 96, t, rc.a, s1, mx);
                    }
                }
                if (!ok) break;
                if constexpr (MODE == kSoftmax) {
                    rc.m = mx;
                } else {
                    const float o = (row + 1 <= 3) ? 0.f : 1.f;
                    const float theta = o * s1 / fi;
                    const float den = sp2(mx) - theta;
                    if (den > 0.f) {
                        rc.kappa = 1.f / den;
                        rc.beta = -theta * rc.kappa;
                    } else {
                        rc.kappa = 0.f;   // all-zero re-weighted row: uniform weights
                        rc.beta = 1.f;
                    }
                }
            }
            // pass 2: weights into TMEM (over the S columns), running row sum
            float s2 = 0.f;
            for (int kt = 0; kt < n; ++kt) {
                if (!(ok = wait_warp(s_full, sf_phase, kErrSFull))) break;
                sf_phase ^= 1;
                ptx::tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t r0[32], r1[32], pk[32];
                    ptx::tmem_ld32(s_col + h * 64, r0);
                    ptx::tmem_ld32(s_col + h * 64 + 32, r1);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence(r0);
                    ptx::reg_fence(r1);
                    if (kt == qt) {
                        weight_chunk<MODE, PK, true>(r0, h * 64, t, rc, prm.p, s2, pk);
                        weight_chunk<MODE, PK, true>(r1, h * 64 + 32, t, rc, prm.p, s2, pk + 16);
                    } else {
                        weight_chunk<MODE, PK, false>(r0, h * 64, t, rc, prm.p, s2, pk);
                        weight_chunk<MODE, PK, false>(r1, h * 64 + 32, t, rc, prm.p, s2, pk + 16);
                    }
                    ptx::tmem_st32(s_col + h * 32, pk);
                }
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(s_free);   // P(kt) is in TMEM
            }
            if (!ok) break;
            // epilogue
            if (!(ok = wait_warp(o_full, of_phase, kErrOFull))) break;
            of_phase ^= 1;
            ptx::tc_fence_after();
            uint32_t o[D / 32][32];
#pragma unroll
            for (int c = 0; c < D / 32; ++c) ptx::tmem_ld32(o_col + c * 32, o[c]);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) ptx::reg_fence(o[c]);
            ptx::tc_fence_before();
            ptx::mbar_arrive(o_free);
            if (row < prm.L) {
                const float inv = 1.f / s2;
                uint4 *dst = reinterpret_cast<uint4 *>(prm.out + ((size_t)bh * prm.L + row) * D);
#pragma unroll
                for (int c = 0; c < D / 8; ++c) {
                    uint4 u;
                    u.x = ptx::pack_bf16x2(__uint_as_float(o[c / 4][(c % 4) * 8 + 0]) * inv,
                                           __uint_as_float(o[c / 4][(c % 4) * 8 + 1]) * inv);
                    u.y = ptx::pack_bf16x2(__uint_as_float(o[c / 4][(c % 4) * 8 + 2]) * inv,
                                           __uint_as_float(o[c / 4][(c % 4) * 8 + 3]) * inv);
                    u.z = ptx::pack_bf16x2(__uint_as_float(o[c / 4][(c % 4) * 8 + 4]) * inv,
                                           __uint_as_float(o[c / 4][(c % 4) * 8 + 5]) * inv);
                    u.w = ptx::pack_bf16x2(__uint_as_float(o[c / 4][(c % 4) * 8 + 6]) * inv,
                                           __uint_as_float(o[c / 4][(c % 4) * 8 + 7]) * inv);
                    dst[c] = u;
                }
            }
        }
    }

    // ------------------------------------------------------------ teardown
    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

}  // namespace tc
}  // namespace lssar
