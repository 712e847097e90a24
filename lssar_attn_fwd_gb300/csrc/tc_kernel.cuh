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
//   pass 1 (LSSAR):    S1_i = sum_j sp2(z_ij),  m_i = max_j z_ij, the softplus sum
//                      taken as sum_j max(z,0) + log2 prod_j (1 + 2^-|z|)
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
// of one tile overlaps the elementwise work of the other.  Items are numbered
// longest first; each CTA starts with item blockIdx.x and then takes the next
// unclaimed item from a global counter (longest-processing-time-first), the
// producer warp publishing each item to the other roles through a small
// shared-memory queue.
// Causal masking: on the diagonal tile the scaled scores above the diagonal
// are replaced by -inf, for which every weight below evaluates to exactly 0.
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
                  kErrOFull, kErrOFree, kErrItem };

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
    unsigned *err;       // device error word
    unsigned *counter;   // work counter, zero at launch
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

constexpr int kItemQ = 4;                     // depth of the work-item queue
constexpr uint32_t kItemConsumers = 1 + 2 * kBM;   // MMA thread + both warpgroups

struct __align__(8) Barriers {
    uint64_t q_full, q_empty;
    uint64_t s_full[2], s_free[2], o_full[2], o_free[2];
    uint64_t kv_full[8], kv_empty[8];
    uint64_t item_full[kItemQ], item_empty[kItemQ];
    int item_q[kItemQ];
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

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// softplus(x)/ln 2 for z = x log2 e: max(z, 0) + log2(1 + 2^-|z|), two lanes.
// sp2(-inf) = 0.
__device__ __forceinline__ float2 sp2x2(float2 z) {
    const float2 u = make_float2(ptx::ex2(-fabsf(z.x)), ptx::ex2(-fabsf(z.y)));
    const float2 v = __fadd2_rn(u, make_float2(1.f, 1.f));
    return __fadd2_rn(make_float2(fmaxf(z.x, 0.f), fmaxf(z.y, 0.f)),
                      make_float2(ptx::lg2(v.x), ptx::lg2(v.y)));
}

__device__ __forceinline__ float sp2(float z) {
    return fmaxf(z, 0.f) + ptx::lg2(1.f + ptx::ex2(-fabsf(z)));
}

template <int PK>
__device__ __forceinline__ float2 powk2(float2 r, int p) {
    if constexpr (PK == 1) {
        return r;
    } else if constexpr (PK == 2) {
        return __fmul2_rn(r, r);
    } else if constexpr (PK == 3) {
        return __fmul2_rn(__fmul2_rn(r, r), r);
    } else if constexpr (PK == 15) {
        const float2 r2 = __fmul2_rn(r, r), r3 = __fmul2_rn(r2, r), r6 = __fmul2_rn(r3, r3);
        return __fmul2_rn(__fmul2_rn(r6, r6), r3);
    } else {
        float2 acc = make_float2(1.f, 1.f);
        while (p) {
            if (p & 1) acc = __fmul2_rn(acc, r);
            r = __fmul2_rn(r, r);
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

// Scores of one 32-column chunk to z = a * s in place; on the diagonal tile
// the columns above row t become -inf.
template <bool DIAG>
__device__ __forceinline__ void to_z(uint32_t (&r)[32], int col0, int t, float a) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        float2 z = __fmul2_rn(make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])),
                              make_float2(a, a));
        if (DIAG) {
            if (col0 + j > t) z.x = -INFINITY;
            if (col0 + j + 1 > t) z.y = -INFINITY;
        }
        r[j] = __float_as_uint(z.x);
        r[j + 1] = __float_as_uint(z.y);
    }
}

// Pass-1 statistics of one chunk of z: running max and, for LSSAR, the two
// parts of sum_j sp2(z_j) = sum_j max(z_j, 0) + log2(prod_j (1 + 2^-|z_j|)).
// The product form needs one FFMA per element instead of a log2: every factor
// lies in (1, 2], so up to 64 factors multiply in fp32 without overflow (the
// caller takes log2 of each 64-factor product once per tile).
template <int MODE>
__device__ __forceinline__ void stats_z(const uint32_t (&r)[32], float2 &relu_acc, float2 &prod,
                                        float &m) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float2 z = make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
        m = max3(m, z.x, z.y);
        if constexpr (MODE == kLssar) {
            const float2 u = make_float2(ptx::ex2(-fabsf(z.x)), ptx::ex2(-fabsf(z.y)));
            prod = __ffma2_rn(prod, u, prod);
            relu_acc = __fadd2_rn(relu_acc, make_float2(fmaxf(z.x, 0.f), fmaxf(z.y, 0.f)));
        }
    }
}

// Pass-2 weights of one chunk of z, summed into acc and packed to 16 bf16x2.
template <int MODE, int PK>
__device__ __forceinline__ void weights_z(const uint32_t (&r)[32], const RowConst &rc, int p,
                                          float2 &acc, uint32_t *pk) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float2 z = make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
        float2 w;
        if constexpr (MODE == kSoftmax) {
            const float2 e = __fadd2_rn(z, make_float2(-rc.m, -rc.m));
            w = make_float2(ptx::ex2(e.x), ptx::ex2(e.y));
        } else if constexpr (MODE == kLssa) {
            w = sp2x2(z);
        } else {
            const float2 t = __ffma2_rn(sp2x2(z), make_float2(rc.kappa, rc.kappa),
                                        make_float2(rc.beta, rc.beta));
            w = powk2<PK>(make_float2(fmaxf(t.x, 0.f), fmaxf(t.y, 0.f)), p);
        }
        acc = __fadd2_rn(acc, w);
        pk[j / 2] = ptx::pack_bf16x2(w.x, w.y);
    }
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
        for (int s = 0; s < kItemQ; ++s) {
            ptx::mbar_init(ptx::smem_u32(&bars->item_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->item_empty[s]), kItemConsumers);
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
    // Consumer side of the work-item queue: returns false on a timed-out wait.
    auto next_item = [&](uint32_t &qi, int &item) -> bool {
        const uint32_t s = qi % kItemQ, use = qi / kItemQ;
        ++qi;
        if (!wait_bar(ptx::smem_u32(&bars->item_full[s]), use & 1, bars, prm.err, kErrItem))
            return false;
        item = *(volatile int *)&bars->item_q[s];
        ptx::mbar_arrive(ptx::smem_u32(&bars->item_empty[s]));
        return true;
    };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::prefetch_tensormap(&tmQ);
            ptx::prefetch_tensormap(&tmK);
            ptx::prefetch_tensormap(&tmV);
            uint32_t ring_idx = 0, q_cnt = 0, qi = 0;
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
            while (ok) {
                // claim and publish the next work item
                const uint32_t s = qi % kItemQ, use = qi / kItemQ;
                const int item = qi == 0 ? (int)blockIdx.x
                                         : (int)(gridDim.x + atomicAdd(prm.counter, 1u));
                ++qi;
                if (use > 0 && !wait_bar(ptx::smem_u32(&bars->item_empty[s]), (use - 1) & 1, bars,
                                         prm.err, kErrItem))
                    break;
                *(volatile int *)&bars->item_q[s] = item;
                ptx::mbar_arrive(ptx::smem_u32(&bars->item_full[s]));
                if (item >= prm.n_items) break;

                int bh, m;
                decode(item, bh, m);
                const int qa = 2 * m, qb = 2 * m + 1;
                const bool vb = qb < prm.n_qtiles;
                const int nk = vb ? qb + 1 : qa + 1;
                if (q_cnt > 0 && !wait_bar(ptx::smem_u32(&bars->q_empty), (q_cnt - 1) & 1, bars,
                                           prm.err, kErrQEmpty))
                    break;
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
            uint32_t ring_idx = 0, q_cnt = 0, qi = 0;
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
            int item;
            while (ok && (ok = next_item(qi, item)) && item < prm.n_items) {
                int bh, m;
                decode(item, bh, m);
                const int qa = 2 * m, qb = 2 * m + 1;
                const bool vb = qb < prm.n_qtiles;
                const int n_w[2] = {qa + 1, vb ? qb + 1 : 0};
                const int nk = vb ? qb + 1 : qa + 1;
                if (!(ok = wait_bar(ptx::smem_u32(&bars->q_full), q_cnt & 1, bars, prm.err, kErrQFull)))
                    break;
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
        uint32_t sf_phase = 0, of_phase = 0, qi = 0;
        const float log2e = 1.4426950408889634f;
        auto wait_warp = [&](uint32_t bar, uint32_t parity, unsigned code) -> bool {
            const bool mine = wait_bar(bar, parity, bars, prm.err, code);
            return __all_sync(0xffffffffu, mine);
        };
        bool ok = true;
        int item;
        while (ok) {
            ok = __all_sync(0xffffffffu, next_item(qi, item));
            if (!ok || item >= prm.n_items) break;
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
                float2 acc[4];
                float mx[4];
                float s1_log = 0.f;   // sum over tiles of log2 of the 64-factor products
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    acc[c] = make_float2(0.f, 0.f);
                    mx[c] = -INFINITY;
                }
                for (int kt = 0; kt < n; ++kt) {
                    if (!(ok = wait_warp(s_full, sf_phase, kErrSFull))) break;
                    sf_phase ^= 1;
                    ptx::tc_fence_after();
                    uint32_t r[4][32];
#pragma unroll
                    for (int c = 0; c < 4; ++c) ptx::tmem_ld32(s_col + 32 * c, r[c]);
                    ptx::tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 4; ++c) ptx::reg_fence(r[c]);
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(s_free);   // S may be overwritten: values are in registers
                    if (kt == qt) {
#pragma unroll
                        for (int c = 0; c < 4; ++c) to_z<true>(r[c], 32 * c, t, rc.a);
                    } else {
#pragma unroll
                        for (int c = 0; c < 4; ++c) to_z<false>(r[c], 32 * c, t, rc.a);
                    }
                    float2 prod[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        prod[c] = make_float2(1.f, 1.f);
                        stats_z<MODE>(r[c], acc[c], prod[c], mx[c]);
                    }
                    if constexpr (MODE == kLssar) {
                        const float pa = (prod[0].x * prod[0].y) * (prod[1].x * prod[1].y);
                        const float pb = (prod[2].x * prod[2].y) * (prod[3].x * prod[3].y);
                        s1_log += ptx::lg2(pa) + ptx::lg2(pb);
                    }
                }
                if (!ok) break;
                const float mxr = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                if constexpr (MODE == kSoftmax) {
                    rc.m = mxr;
                } else {
                    const float s1 = ((acc[0].x + acc[0].y) + (acc[1].x + acc[1].y)) +
                                     ((acc[2].x + acc[2].y) + (acc[3].x + acc[3].y)) + s1_log;
                    const float o = (row + 1 <= 3) ? 0.f : 1.f;
                    const float theta = o * s1 / fi;
                    const float spm = sp2(mxr);
                    const float den = spm - theta;
                    if (den > 0.f) {
                        rc.kappa = 1.f / den;
                        rc.beta = -theta * rc.kappa;
                    } else {
                        // All-zero re-weighted row: only an exactly uniform LSSA row
                        // (all sp equal) gets here; (sp / sp_max)^p = 1 on every
                        // unmasked column gives the uniform prefix mean.
                        rc.kappa = 1.f / spm;
                        rc.beta = 0.f;
                    }
                }
            }
            // pass 2: weights into TMEM (over the S columns), running row sum
            float2 acc2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
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
                        to_z<true>(r0, h * 64, t, rc.a);
                        to_z<true>(r1, h * 64 + 32, t, rc.a);
                    } else {
                        to_z<false>(r0, h * 64, t, rc.a);
                        to_z<false>(r1, h * 64 + 32, t, rc.a);
                    }
                    weights_z<MODE, PK>(r0, rc, prm.p, acc2[0], pk);
                    weights_z<MODE, PK>(r1, rc, prm.p, acc2[1], pk + 16);
                    ptx::tmem_st32(s_col + h * 32, pk);
                }
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(s_free);   // P(kt) is in TMEM
            }
            if (!ok) break;
            const float s2 = (acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y);
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
                    const uint32_t *oc = &o[c / 4][(c % 4) * 8];
                    uint4 u;
                    u.x = ptx::pack_bf16x2(__uint_as_float(oc[0]) * inv, __uint_as_float(oc[1]) * inv);
                    u.y = ptx::pack_bf16x2(__uint_as_float(oc[2]) * inv, __uint_as_float(oc[3]) * inv);
                    u.z = ptx::pack_bf16x2(__uint_as_float(oc[4]) * inv, __uint_as_float(oc[5]) * inv);
                    u.w = ptx::pack_bf16x2(__uint_as_float(oc[6]) * inv, __uint_as_float(oc[7]) * inv);
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
