// Tensor-core causal LSSAR / LSSA / softmax attention forward for sm_103a.
//
// What is computed (notes on "Softplus Attention with Re-weighting Boosts
// Length Extrapolation in Large Language Models", Key designs 1-3, and the
// scaled dot-product formula in its Background section), for row i (1-based)
// and keys j <= i of one head:
//   LSSA/LSSAR scores  z_ij = log2(e) * ln d * ln i * qh_i . kh_j, with qh, kh
//                      the L2-normalised rows prepared in fp16 by a prologue
//                      that also multiplies query row i by log2(e) ln d ln i
//                      (by its negative for the sigmoid normaliser), so that
//                      the score product yields z itself
//   softmax scores     z_ij = log2(e) / sqrt(d) * q_i . k_j (raw bf16 rows)
//   sp2(z) = log2(1 + 2^z) = softplus(x) / ln 2  for z = x log2 e
//   pass 1 (LSSAR):    S1_i = sum_j sp2(z_ij),  m_i = max_j z_ij, the softplus sum
//                      taken as sum_j max(z,0) + log2 prod_j (1 + 2^-|z|)
//   softmax (one pass): a reference maximum per row, raised (and O and the
//                      row sum rescaled by 2^(old - new)) when a K tile's scores
//                      exceed it by more than 8; P = 2^(z - ref)
//   pass 2 weights:    LSSA     w = sp2(z)
//                      LSSAR    w = max(sp2(z) kappa_i + beta_i, 0)^p with
//                               theta_i = O_i S1_i / i, kappa_i = 1/(sp2(m_i) - theta_i),
//                               beta_i = -theta_i kappa_i, i.e. the re-weighted row
//                               ReLU^p(i A - O) divided by its (positive) row maximum,
//                               which the final L1 normalisation cancels; an all-zero
//                               row (sp2(m_i) <= theta_i) gets w = 1 (prefix mean)
//                      softmax  w = 2^(z - ref_i)
//   ablation modes (the notes' ablation table), both followed by re-weighting:
//     softmax normaliser  z as in softmax; pass 1: m_i and S1_i = sum_j 2^(z-m_i)
//                         (running max, sum rescaled per tile); a_ij = 2^(z-m)/S1,
//                         w = max(2^(z-m) kappa_i + beta_i, 0)^p, theta_i = O_i S1_i / i,
//                         kappa_i = 1/(1 - theta_i)
//     sigmoid normaliser  z as in LSSA, sigma = 1/(1 + 2^-z); pass 1: m_i and
//                         S1_i = sum_j sigma(z_ij); w = max(sigma kappa_i + beta_i, 0)^p,
//                         kappa_i = 1/(sigma(m_i) - theta_i).  The registers hold -z
//                         for this mode (scale -a, mask +inf) so 2^-z needs no negation.
//   out_i = (sum_j w_ij v_j) / (sum_j w_ij)
//
// Structure (one persistent CTA per SM; 640 threads = 20 warps at d = 64, 576
// = 18 warps at d = 128):
//   warp 0      TMA producer: Q tiles once per work item, then K (pass 1) and
//               K, V (pass 2) tiles through an NS-stage shared-memory ring.
//   warp 1      TMEM owner and tcgen05.mma issuer: for Q tile 0 of the pair at
//               d = 64, for both tiles at d = 128.
//   warp 2      (d = 64) tcgen05.mma issuer for Q tile 1.  Each issuer runs its
//               tile's chain of waits, MMAs and commits on its own, so the two
//               chains overlap; both walk the whole K/V ring and each releases
//               every stage.  Warp 3 (d = 64) has no role: warps 0-3 form the
//               control warpgroup, which hands registers to the score warps.
//   score warps four warpgroups g = 0..3 (warps 4-19 at d = 64, 2-17 at
//               d = 128): Q tile w = g & 1 of the pair,
//               column half h = g >> 1 of its 128-key S tile.  Thread t of a
//               warpgroup owns query row t (TMEM lane t, lane quarter = warp % 4)
//               and keys [64h, 64h+64) of every tile: it reads S from TMEM,
//               computes statistics / weights, writes its 32 words of P (bf16
//               pairs) to TMEM, and stores its half of the output row.  Each SM
//               sub-partition therefore runs four math warps.  The two halves of
//               a row combine their partial sums and maxima once per item
//               through shared memory (a per-tile mbarrier, bounded wait).
// The control warps run their loops warp-wide (one elected lane issues each
// copy, MMA and commit).  Eighteen or twenty warps put five on some SM
// sub-partitions, which caps the launch at 96 registers per thread; at d = 64
// the control warpgroup then drops to 64 and the score warpgroups rise to 104
// (setmaxnreg; the host launches only at exactly 96).
// d = 64: P has TMEM columns of its own, so a warpgroup releases S as soon as
// it has loaded it and the next S MMA overlaps the weight computation; P is
// double-checked free by a commit after each P.V MMA.  d = 128: TMEM is full
// with S and O, so P is written over the first half of each S column half and
// S is released only once P is in place.
// A work item is a pair of consecutive 128-row Q tiles of one head (2m, 2m+1)
// sharing every K/V tile load; the two warpgroups ping-pong so that the MMA
// of one tile overlaps the elementwise work of the other.  Items are numbered
// longest first.  Each CTA first works through up to two items fixed by the
// host (a long item and its complement, so that the CTAs' loads come out
// nearly equal), then takes the next unclaimed item of the remaining tail
// from a global counter (longest-processing-time-first); without a plan the
// fixed item is item blockIdx.x.  The producer warp publishes each item to
// the other roles through a small shared-memory queue.
// Causal masking: on the diagonal tile the scaled scores above the diagonal
// are replaced by -inf, for which every weight below evaluates to exactly 0.
// TMEM (512 columns): S0 [0,128), S1 [128,256); d = 64: P0 [256,320), P1 [320,384),
// O0 [384,448), O1 [448,512); d = 128: O0 [256,384), O1 [384,512), and P_w over
// S columns [128w, 128w+32) and [128w+64, 128w+96).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "fast_weights.cuh"
#include "lssar_internal.cuh"
#include "softplus_poly.cuh"
#include "tc_ptx.cuh"

namespace lssar {
namespace tc {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kMmaWarp1 = 2;      // second MMA issuer (d = 64)
// Registers per thread.  Every instance is launched with kLaunchRegs; at
// d = 64 the control warpgroup (warps 0-3) then gives registers back and the
// four score warpgroups take them: 128 x 64 + 512 x 104 = 640 x 96.  (At
// d = 128 the one MMA warp, which orders both tiles' MMAs, needs more than 64
// registers: that layout keeps 96 everywhere.)
constexpr int kLaunchRegs = 96;
constexpr int kCtrlRegs = 64;
constexpr int kScoreRegs = 104;
static_assert(128 * kCtrlRegs + 512 * kScoreRegs <= 640 * kLaunchRegs, "register split");
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // a stuck wait gives up after 2 s

// Error codes written to the device error word (first failure wins).
enum : unsigned { kErrQFull = 1, kErrQEmpty, kErrKvFull, kErrKvEmpty, kErrSFull, kErrSFree,
                  kErrOFull, kErrOFree, kErrItem, kErrPFull, kErrPFree, kErrDrain, kErrHalves,
                  kErrTileMax };

// Softmax (one pass): a row's reference maximum is raised only when a tile's
// scores exceed it by more than this (log2 units), so P = 2^(z - ref) stays
// below 2^8 and the rescale of O and of the row sum is rare.
constexpr float kRescaleLog2 = 8.f;

// Shared-memory descriptor strides.  K-major tiles (Q, K): rows of 128 bytes,
// 8-row groups 1024 bytes apart.  MN-major V tiles: 16 keys per MMA = 2048
// bytes, 8-key groups 1024 bytes apart, 64-column blocks 16384 bytes apart.
constexpr uint32_t kKmajorLbo = 16;
constexpr uint32_t kKmajorSbo = 1024;
constexpr uint32_t kVLbo = 16384;
constexpr uint32_t kVSbo = 1024;

constexpr int kMaxHeadsP = 256;   // per-head exponents carried in the kernel parameters
constexpr int kMaxCtas = 256;     // CTAs with a fixed first work list (one per SM)

struct Params {
    int BH;          // B * H
    int L;
    int n_qtiles;    // ceil(L / 128)
    int n_pairs;     // ceil(n_qtiles / 2)
    int n_items;     // BH * n_pairs
    float ln_d;      // ln(d)
    int p;           // re-weighting exponent (used by the generic power path)
    int H;           // heads per batch entry (for the per-head exponents)
    int per_head;    // 1: head h uses p_head[h] (generic power path only)
    int exact_weights;   // 1: LSSAR rows never take the one-exponential weights
    int p_head[kMaxHeadsP];
    // Work schedule: CTA c first processes first_items[c][0], then
    // first_items[c][1] (-1: none), then items tail_base, tail_base + 1, ...
    // as a global counter hands them out (items are numbered longest first).
    int tail_base;
    int first_items[kMaxCtas][2];
    __nv_bfloat16 *out;
    float4 *stats;       // per-row {m, kappa, beta, W} for the backward pass, or null
    unsigned *err;       // device error word
    unsigned *counter;   // work counter, zero at launch
};

template <int D>
struct Cfg {
    static constexpr int kTileBytes = kBM * D * 2;       // one Q, K or V tile
    static constexpr int kStages = D == 64 ? 8 : 4;      // ring stages
    // Q-tile pair buffers: two at d = 64, so that the next item's Q tiles load
    // while the current item runs (at d = 128 shared memory holds one)
    static constexpr int kQBufs = D == 64 ? 2 : 1;
    static constexpr int kQOff = 0;
    static constexpr int kRingOff = kQBufs * 2 * kTileBytes;
    static constexpr int kBarOff = kRingOff + kStages * kTileBytes;
    static constexpr int kBarBytes = 8192;
    static constexpr int kSmemBytes = kBarOff + kBarBytes + 1024;  // + alignment slack
    // MMA-issuing warps: one per Q tile at d = 64 (P in columns of its own);
    // at d = 128, where P is written over S, one warp orders both tiles' MMAs.
    static constexpr int kMmaWarps = D == 64 ? 2 : 1;
    // d = 64: a control warpgroup (warps 0-3: producer, two MMA issuers, one
    // idle) and score warps 4-19 with the register split; d = 128: producer
    // and MMA warp 0-1, score warps 2-17, no split
    static constexpr bool kSplit = D == 64;
    static constexpr int kScoreWarp0 = kSplit ? 4 : 2;
    static constexpr int kThreads = 32 * kScoreWarp0 + 512;
};

constexpr int kItemQ = 4;                     // depth of the work-item queue
// work-item queue consumers: the MMA warps (one arrival each) and four warpgroups
__host__ __device__ constexpr uint32_t item_consumers(int mma_warps) { return mma_warps + 4 * kBM; }
constexpr uint32_t kTileThreads = 2 * kBM;           // the two warpgroups of one Q tile

struct __align__(8) Barriers {
    uint64_t q_full[2], q_empty[2];
    uint64_t s_full[2], s_free[2], o_full[2], o_free[2], p_full[2], p_free[2];
    uint64_t halves[2];   // per Q tile: both column halves have written their row partials
    uint64_t tile_max[2][4];   // softmax, per Q tile and lane quarter: both halves' tile maxima are in
    uint64_t kv_full[8], kv_empty[8];
    uint64_t item_full[kItemQ], item_empty[kItemQ];
    int item_q[kItemQ];
    uint32_t tmem_base;
    int abort_flag;
    // per-row partials exchanged by the two column halves: [tile][half][row]
    float x_s1[2][2][kBM];
    float x_m[2][2][kBM];
    float x_s2[2][2][kBM];
};

static_assert(sizeof(Barriers) <= 8192, "barrier block too large");

constexpr uint32_t kSuspendNs = 1000000;   // hardware suspend per try_wait (upper bound)

// Bounded wait on an mbarrier phase; with honour_abort it also gives up as
// soon as another role of the CTA has raised the abort flag.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, Barriers *b, unsigned *err,
                                         unsigned code, bool honour_abort = true) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (ptx::mbar_try_wait_sleep(bar, parity, kSuspendNs)) return true;
        if ((spin & 15u) == 0) {
            if (honour_abort && *(volatile int *)&b->abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > kWaitLimitNs) {
                atomicCAS(err, 0u, code);
                *(volatile int *)&b->abort_flag = 1;
                return false;
            }
        }
    }
}

__device__ __forceinline__ float min3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// Accesses to the barrier block's exchange arrays (the item queue, the two
// column halves' partials).  The block sits behind a base pointer rebuilt from
// an integer (1024-byte alignment), so plain C++ accesses compile to generic
// loads and stores; with E they are shared-memory instructions by 32-bit
// address, volatile and ordered with the barrier waits.  Measured at the 8K
// shape: LSSAR +1.1 %, while the plain softmax kernel lost 5 % to a different
// register allocation, so that kernel keeps the plain accesses.
template <bool E>
__device__ __forceinline__ float xld(float *p) {
    if constexpr (E) return ptx::ld_shared_f32(ptx::smem_u32(p));
    else return *p;
}
template <bool E>
__device__ __forceinline__ void xst(float *p, float v) {
    if constexpr (E) ptx::st_shared_f32(ptx::smem_u32(p), v);
    else *p = v;
}
template <bool E>
__device__ __forceinline__ int xld(int *p) {
    if constexpr (E) return ptx::ld_shared_s32(ptx::smem_u32(p));
    else return *(volatile int *)p;
}
template <bool E>
__device__ __forceinline__ void xst(int *p, int v) {
    if constexpr (E) ptx::st_shared_s32(ptx::smem_u32(p), v);
    else *(volatile int *)p = v;
}

// softplus(x)/ln 2 for z = x log2 e: max(z, 0) + log2(1 + 2^-|z|), two lanes.
// sp2(-inf) = 0.
__device__ __forceinline__ float2 sp2x2(float2 z) {
    const float2 u = make_float2(ptx::ex2(-fabsf(z.x)), ptx::ex2(-fabsf(z.y)));
    const float2 v = __fadd2_rn(u, make_float2(1.f, 1.f));
    return __fadd2_rn(make_float2(fmaxf(z.x, 0.f), fmaxf(z.y, 0.f)),
                      make_float2(ptx::lg2(v.x), ptx::lg2(v.y)));
}

// sp2 evaluated directly as log2(1 + 2^z).  Exact in real arithmetic and free of
// overflow here because |z| <= log2(e) ln(d) ln(L) * 1.001 < 117 for d <= 128 and
// L <= 2^24 (the C ABI rejects longer sequences); for z < -24 the 1 + 2^z rounds
// to 1 and the (tiny, < 1e-7) softplus reads 0.  sp2(-inf) = 0.
__device__ __forceinline__ float2 sp2x2_direct(float2 z) {
    const float2 e = make_float2(ptx::ex2(z.x), ptx::ex2(z.y));
    const float2 v = __fadd2_rn(e, make_float2(1.f, 1.f));
    return make_float2(ptx::lg2(v.x), ptx::lg2(v.y));
}

__device__ __forceinline__ float sp2(float z) {
    return ptx::lg2(1.f + ptx::ex2(z));
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

// A re-weighted row counts as all-zero when sp2(m) - theta is within a few
// times the evaluation error of sp2 in pass 2: its weights would then follow
// that error rather than the scores.  Pass 2 evaluates sp2 of different
// columns by different formulas (MUFU ex2 and lg2: about 2.4e-7 of the value;
// the polynomial log2: up to 2.2e-6 absolute), and pass 1 sums it in product
// form, so columns with equal scores can differ by about 2.5e-6 + 2.4e-7 sp2.
// The band is 1e-5 sp2(m) + 2e-5: about 40 times the relative and 8 times
// the absolute part.
constexpr float kDegenerateRel = 1e-5f;
constexpr float kDegenerateAbs = 2e-5f;
// Weights of such a row: the saturating FMA sat(phi * 2^126 + 0) is exactly 1
// for every column whose normaliser value phi (softplus, 2^(z - m), sigmoid)
// is positive in fp32 and exactly 0 on the masked columns above the diagonal
// (phi = 0 there), so the output is the prefix mean.  (Columns whose softplus
// rounds to 0 in fp32, scores below -24 on the two-transcendental path, also
// get 0; a row read as uniform has them only if every score is below -24.)
constexpr float kUniformSlope = 8.507059e37f;   // 2^126

struct RowConst {
    float a;       // score scale: z = a * s
    float kappa;   // LSSAR slope
    float beta;    // LSSAR offset
    float m;       // softmax: row maximum of z
    float ck;      // LSSAR one-exponential weights: kappa / ln 2
    bool uniform;  // re-weighted row read as all-zero (prefix mean)
    bool fast;     // LSSAR: the one-exponential weights meet the error bound on this row
};

// One-exponential LSSAR weights of one chunk of z (rows whose bound holds):
// w = sat((z + u / ln 2) kappa + beta)^p with u = 2^-|z|.
template <int PK>
__device__ __forceinline__ void weights_fast_z(const uint32_t (&r)[32], const RowConst &rc, int p,
                                               float2 &acc, uint32_t *pk) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float2 z = make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
        const float2 u = make_float2(ptx::ex2(-fabsf(z.x)), ptx::ex2(-fabsf(z.y)));
        const float2 t = __ffma2_rn(z, make_float2(rc.kappa, rc.kappa), make_float2(rc.beta, rc.beta));
        const float2 w = powk2<PK>(ptx::fma_sat2(u, make_float2(rc.ck, rc.ck), t), p);
        acc = __fadd2_rn(acc, w);
        pk[j / 2] = ptx::pack_bf16x2(w.x, w.y);
    }
}

// Scores of one 32-column chunk to z in place: z = a * s for the softmax
// normalisers (raw q, k); the normalised modes' query rows already carry the
// length scale (the prologue writes a_i qh_i in fp16), so their S is z and
// only the diagonal tile is touched.  On the diagonal tile the columns above
// row t become -inf (+inf for the sigmoid mode, whose registers hold -z).
template <int MODE, bool DIAG>
__device__ __forceinline__ void to_z(uint32_t (&r)[32], int col0, int t, float a) {
    constexpr float kMasked = MODE == kSigmoidRw ? INFINITY : -INFINITY;
    constexpr bool kScaled = uses_normalised_qk(MODE);
    if constexpr (!kScaled || DIAG) {
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            float2 z = make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
            if (!kScaled) z = __fmul2_rn(z, make_float2(a, a));
            if (DIAG) {
                if (col0 + j > t) z.x = kMasked;
                if (col0 + j + 1 > t) z.y = kMasked;
            }
            r[j] = __float_as_uint(z.x);
            r[j + 1] = __float_as_uint(z.y);
        }
    }
}

// Pass-1 statistics of one chunk of z: running max and, for LSSAR, the two
// parts of sum_j sp2(z_j) = sum_j max(z_j, 0) + log2(prod_j (1 + 2^-|z_j|)).
// The product form needs one FFMA per element instead of a log2: every factor
// lies in (1, 2], so up to 64 factors multiply in fp32 without overflow (the
// caller takes log2 of each 64-factor product once per tile).
// Off the diagonal tile (DIAG = false, no masked column) the positive part is
// summed as (z - (-|z|)) / 2 with the -|z| the exponential needs anyway: two
// packed FMAs per pair instead of two max and a packed add.
template <int MODE, bool DIAG>
__device__ __forceinline__ void stats_z(const uint32_t (&r)[32], float2 &relu_acc, float2 &prod,
                                        float &m) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float2 z = make_float2(__uint_as_float(r[j]), __uint_as_float(r[j + 1]));
        if constexpr (MODE == kSigmoidRw) {
            // z holds -z here: m tracks min(-z); relu_acc sums sigmoid
            m = min3(m, z.x, z.y);
            const float2 v = __fadd2_rn(make_float2(ptx::ex2(z.x), ptx::ex2(z.y)), make_float2(1.f, 1.f));
            relu_acc = __fadd2_rn(relu_acc, make_float2(ptx::rcp(v.x), ptx::rcp(v.y)));
        } else {
            m = max3(m, z.x, z.y);
        }
        if constexpr (MODE == kLssar) {
            const float2 nz = make_float2(-fabsf(z.x), -fabsf(z.y));
            const float2 u = make_float2(ptx::ex2(nz.x), ptx::ex2(nz.y));
            prod = __ffma2_rn(prod, u, prod);
            if constexpr (DIAG) {
                relu_acc = __fadd2_rn(relu_acc, make_float2(fmaxf(z.x, 0.f), fmaxf(z.y, 0.f)));
            } else {
                const float2 twice = __ffma2_rn(nz, make_float2(-1.f, -1.f), z);   // z + |z|
                relu_acc = __ffma2_rn(twice, make_float2(0.5f, 0.5f), relu_acc);
            }
        }
    }
}

// Softmax-normaliser statistics of one tile (two chunks of z): running max
// m_run and sum s1 = sum_j 2^(z_j - m_run), rescaled when the max grows.
// Fully masked prefixes (all -inf so far) leave both untouched.
__device__ __forceinline__ void softmax_tile_stats(const uint32_t (&r0)[32], const uint32_t (&r1)[32],
                                                   float &m_run, float &s1) {
    float tm = -INFINITY;
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        tm = max3(tm, __uint_as_float(r0[j]), __uint_as_float(r0[j + 1]));
        tm = max3(tm, __uint_as_float(r1[j]), __uint_as_float(r1[j + 1]));
    }
    const float mn = fmaxf(m_run, tm);
    if (mn == -INFINITY) return;
    if (mn != m_run) s1 *= ptx::ex2(m_run - mn);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
        const float2 e0 = __fadd2_rn(make_float2(__uint_as_float(r0[j]), __uint_as_float(r0[j + 1])),
                                     make_float2(-mn, -mn));
        const float2 e1 = __fadd2_rn(make_float2(__uint_as_float(r1[j]), __uint_as_float(r1[j + 1])),
                                     make_float2(-mn, -mn));
        acc0 = __fadd2_rn(acc0, make_float2(ptx::ex2(e0.x), ptx::ex2(e0.y)));
        acc1 = __fadd2_rn(acc1, make_float2(ptx::ex2(e1.x), ptx::ex2(e1.y)));
    }
    s1 += (acc0.x + acc0.y) + (acc1.x + acc1.y);
    m_run = mn;
}

// Pairs of each 16-pair chunk whose LSSAR softplus takes the polynomial log2
// (spread evenly over the chunk), to share the pass-2 work between the MUFU
// and FMA pipes.  The longer power chains (p = 15, runtime p) leave the FMA
// pipe less room.  Measured at the 8K shape, kernel TFLOP/s for 0/3/5/7 of 16:
// p = 15 607.6/626.5/622.0/619.0, p = 3 632.8/645.4/678.0/668.1.
__host__ __device__ constexpr int poly_pairs(int pk) { return (pk == 15 || pk == 0) ? 3 : 5; }

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
            w = sp2x2_direct(z);
        } else {
            float2 phi;   // the normaliser's nonnegative value (up to a per-row factor)
            if constexpr (MODE == kLssar) {
                if (poly_pair(j / 2, poly_pairs(PK))) phi = sp2x2_poly(z);
                else phi = sp2x2_direct(z);
            } else if constexpr (MODE == kSoftmaxRw) {
                const float2 e = __fadd2_rn(z, make_float2(-rc.m, -rc.m));
                phi = make_float2(ptx::ex2(e.x), ptx::ex2(e.y));
            } else {   // kSigmoidRw, z holds -z
                const float2 v = __fadd2_rn(make_float2(ptx::ex2(z.x), ptx::ex2(z.y)), make_float2(1.f, 1.f));
                phi = make_float2(ptx::rcp(v.x), ptx::rcp(v.y));
            }
            // ReLU of the re-weighting input by a saturating FMA: phi kappa + beta
            // never exceeds 1 except by rounding (the row maximum maps to 1)
            w = powk2<PK>(ptx::fma_sat2(phi, make_float2(rc.kappa, rc.kappa), make_float2(rc.beta, rc.beta)), p);
        }
        acc = __fadd2_rn(acc, w);
        pk[j / 2] = ptx::pack_bf16x2(w.x, w.y);
    }
}

template <int D, int MODE, int PK>
__global__ void __launch_bounds__(Cfg<D>::kThreads, 1)
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
    // Plain softmax runs in one pass (online maximum, O rescaled in TMEM);
    // LSSA needs no statistics pass; the re-weighting modes need the whole
    // row's first-stage sum before any weight, hence two passes.
    constexpr bool kOnePassSoftmax = MODE == kSoftmax;
    constexpr bool kTwoPass = MODE != kLssa && !kOnePassSoftmax;
    constexpr bool kSepP = D == 64;                       // P in TMEM columns of its own
    constexpr bool kExplicitSmem = MODE != kSoftmax;      // exchange arrays by ld/st.shared
    constexpr int kPCol = 2 * kBN;                        // P_w at kPCol + 64 w (d = 64)
    constexpr int kOCol = kSepP ? 2 * kBN + 128 : 2 * kBN;  // O_w at kOCol + D w
    // S = Q K^T: fp16 normalised operands (LSSA, LSSAR, sigmoid), raw bf16 (softmax modes).
    constexpr bool kRawQK = !uses_normalised_qk(MODE);
    constexpr uint32_t kIdescS = ptx::idesc_f16(kRawQK, kBM, kBN, false, false);
    // O += P V: P bf16 from TMEM (K-major), V bf16 MN-major.
    constexpr uint32_t kIdescPV = ptx::idesc_f16(true, kBM, D, false, true);

    if (threadIdx.x == 0) {
        for (int b = 0; b < C::kQBufs; ++b) {
            ptx::mbar_init(ptx::smem_u32(&bars->q_full[b]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->q_empty[b]), C::kMmaWarps);   // one commit per MMA warp
        }
        for (int w = 0; w < 2; ++w) {
            ptx::mbar_init(ptx::smem_u32(&bars->s_full[w]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->s_free[w]), kTileThreads);
            ptx::mbar_init(ptx::smem_u32(&bars->o_full[w]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->o_free[w]), kTileThreads);
            ptx::mbar_init(ptx::smem_u32(&bars->p_full[w]), kTileThreads);
            ptx::mbar_init(ptx::smem_u32(&bars->p_free[w]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->halves[w]), kTileThreads);
            for (int qq = 0; qq < 4; ++qq) ptx::mbar_init(ptx::smem_u32(&bars->tile_max[w][qq]), 64);
        }
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(ptx::smem_u32(&bars->kv_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->kv_empty[s]), C::kMmaWarps);   // one commit per MMA warp
        }
        for (int s = 0; s < kItemQ; ++s) {
            ptx::mbar_init(ptx::smem_u32(&bars->item_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->item_empty[s]), item_consumers(C::kMmaWarps));
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
    // The launch may overlap the normalisation prologue (a programmatic
    // dependent launch): everything above is local setup; the prologue's
    // outputs (q-hat, k-hat, the zeroed work counter) are read only after this.
    ptx::grid_dependency_wait();

    const int BH = prm.BH;
    auto decode = [&](int item, int &bh, int &m) {
        m = prm.n_pairs - 1 - item / BH;   // longest pairs first
        bh = item % BH;
    };
    // Consumer side of the work-item queue: returns false on a timed-out wait.
    auto next_item = [&](uint32_t &qi, int &item, bool arrive = true) -> bool {
        const uint32_t s = qi % kItemQ, use = qi / kItemQ;
        ++qi;
        if (!wait_bar(ptx::smem_u32(&bars->item_full[s]), use & 1, bars, prm.err, kErrItem))
            return false;
        item = xld<kExplicitSmem>(&bars->item_q[s]);
        if (arrive) ptx::mbar_arrive(ptx::smem_u32(&bars->item_empty[s]));
        return true;
    };
    // A wait taken by every lane of a control warp; the outcome is made
    // warp-uniform so that the warp's control flow never diverges.
    auto wait_all = [&](uint32_t bar, uint32_t parity, unsigned code, bool honour_abort = true) -> bool {
        return __all_sync(0xffffffffu, wait_bar(bar, parity, bars, prm.err, code, honour_abort));
    };

    if (warp < C::kScoreWarp0) {
    if constexpr (C::kSplit) ptx::setmaxnreg_dec<kCtrlRegs>();   // the control warpgroup gives registers back
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // (the whole warp runs the loop; one elected lane issues the copies)
        {
            if (ptx::elect_one()) {
                ptx::prefetch_tensormap(&tmQ);
                ptx::prefetch_tensormap(&tmK);
                ptx::prefetch_tensormap(&tmV);
            }
            uint32_t ring_idx = 0, q_cnt = 0, qi = 0;
            bool ok = true;
            auto push = [&](const CUtensorMap *map, int tile, int bh) -> bool {
                const uint32_t s = ring_idx % NS, use = ring_idx / NS;
                if (use > 0 && !wait_all(ptx::smem_u32(&bars->kv_empty[s]), (use - 1) & 1, kErrKvEmpty))
                    return false;
                const uint32_t full = ptx::smem_u32(&bars->kv_full[s]);
                const bool in_range = dcheck(tile >= 0 && tile < prm.n_qtiles && bh >= 0 && bh < prm.BH,
                                             prm.err, kDbgTma);
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(full, TB);
#pragma unroll
                    for (int b = 0; b < D / 64; ++b)
                        if (in_range) ptx::tma_load_3d(ptx::smem_u32(ring + s * TB + b * 16384), map, full, b * 64,
                                         tile * kBN, bh);
                }
                __syncwarp();
                ++ring_idx;
                return true;
            };
            while (ok) {
                // claim and publish the next work item
                const uint32_t s = qi % kItemQ, use = qi / kItemQ;
                const int fixed = qi < 2 ? prm.first_items[blockIdx.x][qi] : -1;
                int item = fixed;
                if (fixed < 0) {
                    if (lane == 0) item = (int)(prm.tail_base + atomicAdd(prm.counter, 1u));
                    item = __shfl_sync(0xffffffffu, item, 0);
                }
                ++qi;
                if (use > 0 && !wait_all(ptx::smem_u32(&bars->item_empty[s]), (use - 1) & 1, kErrItem))
                    break;
                if (lane == 0) {
                    xst<kExplicitSmem>(&bars->item_q[s], item);
                    ptx::mbar_arrive(ptx::smem_u32(&bars->item_full[s]));
                }
                __syncwarp();
                if (item >= prm.n_items) break;

                int bh, m;
                decode(item, bh, m);
                const int qa = 2 * m, qb = 2 * m + 1;
                const bool vb = qb < prm.n_qtiles;
                const int nk = vb ? qb + 1 : qa + 1;
                if (!dcheck(item >= 0 && m >= 0 && m < prm.n_pairs && bh >= 0 && bh < prm.BH, prm.err, kDbgItem))
                    break;
                const uint32_t qbuf = q_cnt % C::kQBufs, quse = q_cnt / C::kQBufs;
                if (quse > 0 && !wait_all(ptx::smem_u32(&bars->q_empty[qbuf]), (quse - 1) & 1, kErrQEmpty))
                    break;
                const uint32_t qf = ptx::smem_u32(&bars->q_full[qbuf]);
                uint8_t *qdst = sQ + qbuf * 2 * TB;
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(qf, (vb ? 2 : 1) * TB);
#pragma unroll
                    for (int b = 0; b < D / 64; ++b) {
                        ptx::tma_load_3d(ptx::smem_u32(qdst + b * 16384), &tmQ, qf, b * 64, qa * kBM, bh);
                        if (vb)
                            ptx::tma_load_3d(ptx::smem_u32(qdst + TB + b * 16384), &tmQ, qf, b * 64,
                                             qb * kBM, bh);
                    }
                }
                __syncwarp();
                ++q_cnt;
                if (kTwoPass)
                    for (int kt = 0; ok && kt < nk; ++kt) ok = push(&tmK, kt, bh);
                if (ok) ok = push(&tmK, 0, bh);
                for (int kt = 0; ok && kt < nk; ++kt) {
                    if (kt + 1 < nk) ok = push(&tmK, kt + 1, bh);
                    if (ok) ok = push(&tmV, kt, bh);
                }
            }
            // No copy may be in flight when the CTA ends, also after an abort:
            // wait (bounded) until the last stages and Q tiles issued have landed.
            for (uint32_t i = ring_idx > (uint32_t)NS ? ring_idx - NS : 0; i < ring_idx; ++i)
                wait_bar(ptx::smem_u32(&bars->kv_full[i % NS]), (i / NS) & 1, bars, prm.err, kErrDrain, false);
            for (uint32_t i = q_cnt > (uint32_t)C::kQBufs ? q_cnt - C::kQBufs : 0; i < q_cnt; ++i)
                wait_bar(ptx::smem_u32(&bars->q_full[i % C::kQBufs]), (i / C::kQBufs) & 1, bars, prm.err,
                         kErrDrain, false);
        }
        __syncwarp();
    } else if (warp == 1 || (C::kMmaWarps == 2 && warp == kMmaWarp1)) {
        // ------------------------------------------------------------ MMA issuers
        // d = 64: warp 1 issues for Q tile 0 of each pair and warp kMmaWarp1 for
        // tile 1, so that the two tiles' chains of waits and issues overlap;
        // d = 128: warp 1 issues for both tiles (NT = 2).  The whole warp runs
        // the loop; one elected lane issues the MMAs and commits.  Every MMA
        // warp walks the producer's whole stage sequence and commits every
        // stage's release (a stage is free after one commit per MMA warp).
        constexpr int NT = C::kMmaWarps == 2 ? 1 : 2;   // Q tiles per MMA warp
        const int wbase = warp == 1 ? 0 : 1;
        auto tile = [&](int t) { return NT == 2 ? t : wbase; };
        uint32_t ring_idx = 0, q_cnt = 0, qi = 0;
        uint32_t sf_phase[NT], of_phase[NT], pf_phase[NT];
        bool s_pending[NT], o_pending[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            sf_phase[t] = of_phase[t] = pf_phase[t] = 0;
            s_pending[t] = o_pending[t] = false;
        }
        bool ok = true;
        auto acquire = [&](uint32_t &slot) -> bool {
            slot = ring_idx % NS;
            const uint32_t use = ring_idx / NS;
            ++ring_idx;
            if (!wait_all(ptx::smem_u32(&bars->kv_full[slot]), use & 1, kErrKvFull)) return false;
            ptx::tc_fence_after();
            return true;
        };
        // S of tile t may be overwritten once its warpgroups have released it
        auto touch_s = [&](int t) -> bool {
            if (!s_pending[t]) return true;
            if (!wait_all(ptx::smem_u32(&bars->s_free[tile(t)]), sf_phase[t], kErrSFree)) return false;
            sf_phase[t] ^= 1;
            s_pending[t] = false;
            ptx::tc_fence_after();
            return true;
        };
        auto wait_o_free = [&](int t) -> bool {
            if (!o_pending[t]) return true;
            if (!wait_all(ptx::smem_u32(&bars->o_free[tile(t)]), of_phase[t], kErrOFree)) return false;
            of_phase[t] ^= 1;
            o_pending[t] = false;
            ptx::tc_fence_after();
            return true;
        };
        auto commit = [&](uint64_t *bar) {
            const uint32_t b = ptx::smem_u32(bar);
            if (ptx::elect_one()) ptx::mma_commit(b);
            __syncwarp();
        };
        // Descriptors are built once; a K step moves the start address field
        // (16-byte units, bits 0-13), which never carries for these offsets.
        const uint64_t desc_q0 = ptx::smem_desc_sw128(ptx::smem_u32(sQ), kKmajorLbo, kKmajorSbo);
        const uint64_t desc_k0 = ptx::smem_desc_sw128(ptx::smem_u32(ring), kKmajorLbo, kKmajorSbo);
        const uint64_t desc_v0 = ptx::smem_desc_sw128(ptx::smem_u32(ring), kVLbo, kVSbo);
        uint32_t qoff = 0;   // byte offset of the current item's Q buffer
        // the TMEM columns the MMAs write and read stay inside the 512 allocated
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const int w = tile(t);
            dcheck(tmem_in_range(tmem + w * kBN, tmem, kBN, 512) &&
                       tmem_in_range(tmem + kOCol + w * D, tmem, D, 512) &&
                       (!kSepP || tmem_in_range(tmem + kPCol + 64 * w, tmem, 64, 512)),
                   prm.err, kDbgTmem);
        }
        auto issue_s = [&](int t, uint32_t kslot) {
            const int w = tile(t);
            const uint64_t dq = desc_q0 + (uint64_t)((qoff + w * TB) >> 4);
            const uint64_t dk = desc_k0 + (uint64_t)((kslot * TB) >> 4);
            const uint32_t full = ptx::smem_u32(&bars->s_full[w]);
            if (ptx::elect_one()) {
#pragma unroll
                for (int k = 0; k < D / 16; ++k) {
                    const uint32_t off = ((k / 4) * 16384 + (k % 4) * 32) >> 4;
                    ptx::mma_ss(tmem + w * kBN, dq + off, dk + off, kIdescS, k > 0);
                }
                ptx::mma_commit(full);
            }
            __syncwarp();
            s_pending[t] = true;
        };
        auto issue_pv = [&](int t, uint32_t vslot, bool accumulate) {
            const int w = tile(t);
            const uint64_t dv = desc_v0 + (uint64_t)((vslot * TB) >> 4);
            // P words of keys 16k..16k+15: d = 64, 8k of P_w; d = 128, words
            // (k%4)*8 of the S column half k/4
            if (ptx::elect_one()) {
#pragma unroll
                for (int k = 0; k < kBN / 16; ++k)
                    ptx::mma_ts(tmem + kOCol + w * D,
                                kSepP ? tmem + kPCol + 64 * w + 8 * k
                                      : tmem + w * kBN + (k / 4) * 64 + (k % 4) * 8,
                                dv + (uint64_t)((k * 2048) >> 4), kIdescPV,
                                (accumulate || k > 0) ? 1u : 0u);
            }
            __syncwarp();
        };
        int item;
        while (ok && (ok = __all_sync(0xffffffffu, next_item(qi, item, lane == 0))) && item < prm.n_items) {
            int bh, m;
            decode(item, bh, m);
            const int qa = 2 * m, qb = 2 * m + 1;
            const bool vb = qb < prm.n_qtiles;
            const int n_w[2] = {qa + 1, vb ? qb + 1 : 0};   // K tiles of each Q tile
            const int nk = vb ? qb + 1 : qa + 1;            // K tiles the producer streams
            const uint32_t qbuf = q_cnt % C::kQBufs;
            if (!(ok = wait_all(ptx::smem_u32(&bars->q_full[qbuf]), (q_cnt / C::kQBufs) & 1, kErrQFull)))
                break;
            ++q_cnt;
            qoff = qbuf * 2 * TB;
            ptx::tc_fence_after();
            uint32_t slot;
            if (kTwoPass) {
                for (int kt = 0; ok && kt < nk; ++kt) {
                    if (!(ok = acquire(slot))) break;
#pragma unroll
                    for (int t = 0; t < NT; ++t)
                        if (ok && kt < n_w[tile(t)] && (ok = touch_s(t))) issue_s(t, slot);
                    commit(&bars->kv_empty[slot]);
                }
            }
            if (!ok || !(ok = acquire(slot))) break;
#pragma unroll
            for (int t = 0; t < NT; ++t)
                if (ok && n_w[tile(t)] > 0 && (ok = touch_s(t))) issue_s(t, slot);
            commit(&bars->kv_empty[slot]);
            for (int kt = 0; ok && kt < nk; ++kt) {
                const bool has_next = kt + 1 < nk;
                uint32_t kslot = 0, vslot;
                if (has_next && !(ok = acquire(kslot))) break;
                if constexpr (kSepP) {
                    // next scores as soon as the warpgroups have loaded S(kt)
#pragma unroll
                    for (int t = 0; t < NT; ++t)
                        if (ok && kt + 1 < n_w[tile(t)] && (ok = touch_s(t))) issue_s(t, kslot);
                    if (!ok) break;
                    if (has_next) commit(&bars->kv_empty[kslot]);
                    if (!(ok = acquire(vslot))) break;
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        const int w = tile(t);
                        if (!ok || kt >= n_w[w]) continue;
                        if (!(ok = wait_all(ptx::smem_u32(&bars->p_full[w]), pf_phase[t], kErrPFull))) continue;
                        pf_phase[t] ^= 1;
                        ptx::tc_fence_after();
                        if (kt == 0 && !(ok = wait_o_free(t))) continue;
                        issue_pv(t, vslot, kt > 0);
                        commit(&bars->p_free[w]);
                        if (kt + 1 == n_w[w]) {
                            commit(&bars->o_full[w]);
                            o_pending[t] = true;
                        }
                    }
                    commit(&bars->kv_empty[vslot]);
                } else {
                    if (!(ok = acquire(vslot))) break;
#pragma unroll
                    for (int t = 0; t < NT; ++t) {
                        const int w = tile(t);
                        if (!ok || kt >= n_w[w]) continue;
                        if (!(ok = touch_s(t))) continue;   // P_w(kt) is in TMEM
                        if (kt == 0 && !(ok = wait_o_free(t))) continue;
                        issue_pv(t, vslot, kt > 0);
                        if (kt + 1 < n_w[w]) {
                            issue_s(t, kslot);
                        } else {
                            commit(&bars->o_full[w]);
                            o_pending[t] = true;
                        }
                    }
                    commit(&bars->kv_empty[vslot]);
                    if (has_next) commit(&bars->kv_empty[kslot]);
                }
            }
            commit(&bars->q_empty[qbuf]);
        }
        __syncwarp();
    }   // warp 3 of the control warpgroup (d = 64) has no role
    } else {
        if constexpr (C::kSplit) ptx::setmaxnreg_inc<kScoreRegs>();   // each score warpgroup takes them
        // ------------------------------------------------------------ score warpgroups
        const int g = (warp - C::kScoreWarp0) >> 2;    // 0..3
        const int w = g & 1;                        // Q tile of the pair
        const int h = g >> 1;                       // column half of the S tile
        const int t = (warp & 3) * 32 + lane;       // row within the Q tile = TMEM lane
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_col = tmem + lane_addr + w * kBN + h * 64;
        const uint32_t o_col = tmem + lane_addr + kOCol + w * D + h * (D / 2);
        const uint32_t p_col = kSepP ? tmem + lane_addr + kPCol + 64 * w + 32 * h : s_col;
        const uint32_t p_full = ptx::smem_u32(&bars->p_full[w]);
        const uint32_t p_free = ptx::smem_u32(&bars->p_free[w]);
        uint32_t pf_phase = 0;
        // every TMEM access of this warp stays inside the allocation and in
        // its own lane quarter
        dcheck(tmem_in_range(s_col, tmem, 64, 512) && tmem_in_range(o_col, tmem, D / 2, 512) &&
                   tmem_in_range(p_col, tmem, 32, 512) && ((s_col >> 16) & ~31u) == (uint32_t)((warp & 3) * 32),
               prm.err, kDbgTmem);
        bool p_pending = false;   // a P.V MMA may still be reading this warpgroup's P words
        const uint32_t s_full = ptx::smem_u32(&bars->s_full[w]);
        const uint32_t s_free = ptx::smem_u32(&bars->s_free[w]);
        const uint32_t o_full = ptx::smem_u32(&bars->o_full[w]);
        const uint32_t o_free = ptx::smem_u32(&bars->o_free[w]);
        const uint32_t halves = ptx::smem_u32(&bars->halves[w]);   // this tile's two column halves
        uint32_t hv_phase = 0;
        // softmax: the two warps holding the two column halves of rows
        // 32 (warp % 4) .. +31 of tile w meet here once per K tile
        const uint32_t tmax_bar = ptx::smem_u32(&bars->tile_max[w][warp & 3]);
        uint32_t tm_phase = 0;
        // this row's two tile-maximum slots (alternating by K tile) and the
        // offset of the partner half's slot
        const uint32_t tm_slot0 = ptx::smem_u32(&bars->x_s1[w][h][t]);
        const uint32_t tm_slot1 = ptx::smem_u32(&bars->x_m[w][h][t]);
        const uint32_t tm_other = (uint32_t)((h ? -1 : 1) * (int)(kBM * sizeof(float)));
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
            const int p_row = (PK == 0 && prm.per_head) ? prm.p_head[bh % prm.H] : prm.p;
            RowConst rc;
            if constexpr (kRawQK)
                rc.a = log2e * rsqrtf((float)D);
            else if constexpr (MODE == kSigmoidRw)
                rc.a = -log2e * prm.ln_d * logf(fi);   // registers hold -z
            else
                rc.a = log2e * prm.ln_d * logf(fi);
            rc.kappa = 0.f;
            rc.beta = 0.f;
            rc.m = kOnePassSoftmax ? -INFINITY : 0.f;
            rc.ck = 0.f;
            rc.uniform = false;
            rc.fast = false;
            if constexpr (kTwoPass) {
                float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                constexpr float kInit = MODE == kSigmoidRw ? INFINITY : -INFINITY;
                float mx[2] = {kInit, kInit};
                float s1_log = 0.f;   // sum over tiles of log2 of the 64-factor products
                float sm_run = -INFINITY, sm_sum = 0.f;   // softmax normaliser statistics
                for (int kt = 0; kt < n; ++kt) {
                    if (!(ok = wait_warp(s_full, sf_phase, kErrSFull))) break;
                    sf_phase ^= 1;
                    ptx::tc_fence_after();
                    uint32_t r[2][32];
                    ptx::tmem_ld32(s_col, r[0]);
                    ptx::tmem_ld32(s_col + 32, r[1]);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence(r[0]);
                    ptx::reg_fence(r[1]);
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(s_free);   // S may be overwritten: values are in registers
                    if (kt == qt) {
                        to_z<MODE, true>(r[0], 64 * h, t, rc.a);
                        to_z<MODE, true>(r[1], 64 * h + 32, t, rc.a);
                    } else {
                        to_z<MODE, false>(r[0], 64 * h, t, rc.a);
                        to_z<MODE, false>(r[1], 64 * h + 32, t, rc.a);
                    }
                    if constexpr (MODE == kSoftmaxRw) {
                        softmax_tile_stats(r[0], r[1], sm_run, sm_sum);
                    } else {
                        float2 prod[2] = {make_float2(1.f, 1.f), make_float2(1.f, 1.f)};
                        if (kt == qt) {
                            stats_z<MODE, true>(r[0], acc[0], prod[0], mx[0]);
                            stats_z<MODE, true>(r[1], acc[1], prod[1], mx[1]);
                        } else {
                            stats_z<MODE, false>(r[0], acc[0], prod[0], mx[0]);
                            stats_z<MODE, false>(r[1], acc[1], prod[1], mx[1]);
                        }
                        if constexpr (MODE == kLssar)
                            s1_log += ptx::lg2((prod[0].x * prod[0].y) * (prod[1].x * prod[1].y));
                    }
                }
                if (!ok) break;
                // combine the two column halves of the row (max of z, sum of phi)
                if constexpr (MODE == kSoftmaxRw) {
                    xst<kExplicitSmem>(&bars->x_m[w][h][t], sm_run);
                    xst<kExplicitSmem>(&bars->x_s1[w][h][t], sm_sum);
                } else if constexpr (MODE == kSigmoidRw) {
                    xst<kExplicitSmem>(&bars->x_m[w][h][t], -fminf(mx[0], mx[1]));
                    xst<kExplicitSmem>(&bars->x_s1[w][h][t], (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y));
                } else {
                    xst<kExplicitSmem>(&bars->x_m[w][h][t], fmaxf(mx[0], mx[1]));
                    if constexpr (MODE == kLssar)
                        xst<kExplicitSmem>(&bars->x_s1[w][h][t], (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y) + s1_log);
                }
                // both halves' partials are in shared memory (bounded wait)
                ptx::mbar_arrive(halves);
                if (!(ok = wait_warp(halves, hv_phase, kErrHalves))) break;
                hv_phase ^= 1;
                const float m0 = xld<kExplicitSmem>(&bars->x_m[w][0][t]), m1 = xld<kExplicitSmem>(&bars->x_m[w][1][t]);
                const float mxr = fmaxf(m0, m1);
                if constexpr (MODE == kSoftmax) {
                    rc.m = mxr;
                } else if constexpr (MODE == kSoftmaxRw) {
                    // halves with no unmasked column carry m = -inf and a zero sum
                    const float s1 = xld<kExplicitSmem>(&bars->x_s1[w][0][t]) * ptx::ex2(m0 - mxr) +
                                     xld<kExplicitSmem>(&bars->x_s1[w][1][t]) * ptx::ex2(m1 - mxr);
                    rc.m = mxr;
                    const float o = (row + 1 <= 3) ? 0.f : 1.f;
                    const float theta = o * s1 / fi;   // in units of the row maximum 2^0 = 1
                    const float den = 1.f - theta;
                    if (den > kDegenerateRel + kDegenerateAbs) {
                        rc.kappa = 1.f / den;
                        rc.beta = -theta * rc.kappa;
                    } else {
                        rc.kappa = kUniformSlope;   // all-zero re-weighted row (see kUniformSlope)
                        rc.beta = 0.f;
                        rc.uniform = true;
                    }
                } else if constexpr (MODE == kSigmoidRw) {
                    const float s1 = xld<kExplicitSmem>(&bars->x_s1[w][0][t]) + xld<kExplicitSmem>(&bars->x_s1[w][1][t]);
                    const float o = (row + 1 <= 3) ? 0.f : 1.f;
                    const float theta = o * s1 / fi;
                    const float sgm = ptx::rcp(1.f + ptx::ex2(-mxr));
                    const float den = sgm - theta;
                    if (den > kDegenerateRel * sgm + kDegenerateAbs) {
                        rc.kappa = 1.f / den;
                        rc.beta = -theta * rc.kappa;
                    } else {
                        rc.kappa = kUniformSlope;   // all-zero re-weighted row (see kUniformSlope)
                        rc.beta = 0.f;
                        rc.uniform = true;
                    }
                } else {
                    const float s1 = xld<kExplicitSmem>(&bars->x_s1[w][0][t]) + xld<kExplicitSmem>(&bars->x_s1[w][1][t]);
                    const float o = (row + 1 <= 3) ? 0.f : 1.f;
                    const float theta = o * s1 / fi;
                    const float spm = sp2(mxr);
                    const float den = spm - theta;
                    if (den > kDegenerateRel * spm + kDegenerateAbs) {
                        rc.kappa = 1.f / den;
                        rc.beta = -theta * rc.kappa;
                        if constexpr (PK == 15 || PK == 0) {
                            rc.ck = 2.f * kHalfInvLn2 * rc.kappa;
                            rc.fast = !prm.exact_weights && fast_weights_ok(theta, rc.kappa, fi, p_row);
                        }
                    } else {
                        // All-zero re-weighted row: an exactly uniform LSSA row (all sp
                        // equal), or one whose spread is within the band above
                        // (see kUniformSlope for its weights).
                        rc.kappa = kUniformSlope;
                        rc.beta = 0.f;
                        rc.uniform = true;
                    }
                }
            }
            // pass 2: weights into TMEM, running row sum.  The warp takes the
            // one-exponential LSSAR weights when every one of its rows meets
            // the error bound (a warp-uniform choice).
            const bool fastw = __all_sync(0xffffffffu, rc.fast);
            auto weights = [&](const uint32_t (&r)[32], float2 &acc, uint32_t *pk) {
                if constexpr (MODE == kLssar && (PK == 15 || PK == 0)) {
                    if (fastw) {
                        weights_fast_z<PK>(r, rc, p_row, acc, pk);
                        return;
                    }
                }
                weights_z<MODE, PK>(r, rc, p_row, acc, pk);
            };
            float2 acc2[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
            for (int kt = 0; kt < n; ++kt) {
                if (!(ok = wait_warp(s_full, sf_phase, kErrSFull))) break;
                sf_phase ^= 1;
                ptx::tc_fence_after();
                uint32_t r0[32], r1[32];
                ptx::tmem_ld32(s_col, r0);
                ptx::tmem_ld32(s_col + 32, r1);
                ptx::tmem_ld_wait();
                ptx::reg_fence(r0);
                ptx::reg_fence(r1);
                if constexpr (kOnePassSoftmax) {
                    if constexpr (kSepP) {
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(s_free);   // the next S MMA may start now
                    }
                    if (kt == qt) {
                        to_z<MODE, true>(r0, 64 * h, t, rc.a);
                        to_z<MODE, true>(r1, 64 * h + 32, t, rc.a);
                    } else {
                        to_z<MODE, false>(r0, 64 * h, t, rc.a);
                        to_z<MODE, false>(r1, 64 * h + 32, t, rc.a);
                    }
                    // the row's maximum over this K tile: both column halves'
                    // maxima meet in shared memory (slots alternate by tile)
                    float tm = -INFINITY;
#pragma unroll
                    for (int j = 0; j < 32; j += 2) {
                        tm = max3(tm, __uint_as_float(r0[j]), __uint_as_float(r0[j + 1]));
                        tm = max3(tm, __uint_as_float(r1[j]), __uint_as_float(r1[j + 1]));
                    }
                    const uint32_t slot = (kt & 1) ? tm_slot1 : tm_slot0;
                    ptx::st_shared_f32(slot, tm);
                    ptx::mbar_arrive(tmax_bar);
                    if (!(ok = wait_warp(tmax_bar, tm_phase, kErrTileMax))) break;
                    tm_phase ^= 1;
                    tm = fmaxf(tm, ptx::ld_shared_f32(slot + tm_other));
                    // raise the reference when the tile exceeds it by more than
                    // kRescaleLog2 (the same decision in both halves: the same
                    // maxima); O and the row sum are then multiplied by 2^(old - new)
                    const bool raise = tm > rc.m + kRescaleLog2;
                    const float alpha = raise ? ptx::ex2(rc.m - tm) : 1.f;
                    if (raise) {
                        rc.m = tm;
                        acc2[0] = __fmul2_rn(acc2[0], make_float2(alpha, alpha));
                        acc2[1] = __fmul2_rn(acc2[1], make_float2(alpha, alpha));
                    }
                    // this tile's weights first (the registers of S are then free)
                    uint32_t pk0[16], pk1[16];
                    weights(r0, acc2[0], pk0);
                    weights(r1, acc2[1], pk1);
                    // O holds the previous K tiles' P.V once that MMA has
                    // completed (d = 64: the P-free commit after it; d = 128:
                    // S(kt), issued after it by the same thread, is complete)
                    if constexpr (kSepP) {
                        if (p_pending) {
                            if (!(ok = wait_warp(p_free, pf_phase, kErrPFree))) break;
                            pf_phase ^= 1;
                            ptx::tc_fence_after();
                            p_pending = false;
                        }
                    }
                    // P first (its registers are free once the stores are issued), then O
                    ptx::tmem_st16(p_col, pk0);
                    ptx::tmem_st16(p_col + 16, pk1);
                    if (__any_sync(0xffffffffu, raise) && kt > 0) {
                        constexpr int NC = D / 64;   // 32-column chunks of this half's O
#pragma unroll
                        for (int c = 0; c < NC; ++c) {
                            uint32_t oc[32];
                            ptx::tmem_ld32(o_col + c * 32, oc);
                            ptx::tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < 32; j += 2) {
                                const float2 x = __fmul2_rn(
                                    make_float2(__uint_as_float(oc[j]), __uint_as_float(oc[j + 1])),
                                    make_float2(alpha, alpha));
                                oc[j] = __float_as_uint(x.x);
                                oc[j + 1] = __float_as_uint(x.y);
                            }
                            ptx::tmem_st32(o_col + c * 32, oc);
                        }
                    }
                    ptx::tmem_st_wait();
                    ptx::tc_fence_before();
                    if constexpr (kSepP) {
                        ptx::mbar_arrive(p_full);   // P(kt) is in TMEM
                        p_pending = true;
                    } else {
                        ptx::mbar_arrive(s_free);   // P(kt) is in TMEM over the S columns
                    }
                    continue;
                }
                if constexpr (kSepP) {
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(s_free);   // the next S MMA may start now
                    // both chunks' weights first: the previous P.V MMA reads P
                    // meanwhile, and the wait for it comes just before the stores
                    uint32_t pk0[16], pk1[16];
                    if (kt == qt) to_z<MODE, true>(r0, 64 * h, t, rc.a);
                    else to_z<MODE, false>(r0, 64 * h, t, rc.a);
                    weights(r0, acc2[0], pk0);
                    if (kt == qt) to_z<MODE, true>(r1, 64 * h + 32, t, rc.a);
                    else to_z<MODE, false>(r1, 64 * h + 32, t, rc.a);
                    weights(r1, acc2[1], pk1);
                    if (p_pending) {
                        if (!(ok = wait_warp(p_free, pf_phase, kErrPFree))) break;
                        pf_phase ^= 1;
                        ptx::tc_fence_after();
                    }
                    ptx::tmem_st16(p_col, pk0);
                    ptx::tmem_st16(p_col + 16, pk1);
                    ptx::tmem_st_wait();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(p_full);   // P(kt) is in TMEM
                    p_pending = true;
                    continue;
                }
                // d = 128: each 16-word half of this thread's P row is stored over S
                // columns already loaded above as soon as it is ready
                {
                    uint32_t pk[16];
                    if (kt == qt) to_z<MODE, true>(r0, 64 * h, t, rc.a);
                    else to_z<MODE, false>(r0, 64 * h, t, rc.a);
                    weights(r0, acc2[0], pk);
                    ptx::tmem_st16(p_col, pk);
                }
                {
                    uint32_t pk[16];
                    if (kt == qt) to_z<MODE, true>(r1, 64 * h + 32, t, rc.a);
                    else to_z<MODE, false>(r1, 64 * h + 32, t, rc.a);
                    weights(r1, acc2[1], pk);
                    ptx::tmem_st16(p_col + 16, pk);
                }
                ptx::tmem_st_wait();
                ptx::tc_fence_before();
                ptx::mbar_arrive(s_free);   // P(kt) is in TMEM over the S columns
            }
            if (!ok) break;
            xst<kExplicitSmem>(&bars->x_s2[w][h][t], (acc2[0].x + acc2[0].y) + (acc2[1].x + acc2[1].y));
            ptx::mbar_arrive(halves);
            if (!(ok = wait_warp(halves, hv_phase, kErrHalves))) break;
            hv_phase ^= 1;
            const float s2 = xld<kExplicitSmem>(&bars->x_s2[w][0][t]) + xld<kExplicitSmem>(&bars->x_s2[w][1][t]);
            // epilogue: this half's D/2 output columns
            if (!(ok = wait_warp(o_full, of_phase, kErrOFull))) break;
            of_phase ^= 1;
            ptx::tc_fence_after();
            constexpr int NC = D / 64;   // 32-column chunks per half
            uint32_t o[NC][32];
#pragma unroll
            for (int c = 0; c < NC; ++c) ptx::tmem_ld32(o_col + c * 32, o[c]);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < NC; ++c) ptx::reg_fence(o[c]);
            ptx::tc_fence_before();
            ptx::mbar_arrive(o_free);
            if (row < prm.L && h == 0 && prm.stats != nullptr) {
                // Row statistics for the backward pass: the weights are
                // w = max(phi kappa + beta, 0)^p (p = 1, kappa = 1, beta = 0 in the
                // modes without re-weighting) and W = sum_j w.  A uniform row is
                // stored as kappa = 0, beta = 1, W = i: constant weights, so its
                // scores receive no gradient.
                float4 st;
                st.x = rc.m;
                if constexpr (is_reweight(MODE)) {
                    st.y = rc.uniform ? 0.f : rc.kappa;
                    st.z = rc.uniform ? 1.f : rc.beta;
                    st.w = rc.uniform ? fi : s2;
                } else {
                    st.y = 1.f;
                    st.z = 0.f;
                    st.w = s2;
                }
                if (dcheck(bh < prm.BH && row < prm.L, prm.err, kDbgGlobal))
                    prm.stats[(size_t)bh * prm.L + row] = st;
            }
            if (row < prm.L && dcheck(bh >= 0 && bh < prm.BH, prm.err, kDbgGlobal)) {
                const float inv = 1.f / s2;
                uint4 *dst = reinterpret_cast<uint4 *>(prm.out + ((size_t)bh * prm.L + row) * D +
                                                       h * (D / 2));
#pragma unroll
                for (int c = 0; c < D / 16; ++c) {
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
