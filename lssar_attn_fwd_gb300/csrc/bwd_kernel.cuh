// Tensor-core backward pass of causal LSSAR / LSSA / softmax attention for sm_103a.
//
// Gradients of sum(dout * out) (the notes on "Softplus Attention with
// Re-weighting Boosts Length Extrapolation in Large Language Models" train
// with this attention; the formulas are the chain rule through Key designs
// 1-2 in the forward kernel's log2 units).  For query row i (1-based) and key
// j <= i, with the forward's saved row constants {m, kappa, beta, W}:
//   z_ij = a_i s_ij         s = qh_i . kh_j (fp16 normalised rows) or q_i . k_j (softmax)
//   b_ij = phi(z_ij)        log2(1 + 2^z) | 2^(z - m_i) | 1/(1 + 2^-z)
//   w_ij = max(b kappa_i + beta_i, 0)^p = u_ij * max(b kappa_i + beta_i, 0)
//   P_ij = w_ij / W_i,   dP_ij = dout_i . v_j,   D_i = sum_j P_ij dP_ij
//   F_i  = p kappa_i / W_i,   dS1_i = -(O_i / i) F_i sum_j (dP_ij - D_i) u_ij
//   ds_ij = a_i phi'(z_ij) (F_i (dP_ij - D_i) u_ij + dS1_i)
//   dqh_i = sum_j ds_ij kh_j,  dkh_j = sum_i ds_ij qh_i,  dv_j = sum_i P_ij dout_i
// (without re-weighting: p = 1, kappa = 1, beta = 0, u = 1, dS1 = 0).
//
// Two launches of one kernel template:
//   row pass (PASS = kRowPass), one item per 128-query tile, anchor = (qh, dout):
//     pass 1 over the key tiles: S = Qh Kh^T, dP = dO V^T; per row D_i, the
//     sum for dS1_i and the range of dP (which bounds |ds| for the fp16 scale
//     r_i); pass 2: S, dP again, ds / r_i -> TMEM, dQh += (ds / r_i) Kh.
//     Writes dq (the gradient of the row normalisation applied to dqh in the
//     epilogue), the per-query record used by the column pass, and the
//     per-head maximum R of r_i.
//   column pass (PASS = kColPass), one item per 128-key tile, anchor = (kh, v):
//     one pass over the query tiles i >= j: S^T = Kh Qh^T, dP^T = V dO^T,
//     P^T and ds^T / R -> TMEM, dV += P^T dO, dKh += (ds^T / R) Qh.  The
//     query records arrive with each tile (bulk copy into the stage).  Writes
//     dv and dk (the normalisation gradient applied to dkh in the epilogue).
// In the normalised modes the prologue writes the query rows as a_i qh_i
// (fp16), exactly as the forward does, so S is z itself; the column pass's
// product with those rows then takes ds_ij / a_i.
// The same stage tile serves as the K-major B operand of a score product and
// as the MN-major B operand of an accumulation (the 128B-swizzled TMA layout
// is both); ds is rounded to the score operands' type (fp16 for the
// normalised modes), scaled into [-1, 1] per row (row pass) or per head
// (column pass) so that fp16 cannot overflow.
//
// Roles (576 threads): warp 0 TMA producer, warp 1 TMEM owner + single-thread
// MMA issuer, warps 2-17 four math warpgroups; warpgroup g owns partner
// columns [32g, 32g+32) of every tile, thread t owns anchor row t (TMEM lane).
// TMEM: S [0,128), dP [128,256), Acc1 [256,256+D), Acc2 (column pass)
// [256+D,256+2D), A operands (packed 16-bit pairs, 64 columns each) after
// them; column pass at d = 128: the A operands overwrite the first half of
// each warpgroup's S / dP columns.
// Every mbarrier wait is bounded; on expiry the kernel records a code in the
// device error word, raises an abort flag and all roles leave their loops.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "fast_weights.cuh"
#include "lssar_internal.cuh"
#include "tc_ptx.cuh"

namespace lssar {
namespace tcb {

using Diag = std::true_type;       // the causal diagonal tile of an item
using OffDiag = std::false_type;   // a tile without masked elements
using Fast = std::true_type;       // one-exponential LSSAR weights (rows within the bound)
using Exact = std::false_type;     // log2(1 + 2^z) weights

constexpr int kBM = 128;                  // anchor rows of an item (TMEM lanes)
constexpr int kBN = 128;                  // partner rows of a streamed tile
constexpr int kMathWarp0 = 2;
constexpr int kMathThreads = 4 * kBM;
constexpr int kAccWarp = 18;      // accumulation issuer, when there are two issuers
constexpr int kItemQ = 4;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kSuspendNs = 1000000;

enum Pass : int { kRowPass = 0, kColPass = 1 };

// Error codes in the device error word (the forward kernel uses 1-11).
enum : unsigned { kErrXFull = 21, kErrXEmpty, kErrRingFull, kErrRingEmpty, kErrSFull, kErrSFree,
                  kErrAFull, kErrAFree, kErrAccFull, kErrAccFree, kErrItem, kErrRed, kErrDrain, kErrFin };

constexpr uint32_t kKmajorLbo = 16, kKmajorSbo = 1024;    // K-major tiles
constexpr uint32_t kMnLbo = 16384, kMnSbo = 1024;         // the same tiles read MN-major

struct Params {
    int BH, L;
    int n_tiles;               // ceil(L / 128)
    int n_items;               // BH * n_tiles
    float ln_d;
    int p;                     // exponent (generic power path)
    int H;                     // heads per batch entry (for the per-head exponents)
    int per_head;              // 1: head h uses p_head[h] (generic power path only)
    int exact_weights;         // 1: LSSAR rows never take the one-exponential weights
    int p_head[256];
    const float4 *stats;       // row pass: [BH][L] {m, kappa, beta, W}
    float *rowc;               // [BH][n_tiles][8 fields][128] per-query records (row pass writes)
    unsigned *rmax;            // [BH] max of r_i as float bits (zero before the row pass)
    const __nv_bfloat16 *xraw; // row pass: q, column pass: k (raw rows, for the normalisation gradient)
    __nv_bfloat16 *grad;       // row pass: dq, column pass: dk; [BH][L][D]
    __nv_bfloat16 *dv;         // column pass: dv [BH][L][D]
    unsigned *err;             // device error word
    unsigned *counter;         // work counter, zero at launch
};

template <int D>
struct Cfg {
    static constexpr int kTB = kBN * D * 2;                    // one 128-row tile
    static constexpr int kConstBytes = kBN * 32;               // 128 query records
    static constexpr int kStageBytes = 2 * kTB + kConstBytes;  // partner tiles + records
    static constexpr int kStages = D == 64 ? 4 : 2;
    static constexpr int kRingOff = 2 * kTB;                   // after the two anchor tiles
    static constexpr int kBarOff = kRingOff + kStages * kStageBytes;
    static constexpr int kBarBytes = 16384;
    static constexpr int kSmemBytes = kBarOff + kBarBytes + 1024;
};

template <int D, int PASS>
struct Tmem {
    static constexpr bool kAlias = PASS == kColPass && D == 128;
    static constexpr uint32_t kS = 0, kDP = 128, kAcc1 = 256, kAcc2 = 256 + D;
    static constexpr uint32_t kA1 = kAlias ? 0u : (PASS == kRowPass ? 256u + D : 256u + 2 * D);
    static constexpr uint32_t kA2 = kAlias ? 128u : kA1 + 64;
    // Two MMA issuers (warp 1: S and dP; warp kAccWarp: the accumulations)
    // unless A is written over S / dP, where the next scores must follow the
    // accumulation in one issue order.
    static constexpr int kIssuers = kAlias ? 1 : 2;
    static constexpr int kThreads = 576 + 32 * (kIssuers - 1);
    static constexpr uint32_t kItemConsumers = kIssuers + kMathThreads;
};
static_assert(Tmem<128, kRowPass>::kA1 + 64 <= 512 && Tmem<64, kColPass>::kA2 + 64 <= 512, "TMEM");
static_assert(Cfg<64>::kSmemBytes <= 232448 && Cfg<128>::kSmemBytes <= 232448, "shared memory per CTA");

struct __align__(8) Barriers {
    uint64_t x_full, x_empty;
    uint64_t ring_full[4], ring_empty[4];
    uint64_t s_full, s_free, a_full, a_free, acc_full, acc_free;
    uint64_t red;              // row pass: the four warpgroups' partials are in x_red
    uint64_t fin;              // epilogue: the four warpgroups' partials are in x_fin
    uint64_t item_full[kItemQ], item_empty[kItemQ];
    int item_q[kItemQ];
    uint32_t tmem_base;
    int abort_flag;
    float x_red[5][4][kBM];    // row pass: partial row sums of the four warpgroups
    float x_fin[2][4][kBM];    // epilogue: partial |x|^2 and x.g of the four warpgroups
};
static_assert(sizeof(Barriers) <= 16384, "barrier block too large");

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

__device__ __forceinline__ float max3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

__device__ __forceinline__ float min3(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// u = base^(p-1) (and w = u * base by the caller); p = 1 gives the ReLU's
// derivative, 1 for base > 0.
template <int PK>
__device__ __forceinline__ float2 pow_pm1(float2 b, int p) {
    if constexpr (PK == 3) {
        return __fmul2_rn(b, b);
    } else if constexpr (PK == 15) {
        const float2 b2 = __fmul2_rn(b, b), b3 = __fmul2_rn(b2, b), b6 = __fmul2_rn(b3, b3);
        const float2 b7 = __fmul2_rn(b6, b);
        return __fmul2_rn(b7, b7);
    } else {
        if (p == 1) return make_float2(b.x > 0.f ? 1.f : 0.f, b.y > 0.f ? 1.f : 0.f);
        float2 acc = make_float2(1.f, 1.f), r = b;
        int e = p - 1;
        while (e) {
            if (e & 1) acc = __fmul2_rn(acc, r);
            r = __fmul2_rn(r, r);
            e >>= 1;
        }
        return acc;
    }
}

// Per-element quantities of a pair of scores z (already scaled).
struct Elem {
    float2 u;       // base^(p-1) (1 without re-weighting)
    float2 w;       // the weight
    float2 slope;   // dphi/dz
};

// z of a pair of scores: the normalised modes' query rows carry the length
// scale already (the prologue writes a_i qh_i), so S is z; the softmax
// normalisers scale raw q.k by a = log2(e) / sqrt(d).
template <int MODE>
__device__ __forceinline__ float2 score_z(uint32_t s0, uint32_t s1, float a) {
    const float2 s = make_float2(__uint_as_float(s0), __uint_as_float(s1));
    if constexpr (uses_normalised_qk(MODE)) return s;
    else return __fmul2_rn(s, make_float2(a, a));
}

// Two elements (one per lane of the float2), each with its own row constants.
template <int MODE, int PK>
__device__ __forceinline__ Elem element(float2 z, float2 m, float2 kappa, float2 beta, int p) {
    constexpr float kLn2 = 0.6931471805599453f;
    Elem r;
    float2 b;
    if constexpr (MODE == kSoftmax || MODE == kSoftmaxRw) {
        const float2 e = __fadd2_rn(z, make_float2(-m.x, -m.y));
        b = make_float2(ptx::ex2(e.x), ptx::ex2(e.y));
        r.slope = __fmul2_rn(b, make_float2(kLn2, kLn2));
    } else if constexpr (MODE == kSigmoidRw) {
        const float2 e = __fadd2_rn(make_float2(ptx::ex2(-z.x), ptx::ex2(-z.y)), make_float2(1.f, 1.f));
        b = make_float2(ptx::rcp(e.x), ptx::rcp(e.y));
        const float2 omb = __fadd2_rn(make_float2(1.f, 1.f), make_float2(-b.x, -b.y));
        r.slope = __fmul2_rn(__fmul2_rn(b, omb), make_float2(kLn2, kLn2));
    } else {
        // sp2(z) = log2(1 + 2^z); dsp2/dz = 2^(z - sp2(z)), the logistic function
        const float2 e = __fadd2_rn(make_float2(ptx::ex2(z.x), ptx::ex2(z.y)), make_float2(1.f, 1.f));
        b = make_float2(ptx::lg2(e.x), ptx::lg2(e.y));
        const float2 d = __fadd2_rn(z, make_float2(-b.x, -b.y));
        r.slope = make_float2(ptx::ex2(d.x), ptx::ex2(d.y));
    }
    if constexpr (is_reweight(MODE)) {
        // ReLU by a saturating FMA: b kappa + beta never exceeds 1 except by rounding
        const float2 base = ptx::fma_sat2(b, kappa, beta);
        r.u = pow_pm1<PK>(base, p);
        r.w = __fmul2_rn(r.u, base);
    } else {
        r.u = make_float2(1.f, 1.f);
        r.w = b;
    }
    return r;
}

// LSSAR on a row whose one-exponential bound holds (for p and p - 1): the
// weight's softplus as z + e / ln 2 with e = 2^-|z| (the forward's weight
// pass does the same on such rows), and the exact logistic slope from the
// same exponential, phi'(z) = 1 / (1 + e) for z >= 0 and e / (1 + e) below.
// With Slope false the slope is left out (the statistics sweep needs none).
template <int PK, bool Slope>
__device__ __forceinline__ Elem element_fast(float2 z, float2 kappa, float2 beta, float2 ck, int p) {
    Elem r;
    const float2 e = make_float2(ptx::ex2(-fabsf(z.x)), ptx::ex2(-fabsf(z.y)));
    const float2 base = ptx::fma_sat2(e, ck, __ffma2_rn(z, kappa, beta));
    r.u = pow_pm1<PK>(base, p);
    r.w = __fmul2_rn(r.u, base);
    if constexpr (Slope) {
        const float2 e1 = __fadd2_rn(e, make_float2(1.f, 1.f));
        const float2 rc = make_float2(ptx::rcp(e1.x), ptx::rcp(e1.y));
        r.slope = __fmul2_rn(rc, make_float2(z.x >= 0.f ? 1.f : e.x, z.y >= 0.f ? 1.f : e.y));
    } else {
        r.slope = make_float2(0.f, 0.f);
    }
    return r;
}

template <int MODE>
__device__ __forceinline__ uint32_t pack_ds(float lo, float hi) {
    if constexpr (uses_normalised_qk(MODE))
        return ptx::pack_f16x2(lo, hi);
    else
        return ptx::pack_bf16x2(lo, hi);
}

template <int D, int MODE, int PK, int PASS>
__global__ void __launch_bounds__(Tmem<D, PASS>::kThreads, 1)
lssar_bwd_kernel(const __grid_constant__ CUtensorMap tmX1, const __grid_constant__ CUtensorMap tmX2,
                 const __grid_constant__ CUtensorMap tmY1, const __grid_constant__ CUtensorMap tmY2,
                 const Params prm) {
    using C = Cfg<D>;
    using T = Tmem<D, PASS>;
    constexpr int NS = C::kStages;
    constexpr int TB = C::kTB;
    constexpr bool kRaw = !uses_normalised_qk(MODE);
    constexpr bool kRow = PASS == kRowPass;
    // the row pass's LSSAR sweeps have a one-exponential variant (p = 15 and
    // the generic power path; at p = 3 the bound never holds)
    constexpr bool kFastModes = kRow && MODE == kLssar && (PK == 15 || PK == 0);
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base as an offset from the array itself: a pointer
    // rebuilt from an integer would lose the shared address space, and every
    // access through it would compile to a generic load or store
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sX = smem;
    uint8_t *ring = smem + C::kRingOff;
    Barriers *bars = reinterpret_cast<Barriers *>(smem + C::kBarOff);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    // S = X1 Y1^T (score operands' type), dP = X2 Y2^T (bf16), M = N = 128
    constexpr uint32_t kIdescS = ptx::idesc_f16(kRaw, kBM, kBN, false, false);
    constexpr uint32_t kIdescDP = ptx::idesc_f16(true, kBM, kBN, false, false);
    // Acc1 += A1 Y1 (A1 from TMEM, Y1 MN-major), Acc2 += A2 Y2 (bf16)
    constexpr uint32_t kIdescA1 = ptx::idesc_f16(kRaw, kBM, D, false, true);
    constexpr uint32_t kIdescA2 = ptx::idesc_f16(true, kBM, D, false, true);

    if (threadIdx.x == 0) {
        ptx::mbar_init(ptx::smem_u32(&bars->x_full), 1);
        ptx::mbar_init(ptx::smem_u32(&bars->x_empty), 1);
        for (int s = 0; s < NS; ++s) {
            ptx::mbar_init(ptx::smem_u32(&bars->ring_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->ring_empty[s]), T::kIssuers);   // one commit per issuer
        }
        ptx::mbar_init(ptx::smem_u32(&bars->s_full), 1);
        ptx::mbar_init(ptx::smem_u32(&bars->s_free), kMathThreads);
        ptx::mbar_init(ptx::smem_u32(&bars->a_full), kMathThreads);
        ptx::mbar_init(ptx::smem_u32(&bars->a_free), 1);
        ptx::mbar_init(ptx::smem_u32(&bars->acc_full), 1);
        ptx::mbar_init(ptx::smem_u32(&bars->acc_free), kMathThreads);
        ptx::mbar_init(ptx::smem_u32(&bars->red), kMathThreads);
        ptx::mbar_init(ptx::smem_u32(&bars->fin), kMathThreads);
        for (int s = 0; s < kItemQ; ++s) {
            ptx::mbar_init(ptx::smem_u32(&bars->item_full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&bars->item_empty[s]), T::kItemConsumers);
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
    // The launch may overlap the kernel before it (a programmatic dependent
    // launch): everything above is local setup; what earlier work wrote (the
    // normalised rows, the zeroed counters, the row pass's records) is read
    // only after this.  The row pass then lets the column pass launch: its
    // CTAs take an SM as this pass's CTAs leave, and wait here in turn.
    ptx::grid_dependency_wait();
    if constexpr (kRow) ptx::launch_dependents();

    const int BH = prm.BH;
    // item -> head, anchor tile, partner tiles [p0, p1); longest items first
    auto decode = [&](int item, int &bh, int &at, int &p0, int &p1) {
        bh = item % BH;
        if (kRow) {
            at = prm.n_tiles - 1 - item / BH;
            p0 = 0;
            p1 = at + 1;
        } else {
            at = item / BH;
            p0 = at;
            p1 = prm.n_tiles;
        }
    };
    auto next_item = [&](uint32_t &qi, int &item, bool arrive = true) -> bool {
        const uint32_t s = qi % kItemQ, use = qi / kItemQ;
        ++qi;
        if (!wait_bar(ptx::smem_u32(&bars->item_full[s]), use & 1, bars, prm.err, kErrItem))
            return false;
        item = *(volatile int *)&bars->item_q[s];
        if (arrive) ptx::mbar_arrive(ptx::smem_u32(&bars->item_empty[s]));
        return true;
    };
    // A wait taken by every lane of a control warp; the outcome is made
    // warp-uniform so that the warp's control flow never diverges.
    auto wait_all = [&](uint32_t bar, uint32_t parity, unsigned code) -> bool {
        return __all_sync(0xffffffffu, wait_bar(bar, parity, bars, prm.err, code));
    };
    constexpr int kPasses = kRow ? 2 : 1;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // (the whole warp runs the loop; one elected lane issues the copies)
        {
            if (ptx::elect_one()) {
                ptx::prefetch_tensormap(&tmX1);
                ptx::prefetch_tensormap(&tmX2);
                ptx::prefetch_tensormap(&tmY1);
                ptx::prefetch_tensormap(&tmY2);
            }
            uint32_t ring_idx = 0, x_cnt = 0, qi = 0;
            bool ok = true;
            while (ok) {
                const uint32_t s = qi % kItemQ, use = qi / kItemQ;
                int item = (int)blockIdx.x;
                if (qi > 0) {
                    if (lane == 0) item = (int)(gridDim.x + atomicAdd(prm.counter, 1u));
                    item = __shfl_sync(0xffffffffu, item, 0);
                }
                ++qi;
                if (use > 0 && !wait_all(ptx::smem_u32(&bars->item_empty[s]), (use - 1) & 1, kErrItem))
                    break;
                if (lane == 0) {
                    *(volatile int *)&bars->item_q[s] = item;
                    ptx::mbar_arrive(ptx::smem_u32(&bars->item_full[s]));
                }
                __syncwarp();
                if (item >= prm.n_items) break;
                int bh, at, p0, p1;
                decode(item, bh, at, p0, p1);
                if (!dcheck(bh >= 0 && bh < prm.BH && at >= 0 && at < prm.n_tiles && p0 >= 0 && p1 <= prm.n_tiles,
                            prm.err, kDbgItem))
                    break;
                if (x_cnt > 0 && !wait_all(ptx::smem_u32(&bars->x_empty), (x_cnt - 1) & 1, kErrXEmpty))
                    break;
                const uint32_t xf = ptx::smem_u32(&bars->x_full);
                if (ptx::elect_one()) {
                    ptx::mbar_arrive_expect_tx(xf, 2 * TB);
#pragma unroll
                    for (int b = 0; b < D / 64; ++b) {
                        ptx::tma_load_3d(ptx::smem_u32(sX + b * 16384), &tmX1, xf, b * 64, at * kBM, bh);
                        ptx::tma_load_3d(ptx::smem_u32(sX + TB + b * 16384), &tmX2, xf, b * 64, at * kBM, bh);
                    }
                }
                __syncwarp();
                ++x_cnt;
                for (int pass = 0; ok && pass < kPasses; ++pass) {
                    for (int t = p0; ok && t < p1; ++t) {
                        const uint32_t st = ring_idx % NS, su = ring_idx / NS;
                        if (su > 0 && !wait_all(ptx::smem_u32(&bars->ring_empty[st]), (su - 1) & 1,
                                                kErrRingEmpty)) {
                            ok = false;
                            break;
                        }
                        uint8_t *stage = ring + st * C::kStageBytes;
                        const uint32_t full = ptx::smem_u32(&bars->ring_full[st]);
                        // streamed tile and its records inside their tensors
                        const bool in_range = dcheck(t >= 0 && t < prm.n_tiles, prm.err, kDbgTma);
                        if (in_range && ptx::elect_one()) {
                            ptx::mbar_arrive_expect_tx(full, 2 * TB + (kRow ? 0 : C::kConstBytes));
#pragma unroll
                            for (int b = 0; b < D / 64; ++b) {
                                ptx::tma_load_3d(ptx::smem_u32(stage + b * 16384), &tmY1, full, b * 64,
                                                 t * kBN, bh);
                                ptx::tma_load_3d(ptx::smem_u32(stage + TB + b * 16384), &tmY2, full, b * 64,
                                                 t * kBN, bh);
                            }
                            if (!kRow)
                                ptx::bulk_load(ptx::smem_u32(stage + 2 * TB),
                                               prm.rowc + ((size_t)bh * prm.n_tiles + t) * 8 * kBN,
                                               C::kConstBytes, full);
                        }
                        __syncwarp();
                        ++ring_idx;
                    }
                }
            }
            // No copy may be in flight when the CTA ends, also after an abort:
            // wait (bounded) until the last stages and anchor tiles issued have landed.
            for (uint32_t i = ring_idx > (uint32_t)NS ? ring_idx - NS : 0; i < ring_idx; ++i)
                wait_bar(ptx::smem_u32(&bars->ring_full[i % NS]), (i / NS) & 1, bars, prm.err, kErrDrain, false);
            if (x_cnt > 0)
                wait_bar(ptx::smem_u32(&bars->x_full), (x_cnt - 1) & 1, bars, prm.err, kErrDrain, false);
        }
        __syncwarp();
    } else if (warp == 1 || (T::kIssuers == 2 && warp == kAccWarp)) {
        // ------------------------------------------------------------ MMA issuers
        // With two issuers, warp 1 issues S and dP of every partner tile and
        // warp kAccWarp the accumulations, so the two chains of waits and issues
        // overlap; both walk the whole stage sequence and commit every stage's
        // release (a stage is free after one commit per issuer).  With one
        // issuer, warp 1 issues everything in one order.  The whole warp runs
        // the loop; one elected lane issues the MMAs and commits.
        const bool do_scores = warp == 1;
        {
            uint32_t ring_idx = 0, x_cnt = 0, qi = 0;
            uint32_t sf_phase = 0, af_phase = 0, accf_phase = 0;
            bool s_pending = false, acc_pending = false;
            bool ok = true;
            auto acquire = [&](uint32_t &slot) -> bool {
                slot = ring_idx % NS;
                const uint32_t use = ring_idx / NS;
                ++ring_idx;
                if (!wait_all(ptx::smem_u32(&bars->ring_full[slot]), use & 1, kErrRingFull)) return false;
                ptx::tc_fence_after();
                return true;
            };
            auto commit = [&](uint64_t *bar) {
                const uint32_t b = ptx::smem_u32(bar);
                if (ptx::elect_one()) ptx::mma_commit(b);
                __syncwarp();
            };
            auto touch_s = [&]() -> bool {
                if (!s_pending) return true;
                if (!wait_all(ptx::smem_u32(&bars->s_free), sf_phase, kErrSFree)) return false;
                sf_phase ^= 1;
                s_pending = false;
                ptx::tc_fence_after();
                return true;
            };
            const uint64_t dx1 = ptx::smem_desc_sw128(ptx::smem_u32(sX), kKmajorLbo, kKmajorSbo);
            const uint64_t dx2 = ptx::smem_desc_sw128(ptx::smem_u32(sX + TB), kKmajorLbo, kKmajorSbo);
            const uint64_t dy0 = ptx::smem_desc_sw128(ptx::smem_u32(ring), kKmajorLbo, kKmajorSbo);
            const uint64_t dm0 = ptx::smem_desc_sw128(ptx::smem_u32(ring), kMnLbo, kMnSbo);
            // S and dP of the partner tile in `slot`
            auto issue_scores = [&](uint32_t slot) {
                const uint64_t y1 = dy0 + (uint64_t)((slot * C::kStageBytes) >> 4);
                const uint64_t y2 = dy0 + (uint64_t)((slot * C::kStageBytes + TB) >> 4);
                const uint32_t full = ptx::smem_u32(&bars->s_full);
                if (ptx::elect_one()) {
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = ((k / 4) * 16384 + (k % 4) * 32) >> 4;
                        ptx::mma_ss(tmem + T::kS, dx1 + off, y1 + off, kIdescS, k > 0);
                    }
#pragma unroll
                    for (int k = 0; k < D / 16; ++k) {
                        const uint32_t off = ((k / 4) * 16384 + (k % 4) * 32) >> 4;
                        ptx::mma_ss(tmem + T::kDP, dx2 + off, y2 + off, kIdescDP, k > 0);
                    }
                    ptx::mma_commit(full);
                }
                __syncwarp();
                // with the A operands over S / dP the warpgroups signal a_full only
                s_pending = !T::kAlias;
            };
            // A operand words of partner columns 16k..16k+15
            auto a_addr = [&](uint32_t base, int k) -> uint32_t {
                return T::kAlias ? tmem + base + 32 * (k / 2) + 8 * (k % 2) : tmem + base + 8 * k;
            };
            auto issue_acc = [&](uint32_t slot, bool accumulate) {
                const uint64_t m1 = dm0 + (uint64_t)((slot * C::kStageBytes) >> 4);
                const uint64_t m2 = dm0 + (uint64_t)((slot * C::kStageBytes + TB) >> 4);
                if (ptx::elect_one()) {
#pragma unroll
                    for (int k = 0; k < kBN / 16; ++k)
                        ptx::mma_ts(tmem + T::kAcc1, a_addr(T::kA1, k), m1 + (uint64_t)((k * 2048) >> 4),
                                    kIdescA1, (accumulate || k > 0) ? 1u : 0u);
                    if (!kRow) {
#pragma unroll
                        for (int k = 0; k < kBN / 16; ++k)
                            ptx::mma_ts(tmem + T::kAcc2, a_addr(T::kA2, k), m2 + (uint64_t)((k * 2048) >> 4),
                                        kIdescA2, (accumulate || k > 0) ? 1u : 0u);
                    }
                }
                __syncwarp();
            };
            int item;
            while (ok && (ok = __all_sync(0xffffffffu, next_item(qi, item, lane == 0))) && item < prm.n_items) {
                int bh, at, p0, p1;
                decode(item, bh, at, p0, p1);
                const int n = p1 - p0;
                uint32_t slot;
                if constexpr (T::kIssuers == 2) {
                    if (do_scores) {
                        if (!(ok = wait_all(ptx::smem_u32(&bars->x_full), x_cnt & 1, kErrXFull))) break;
                        ++x_cnt;
                        ptx::tc_fence_after();
                        // row pass: the statistics sweep, then the accumulation sweep
                        for (int sweep = 0; ok && sweep < kPasses; ++sweep)
                            for (int t = 0; t < n; ++t) {
                                if (!(ok = acquire(slot)) || !(ok = touch_s())) break;
                                issue_scores(slot);
                                commit(&bars->ring_empty[slot]);
                            }
                        if (!ok) break;
                        commit(&bars->x_empty);
                    } else {
                        if (kRow)   // the statistics sweep's stages: released as they arrive
                            for (int t = 0; ok && t < n; ++t) {
                                if (!(ok = acquire(slot))) break;
                                commit(&bars->ring_empty[slot]);
                            }
                        for (int t = 0; ok && t < n; ++t) {
                            if (!(ok = acquire(slot))) break;
                            if (!(ok = wait_all(ptx::smem_u32(&bars->a_full), af_phase, kErrAFull))) break;
                            af_phase ^= 1;
                            ptx::tc_fence_after();
                            if (t == 0 && acc_pending) {
                                if (!(ok = wait_all(ptx::smem_u32(&bars->acc_free), accf_phase, kErrAccFree))) break;
                                accf_phase ^= 1;
                                acc_pending = false;
                                ptx::tc_fence_after();
                            }
                            issue_acc(slot, t > 0);
                            commit(&bars->a_free);
                            commit(&bars->ring_empty[slot]);
                        }
                        if (!ok) break;
                        commit(&bars->acc_full);
                        acc_pending = true;
                    }
                    continue;
                }
                if (!(ok = wait_all(ptx::smem_u32(&bars->x_full), x_cnt & 1, kErrXFull))) break;
                ++x_cnt;
                ptx::tc_fence_after();
                if (kRow) {
                    // pass 1: scores only
                    for (int t = 0; ok && t < n; ++t) {
                        if (!(ok = acquire(slot)) || !(ok = touch_s())) break;
                        issue_scores(slot);
                        commit(&bars->ring_empty[slot]);
                    }
                    if (!ok) break;
                }
                // accumulation pass
                uint32_t cur;
                if (!(ok = acquire(cur)) || !(ok = touch_s())) break;
                issue_scores(cur);
                for (int t = 0; ok && t < n; ++t) {
                    const bool has_next = t + 1 < n;
                    uint32_t nxt = 0;
                    if (!T::kAlias && has_next) {
                        // next scores as soon as the warpgroups have loaded these
                        if (!(ok = acquire(nxt)) || !(ok = touch_s())) break;
                        issue_scores(nxt);
                    }
                    if (!(ok = wait_all(ptx::smem_u32(&bars->a_full), af_phase, kErrAFull))) break;
                    af_phase ^= 1;
                    ptx::tc_fence_after();
                    if (t == 0 && acc_pending) {
                        if (!(ok = wait_all(ptx::smem_u32(&bars->acc_free), accf_phase, kErrAccFree))) break;
                        accf_phase ^= 1;
                        acc_pending = false;
                        ptx::tc_fence_after();
                    }
                    issue_acc(cur, t > 0);
                    commit(&bars->a_free);
                    commit(&bars->ring_empty[cur]);
                    if (T::kAlias && has_next) {
                        // A was written over S / dP: the next scores follow the
                        // accumulation in issue order
                        if (!(ok = acquire(nxt))) break;
                        issue_scores(nxt);
                    }
                    cur = nxt;
                }
                if (!ok) break;
                commit(&bars->acc_full);
                commit(&bars->x_empty);
                acc_pending = true;
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ math warpgroups
        const int g = (warp - kMathWarp0) >> 2;
        const int t = (warp & 3) * 32 + lane;            // anchor row within the tile = TMEM lane
        const uint32_t lane_addr = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t s_col = tmem + lane_addr + T::kS + 32 * g;
        const uint32_t dp_col = tmem + lane_addr + T::kDP + 32 * g;
        const uint32_t a1_col = tmem + lane_addr + (T::kAlias ? T::kS + 32 * g : T::kA1 + 16 * g);
        const uint32_t a2_col = tmem + lane_addr + (T::kAlias ? T::kDP + 32 * g : T::kA2 + 16 * g);
        const uint32_t acc1_col = tmem + lane_addr + T::kAcc1 + g * (D / 4);
        const uint32_t acc2_col = tmem + lane_addr + T::kAcc2 + g * (D / 4);
        dcheck(tmem_in_range(s_col, tmem, 32, 512) && tmem_in_range(dp_col, tmem, 32, 512) &&
                   tmem_in_range(a1_col, tmem, 16, 512) && tmem_in_range(a2_col, tmem, 16, 512) &&
                   tmem_in_range(acc1_col, tmem, D / 4, 512) && tmem_in_range(acc2_col, tmem, D / 4, 512),
               prm.err, kDbgTmem);
        const uint32_t s_full = ptx::smem_u32(&bars->s_full), s_free = ptx::smem_u32(&bars->s_free);
        const uint32_t a_full = ptx::smem_u32(&bars->a_full), a_free = ptx::smem_u32(&bars->a_free);
        uint32_t sf_phase = 0, af_phase = 0, accf_phase = 0, red_phase = 0, fin_phase = 0, qi = 0, ring_idx = 0;
        bool a_pending = false;
        const float log2e = 1.4426950408889634f;
        int pe = is_reweight(MODE) ? prm.p : 1;   // this item's exponent (per head when asked)
        auto wait_warp = [&](uint32_t bar, uint32_t parity, unsigned code) -> bool {
            const bool mine = wait_bar(bar, parity, bars, prm.err, code);
            return __all_sync(0xffffffffu, mine);
        };
        // S and dP of this thread's 32 columns into registers
        auto load_scores = [&](uint32_t (&rs)[32], uint32_t (&rd)[32]) -> bool {
            if (!wait_warp(s_full, sf_phase, kErrSFull)) return false;
            sf_phase ^= 1;
            ptx::tc_fence_after();
            ptx::tmem_ld32(s_col, rs);
            ptx::tmem_ld32(dp_col, rd);
            ptx::tmem_ld_wait();
            ptx::reg_fence(rs);
            ptx::reg_fence(rd);
            if (!T::kAlias) {
                ptx::tc_fence_before();
                ptx::mbar_arrive(s_free);
            }
            return true;
        };
        // A operand words into TMEM, then signal the MMA thread
        auto store_a = [&](const uint32_t (&w1)[16], const uint32_t (&w2)[16]) -> bool {
            if (!T::kAlias && a_pending) {
                if (!wait_warp(a_free, af_phase, kErrAFree)) return false;
                af_phase ^= 1;
                ptx::tc_fence_after();
            }
            ptx::tmem_st16(a1_col, w1);
            if (!kRow) ptx::tmem_st16(a2_col, w2);
            ptx::tmem_st_wait();
            ptx::tc_fence_before();
            ptx::mbar_arrive(a_full);
            a_pending = true;
            return true;
        };
        // The gradient of the L2 row normalisation x -> x / max(|x|, 1e-12)
        // of this thread's anchor row (q in the row pass, k in the column
        // pass), from gv, this warpgroup's D/4 columns of the gradient with
        // respect to the normalised row: y = (g - x (x.g) / |x|^2) / |x| for
        // |x| > 1e-12 (else g / 1e-12) in the normalised modes, y = g in the
        // softmax modes.  |x|^2 and x.g span the whole row, whose columns lie
        // in the four warpgroups, so their partial sums meet in shared memory
        // at a bounded mbarrier (every math thread arrives, also past L).
        auto finish_row = [&](const float (&gv)[D / 4], int bh, int arow, bool valid) -> bool {
            constexpr int Q = D / 4;
            const size_t off = ((size_t)bh * prm.L + arow) * D + g * Q;
            const bool live = valid && dcheck(bh < prm.BH && arow < prm.L, prm.err, kDbgGlobal);
            float y[Q];
            if constexpr (uses_normalised_qk(MODE)) {
                float xv[Q];
                float ss = 0.f, dot = 0.f;
#pragma unroll
                for (int c = 0; c < Q / 8; ++c) {
                    uint4 u = make_uint4(0u, 0u, 0u, 0u);
                    if (live) u = *reinterpret_cast<const uint4 *>(prm.xraw + off + 8 * c);
                    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = __bfloat1622float2(h[e]);
                        xv[8 * c + 2 * e] = f.x;
                        xv[8 * c + 2 * e + 1] = f.y;
                    }
                }
#pragma unroll
                for (int e = 0; e < Q; ++e) {
                    ss = fmaf(xv[e], xv[e], ss);
                    dot = fmaf(xv[e], gv[e], dot);
                }
                bars->x_fin[0][g][t] = ss;
                bars->x_fin[1][g][t] = dot;
                ptx::mbar_arrive(ptx::smem_u32(&bars->fin));
                if (!wait_warp(ptx::smem_u32(&bars->fin), fin_phase, kErrFin)) return false;
                fin_phase ^= 1;
                ss = (bars->x_fin[0][0][t] + bars->x_fin[0][1][t]) + (bars->x_fin[0][2][t] + bars->x_fin[0][3][t]);
                dot = (bars->x_fin[1][0][t] + bars->x_fin[1][1][t]) + (bars->x_fin[1][2][t] + bars->x_fin[1][3][t]);
                const float n = sqrtf(ss);
                if (n > 1e-12f) {
                    const float inv = 1.f / n, radial = dot * inv * inv;
#pragma unroll
                    for (int e = 0; e < Q; ++e) y[e] = (gv[e] - xv[e] * radial) * inv;
                } else {
#pragma unroll
                    for (int e = 0; e < Q; ++e) y[e] = gv[e] * 1e12f;
                }
            } else {
#pragma unroll
                for (int e = 0; e < Q; ++e) y[e] = gv[e];
            }
            if (live) {
#pragma unroll
                for (int c = 0; c < Q / 8; ++c) {
                    uint4 u;
                    u.x = ptx::pack_bf16x2(y[8 * c], y[8 * c + 1]);
                    u.y = ptx::pack_bf16x2(y[8 * c + 2], y[8 * c + 3]);
                    u.z = ptx::pack_bf16x2(y[8 * c + 4], y[8 * c + 5]);
                    u.w = ptx::pack_bf16x2(y[8 * c + 6], y[8 * c + 7]);
                    *reinterpret_cast<uint4 *>(prm.grad + off + 8 * c) = u;
                }
            }
            return true;
        };
        bool ok = true;
        int item;
        while (ok) {
            ok = __all_sync(0xffffffffu, next_item(qi, item));
            if (!ok || item >= prm.n_items) break;
            int bh, at, p0, p1;
            decode(item, bh, at, p0, p1);
            if (is_reweight(MODE) && PK == 0 && prm.per_head) pe = prm.p_head[bh % prm.H];
            const int arow = at * kBM + t;                // anchor row (query or key)
            const bool valid = arow < prm.L;
            if (kRow) {
                // ---------------- row pass: query row arow, key tiles 0..at
                float4 st = make_float4(0.f, 0.f, 0.f, 1.f);
                if (valid) st = prm.stats[(size_t)bh * prm.L + arow];
                const float fi = (float)(arow + 1);
                const float a = !valid ? 0.f : (kRaw ? log2e * rsqrtf((float)D) : log2e * prm.ln_d * logf(fi));
                const float F = (float)pe * st.y / st.w;
                const float2 mm = make_float2(st.x, st.x), kk = make_float2(st.y, st.y), bb = make_float2(st.z, st.z);
                // LSSAR rows whose one-exponential bound holds for p and p - 1
                // (threshold theta = -beta / kappa) take the forward's
                // one-exponential weights; the choice is warp-uniform
                bool fastw = false;
                float2 ck = make_float2(0.f, 0.f);
                if constexpr (kFastModes) {
                    const bool mine = !valid || (st.y > 0.f && fast_weights_ok(-st.z / st.y, st.y, fi, pe) &&
                                                 fast_weights_ok(-st.z / st.y, st.y, fi, pe - 1));
                    fastw = !prm.exact_weights && __all_sync(0xffffffffu, mine);
                    ck = make_float2(2.f * kHalfInvLn2 * st.y, 2.f * kHalfInvLn2 * st.y);
                }
                float2 e_acc = make_float2(0.f, 0.f), du_acc = make_float2(0.f, 0.f), u_acc = make_float2(0.f, 0.f);
                float dmax = -INFINITY, dmin = INFINITY;
                auto stats_tile = [&](const uint32_t (&rs)[32], const uint32_t (&rd)[32], auto diag, auto fast) {
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const float2 z = score_z<MODE>(rs[c], rs[c + 1], a);
                        float2 dP = make_float2(__uint_as_float(rd[c]), __uint_as_float(rd[c + 1]));
                        Elem el;
                        if constexpr (decltype(fast)::value) el = element_fast<PK, false>(z, kk, bb, ck, pe);
                        else el = element<MODE, PK>(z, mm, kk, bb, pe);
                        float2 lo = dP, hi = dP;
                        if constexpr (decltype(diag)::value) {
                            if (32 * g + c > t) { el.w.x = 0.f; el.u.x = 0.f; lo.x = INFINITY; hi.x = -INFINITY; }
                            if (32 * g + c + 1 > t) { el.w.y = 0.f; el.u.y = 0.f; lo.y = INFINITY; hi.y = -INFINITY; }
                        }
                        e_acc = __ffma2_rn(el.w, dP, e_acc);
                        du_acc = __ffma2_rn(el.u, dP, du_acc);
                        u_acc = __fadd2_rn(u_acc, el.u);
                        dmax = max3(dmax, hi.x, hi.y);
                        dmin = min3(dmin, lo.x, lo.y);
                    }
                };
                for (int kt = p0; kt < p1; ++kt) {
                    uint32_t rs[32], rd[32];
                    if (!(ok = load_scores(rs, rd))) break;
                    if (kt == at) stats_tile(rs, rd, Diag(), Exact());
                    else if (kFastModes && fastw) stats_tile(rs, rd, OffDiag(), Fast());
                    else stats_tile(rs, rd, OffDiag(), Exact());
                }
                if (!ok) break;
                bars->x_red[0][g][t] = e_acc.x + e_acc.y;
                bars->x_red[1][g][t] = du_acc.x + du_acc.y;
                bars->x_red[2][g][t] = u_acc.x + u_acc.y;
                bars->x_red[3][g][t] = dmax;
                bars->x_red[4][g][t] = dmin;
                ptx::mbar_arrive(ptx::smem_u32(&bars->red));
                if (!(ok = wait_warp(ptx::smem_u32(&bars->red), red_phase, kErrRed))) break;
                red_phase ^= 1;
                float esum = 0.f, dusum = 0.f, usum = 0.f, mx = -INFINITY, mn = INFINITY;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    esum += bars->x_red[0][h][t];
                    dusum += bars->x_red[1][h][t];
                    usum += bars->x_red[2][h][t];
                    mx = fmaxf(mx, bars->x_red[3][h][t]);
                    mn = fminf(mn, bars->x_red[4][h][t]);
                }
                const float Di = esum / st.w;
                const float o = (is_reweight(MODE) && arow >= 3) ? 1.f : 0.f;
                const float dS1 = -(o / fi) * F * (dusum - Di * usum);
                const float dev = fmaxf(mx - Di, Di - mn);
                float r = a * (F * dev + fabsf(dS1));
                if (!(r > 0.f) || !valid) r = 1.f;
                const float Fp = a * F / r, dS1p = a * dS1 / r;
                if (g == 0) {
                    // the column pass's record of this query, field-major per tile
                    // (all zero past L: no contribution)
                    // normalised modes: the column pass multiplies by the scaled
                    // query rows a_i qh_i, so its ds omits a_i (dscale = 1)
                    const float dscale = kRaw ? a : 1.f;
                    const float fld[8] = {a, st.x, st.y, st.z, 1.f / st.w, dscale * F, Di, dscale * dS1};
                    float *rec = prm.rowc + ((size_t)bh * prm.n_tiles + at) * 8 * kBN + t;
                    if (dcheck(bh < prm.BH && at < prm.n_tiles && t < kBN, prm.err, kDbgGlobal))
#pragma unroll
                        for (int k = 0; k < 8; ++k) rec[k * kBN] = valid ? fld[k] : 0.f;
                    if (valid) atomicMax(prm.rmax + bh, __float_as_uint(dscale * (F * dev + fabsf(dS1))));
                }
                // pass 2: ds / r into TMEM, dqh accumulates in Acc1
                auto ds_tile = [&](const uint32_t (&rs)[32], const uint32_t (&rd)[32], uint32_t (&w1)[16],
                                   auto diag, auto fast) {
#pragma unroll
                    for (int c = 0; c < 32; c += 2) {
                        const float2 z = score_z<MODE>(rs[c], rs[c + 1], a);
                        const float2 dP = make_float2(__uint_as_float(rd[c]), __uint_as_float(rd[c + 1]));
                        Elem el;
                        if constexpr (decltype(fast)::value) el = element_fast<PK, true>(z, kk, bb, ck, pe);
                        else el = element<MODE, PK>(z, mm, kk, bb, pe);
                        const float2 dd = __fadd2_rn(dP, make_float2(-Di, -Di));
                        const float2 gg = __ffma2_rn(__fmul2_rn(dd, el.u), make_float2(Fp, Fp), make_float2(dS1p, dS1p));
                        float2 ds = __fmul2_rn(gg, el.slope);
                        if constexpr (decltype(diag)::value) {
                            if (32 * g + c > t) ds.x = 0.f;
                            if (32 * g + c + 1 > t) ds.y = 0.f;
                        }
                        w1[c / 2] = pack_ds<MODE>(ds.x, ds.y);
                    }
                };
                for (int kt = p0; kt < p1; ++kt) {
                    uint32_t rs[32], rd[32];
                    if (!(ok = load_scores(rs, rd))) break;
                    uint32_t w1[16];
                    if (kt == at) ds_tile(rs, rd, w1, Diag(), Exact());
                    else if (kFastModes && fastw) ds_tile(rs, rd, w1, OffDiag(), Fast());
                    else ds_tile(rs, rd, w1, OffDiag(), Exact());
                    if (!(ok = store_a(w1, w1))) break;
                }
                if (!ok) break;
                // epilogue: dq from dqh = r * Acc1, this warpgroup's D/4 columns
                if (!(ok = wait_warp(ptx::smem_u32(&bars->acc_full), accf_phase, kErrAccFull))) break;
                accf_phase ^= 1;
                ptx::tc_fence_after();
                uint32_t acc[D / 4];
                if constexpr (D == 64) {
                    ptx::tmem_ld16(acc1_col, acc);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence(acc);
                } else {
                    ptx::tmem_ld32(acc1_col, acc);
                    ptx::tmem_ld_wait();
                    ptx::reg_fence(acc);
                }
                ptx::tc_fence_before();
                ptx::mbar_arrive(ptx::smem_u32(&bars->acc_free));
                float gv[D / 4];
#pragma unroll
                for (int e = 0; e < D / 4; ++e) gv[e] = __uint_as_float(acc[e]) * r;
                if (!(ok = finish_row(gv, bh, arow, valid))) break;
            } else {
                // ---------------- column pass: key row arow, query tiles at..n_tiles-1
                const float R = __uint_as_float(prm.rmax[bh]);
                const float invR = R > 0.f ? 1.f / R : 0.f;
                // rec: shared address of this tile's query records, field-major
                // ([field][128 queries]).
                // A warpgroup's 32 columns go in two 16-column halves.
                auto col_half = [&](const uint32_t (&rs)[16], const uint32_t (&rd)[16], uint32_t rec,
                                    int col0, uint32_t (&w1)[8], uint32_t (&w2)[8], auto diag) {
#pragma unroll
                    for (int c = 0; c < 16; c += 4) {
                        const int q0 = col0 + c;
                        float4 f[8];
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            if (k > 1 || kRaw)   // a and m: softmax normalisers only
                                f[k] = ptx::ld_shared_v4(rec + 4u * (k * kBN + q0));
                        // fields: 0 a, 1 m, 2 kappa, 3 beta, 4 1/W, 5 s F, 6 D, 7 s dS1, with
                        // s = a for the softmax normalisers and 1 for the normalised modes
                        // (their query operand carries a_i)
#pragma unroll
                        for (int h = 0; h < 2; ++h) {
                            auto pick = [&](int k) {
                                return h == 0 ? make_float2(f[k].x, f[k].y) : make_float2(f[k].z, f[k].w);
                            };
                            const int cc = c + 2 * h;
                            const float2 z = kRaw ? __fmul2_rn(make_float2(__uint_as_float(rs[cc]),
                                                                           __uint_as_float(rs[cc + 1])), pick(0))
                                                  : make_float2(__uint_as_float(rs[cc]), __uint_as_float(rs[cc + 1]));
                            const float2 dP = make_float2(__uint_as_float(rd[cc]), __uint_as_float(rd[cc + 1]));
                            const float2 mcol = (MODE == kSoftmax || MODE == kSoftmaxRw) ? pick(1) : make_float2(0.f, 0.f);
                            const Elem el = element<MODE, PK>(z, mcol, pick(2), pick(3), pe);
                            float2 P = __fmul2_rn(el.w, pick(4));
                            const float2 dcol = pick(6);
                            const float2 dd = __fadd2_rn(dP, make_float2(-dcol.x, -dcol.y));
                            const float2 gg = __ffma2_rn(__fmul2_rn(dd, el.u), pick(5), pick(7));
                            float2 ds = __fmul2_rn(__fmul2_rn(gg, el.slope), make_float2(invR, invR));
                            if constexpr (decltype(diag)::value) {
                                if (q0 + 2 * h < t) { P.x = 0.f; ds.x = 0.f; }
                                if (q0 + 2 * h + 1 < t) { P.y = 0.f; ds.y = 0.f; }
                            }
                            w1[cc / 2] = pack_ds<MODE>(ds.x, ds.y);
                            w2[cc / 2] = ptx::pack_bf16x2(P.x, P.y);
                        }
                    }
                };
                for (int qt = p0; qt < p1; ++qt) {
                    if (!(ok = wait_warp(s_full, sf_phase, kErrSFull))) break;
                    sf_phase ^= 1;
                    ptx::tc_fence_after();
                    // this tile's query records (the stage's bulk copy has landed:
                    // its mbarrier phase is complete once S was issued)
                    const uint32_t slot = ring_idx % NS, use = ring_idx / NS;
                    ++ring_idx;
                    if (!(ok = wait_warp(ptx::smem_u32(&bars->ring_full[slot]), use & 1, kErrRingFull))) break;
                    const uint32_t rec = ptx::opaque_u32(ptx::smem_u32(ring + slot * C::kStageBytes + 2 * TB));
                    if constexpr (T::kAlias) {
                        // d = 128 (A over S / dP, released by the accumulation):
                        // one 16-column half in registers at a time
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t rs[16], rd[16];
                            ptx::tmem_ld16(s_col + 16 * half, rs);
                            ptx::tmem_ld16(dp_col + 16 * half, rd);
                            ptx::tmem_ld_wait();
                            ptx::reg_fence(rs);
                            ptx::reg_fence(rd);
                            uint32_t w1[8], w2[8];
                            if (qt == at) col_half(rs, rd, rec, 32 * g + 16 * half, w1, w2, Diag());
                            else col_half(rs, rd, rec, 32 * g + 16 * half, w1, w2, OffDiag());
                            // these words overwrite S / dP columns of the first half,
                            // which are already in registers
                            ptx::tmem_st8(a1_col + 8 * half, w1);
                            ptx::tmem_st8(a2_col + 8 * half, w2);
                        }
                    } else {
                        // d = 64: one 16-column half in registers at a time; S / dP
                        // are released once the second half is loaded
                        uint32_t w1[2][8], w2[2][8];
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            uint32_t rsh[16], rdh[16];
                            ptx::tmem_ld16(s_col + 16 * half, rsh);
                            ptx::tmem_ld16(dp_col + 16 * half, rdh);
                            ptx::tmem_ld_wait();
                            ptx::reg_fence(rsh);
                            ptx::reg_fence(rdh);
                            if (half == 1) {
                                ptx::tc_fence_before();
                                ptx::mbar_arrive(s_free);
                            }
                            if (qt == at) col_half(rsh, rdh, rec, 32 * g + 16 * half, w1[half], w2[half], Diag());
                            else col_half(rsh, rdh, rec, 32 * g + 16 * half, w1[half], w2[half], OffDiag());
                        }
                        if (a_pending) {   // the previous tile's A words have been read
                            if (!(ok = wait_warp(a_free, af_phase, kErrAFree))) break;
                            af_phase ^= 1;
                            ptx::tc_fence_after();
                        }
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            ptx::tmem_st8(a1_col + 8 * half, w1[half]);
                            ptx::tmem_st8(a2_col + 8 * half, w2[half]);
                        }
                    }
                    ptx::tmem_st_wait();
                    ptx::tc_fence_before();
                    ptx::mbar_arrive(a_full);
                    a_pending = true;
                }
                if (!ok) break;
                // epilogue: dv = Acc2, and dk from dkh = R * Acc1
                if (!(ok = wait_warp(ptx::smem_u32(&bars->acc_full), accf_phase, kErrAccFull))) break;
                accf_phase ^= 1;
                ptx::tc_fence_after();
                uint32_t acc[D / 4], acc2[D / 4];
                if constexpr (D == 64) {
                    ptx::tmem_ld16(acc1_col, acc);
                    ptx::tmem_ld16(acc2_col, acc2);
                } else {
                    ptx::tmem_ld32(acc1_col, acc);
                    ptx::tmem_ld32(acc2_col, acc2);
                }
                ptx::tmem_ld_wait();
                ptx::reg_fence(acc);
                ptx::reg_fence(acc2);
                ptx::tc_fence_before();
                ptx::mbar_arrive(ptx::smem_u32(&bars->acc_free));
                if (valid && dcheck(bh < prm.BH && arow < prm.L, prm.err, kDbgGlobal)) {
                    const size_t off = ((size_t)bh * prm.L + arow) * D + g * (D / 4);
                    uint4 *dvd = reinterpret_cast<uint4 *>(prm.dv + off);
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        const uint32_t *q8 = &acc2[8 * c];
                        uint4 u;
                        u.x = ptx::pack_bf16x2(__uint_as_float(q8[0]), __uint_as_float(q8[1]));
                        u.y = ptx::pack_bf16x2(__uint_as_float(q8[2]), __uint_as_float(q8[3]));
                        u.z = ptx::pack_bf16x2(__uint_as_float(q8[4]), __uint_as_float(q8[5]));
                        u.w = ptx::pack_bf16x2(__uint_as_float(q8[6]), __uint_as_float(q8[7]));
                        dvd[c] = u;
                    }
                }
                float gv[D / 4];
#pragma unroll
                for (int e = 0; e < D / 4; ++e) gv[e] = __uint_as_float(acc[e]) * R;
                if (!(ok = finish_row(gv, bh, arow, valid))) break;
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

}  // namespace tcb
}  // namespace lssar
