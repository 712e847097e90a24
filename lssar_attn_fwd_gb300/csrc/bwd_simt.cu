// Plain CUDA-core backward pass of causal LSSAR / LSSA / softmax attention.
//
// A second GPU implementation of the gradients, independent of the
// tensor-core backward and used to cross-check it; speed is not a goal.
// fp32 arithmetic with libm transcendentals.
//
// The notes on "Softplus Attention with Re-weighting Boosts Length
// Extrapolation in Large Language Models" train with this attention but give
// no gradient formula; the chain rule through Key designs 1 and 2, in the
// units of the forward kernel (z = a_i s_ij in log2 units), reads for row i:
//   b_ij = phi(z_ij)     sp2(z) = log2(1 + 2^z) | 2^(z - m_i) | 1/(1 + 2^-z)
//   w_ij = max(b kappa_i + beta_i, 0)^p,  W_i = sum_j w_ij  (saved by the forward)
//   dP_ij = dout_i . v_j,  D_i = sum_j (w_ij / W_i) dP_ij  (= dout_i . out_i, taken
//           from the weights so that the bf16 rounding of out does not enter)
//   g_ij = p kappa_i / W_i * (dP_ij - D_i) * max(b kappa_i + beta_i, 0)^(p-1)
//   dS1_i = -(O_i / i) sum_j g_ij          (the threshold theta_i = O_i S1_i / i;
//                                           zero without re-weighting)
//   ds_ij = a_i phi'(z_ij) (g_ij + dS1_i)  (phi' = dphi/dz)
//   dv_j  = sum_i (w_ij / W_i) dout_i
//   dqh_i = sum_j ds_ij kh_j,  dkh_j = sum_i ds_ij qh_i
//   dq_i  = (dqh_i - qh_i (qh_i . dqh_i)) / |q_i|   (normalised modes; the
//                                                   softmax modes use q, k raw)
// The modes without re-weighting are the case p = 1, kappa = 1, beta = 0.
// Scores are formed exactly as the forward forms them (normalised modes: key
// rows scaled by 1/max(|x|, 1e-12), query rows by a_i/max(|x|, 1e-12) with
// a_i = qmul ln i, both rounded to fp16, products summed in fp32 -- the score
// is then z itself; softmax modes: raw bf16 rows), because at large p the
// weights are far more sensitive to a mismatch between the saved row
// constants and the recomputed scores than to the score error itself.
// A uniform (all-zero re-weighted) row is saved as kappa = 0, beta = 1,
// W = i: constant weights 1/i and no gradient through its scores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lssar_internal.cuh"
#include "tc_host.cuh"

namespace lssar {
namespace {

constexpr int kWarpsPerBlock = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float powi(float x, int p) {
    float r = 1.f;
    while (p) {
        if (p & 1) r *= x;
        x *= x;
        p >>= 1;
    }
    return r;
}

// phi(z) and dphi/dz of the mode, z in log2 units.
__device__ __forceinline__ void phi_and_slope(int mode, float z, float m, float &b, float &slope) {
    if (mode == kSoftmax || mode == kSoftmaxRw) {
        b = exp2f(z - m);
        slope = kLn2 * b;
    } else if (mode == kSigmoidRw) {
        b = 1.f / (1.f + exp2f(-z));
        slope = kLn2 * b * (1.f - b);
    } else {
        const float x = z * kLn2;
        b = (fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)))) * kLog2e;   // sp2(z)
        slope = 1.f / (1.f + expf(-x));                            // sigmoid(x)
    }
}

template <int D>
__device__ __forceinline__ void load_row(const __nv_bfloat16 *src, float *dst) {
    const uint4 *r = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        uint4 u = __ldg(r + c);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            dst[8 * c + 2 * e] = f.x;
            dst[8 * c + 2 * e + 1] = f.y;
        }
    }
}

// Dot products of a bf16 row with a row held in shared memory: (x.y, |x|^2).
template <int D>
__device__ __forceinline__ float2 dot_row(const __nv_bfloat16 *x, const float *y) {
    const uint4 *r = reinterpret_cast<const uint4 *>(x);
    float dot = 0.f, ss = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        uint4 u = __ldg(r + c);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            dot = fmaf(f.x, y[8 * c + 2 * e], dot);
            dot = fmaf(f.y, y[8 * c + 2 * e + 1], dot);
            ss = fmaf(f.x, f.x, ss);
            ss = fmaf(f.y, f.y, ss);
        }
    }
    return make_float2(dot, ss);
}

// Score of an fp16-rounded row held in shared memory with a bf16 row
// normalised, multiplied by xscale and rounded the same way:
// (sum_e h(x_e xscale / |x|) y_e, max(|x|, eps)).
template <int D>
__device__ __forceinline__ float2 dot_row_fp16(const __nv_bfloat16 *x, const float *yh, float xscale) {
    const uint4 *r = reinterpret_cast<const uint4 *>(x);
    uint4 u[D / 8];
    float ss = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        u[c] = __ldg(r + c);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u[c]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            ss = fmaf(f.x, f.x, ss);
            ss = fmaf(f.y, f.y, ss);
        }
    }
    const float n = fmaxf(sqrtf(ss), 1e-12f);
    const float inv = (1.f / n) * xscale;
    float dot = 0.f;
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u[c]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            const float2 g = __half22float2(__floats2half2_rn(f.x * inv, f.y * inv));
            dot = fmaf(g.x, yh[8 * c + 2 * e], dot);
            dot = fmaf(g.y, yh[8 * c + 2 * e + 1], dot);
        }
    }
    return make_float2(dot, n);
}

__device__ __forceinline__ float score_scale(int mode, int D, int i) {
    if (!uses_normalised_qk(mode)) return kLog2e * rsqrtf((float)D);
    return kLog2e * logf((float)D) * logf((float)i);
}

// dq of one query row per warp; also saves {D_i, dS1_i} for the key-side kernel.
// Pass 1 over the row's keys gives D_i = sum_j (w_ij / W_i) dP_ij exactly (the
// output itself is not needed) and sum_j g_ij; pass 2 forms ds_ij and dq.
template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bwd_simt_rows(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
              const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ dout,
              const float4 *__restrict__ stats, __nv_bfloat16 *__restrict__ dq,
              float2 *__restrict__ rowws, long long rows_total, int L, int p, int mode, float qmul) {
    __shared__ float sq[kWarpsPerBlock][D];
    __shared__ float sqh[kWarpsPerBlock][D];
    __shared__ float sdo[kWarpsPerBlock][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long g = (long long)blockIdx.x * kWarpsPerBlock + warp;
    if (g >= rows_total) return;
    const long long bh = g / L;
    const int row = (int)(g % L);
    const int i = row + 1;
    const long long qrow = bh * L + row;
    const __nv_bfloat16 *kb = k + bh * (long long)L * D;
    const __nv_bfloat16 *vb = v + bh * (long long)L * D;
    const bool raw = !uses_normalised_qk(mode);

    float qss = 0.f;
    for (int t = lane; t < D; t += 32) {
        const float x = __bfloat162float(q[qrow * D + t]);
        sq[warp][t] = x;
        sdo[warp][t] = __bfloat162float(dout[qrow * D + t]);
        qss = fmaf(x, x, qss);
    }
    qss = warp_sum(qss);
    const float qn = fmaxf(sqrtf(qss), 1e-12f);
    // the forward's query operand: q / max(|q|, eps) * qmul ln i, in fp16
    float qinv = 1.f / qn;
    qinv *= qmul * logf((float)i);
    for (int t = lane; t < D; t += 32) sqh[warp][t] = __half2float(__float2half_rn(sq[warp][t] * qinv));
    __syncwarp();
    const float a = score_scale(mode, D, i);
    const float4 st = stats[qrow];
    const int pe = is_reweight(mode) ? p : 1;
    const float F = (float)pe * st.y / st.w;   // p kappa / W

    // per key j < i: score, phi, slope, u = base^(p-1), w = u base, dP
    auto element = [&](int j, float &slope, float &u, float &w, float &dP, float &kscale) {
        float s;
        if (raw) {
            s = dot_row<D>(kb + (long long)j * D, sq[warp]).x;
            kscale = 1.f;
        } else {
            const float2 sk = dot_row_fp16<D>(kb + (long long)j * D, sqh[warp], 1.f);
            s = sk.x;   // z itself
            kscale = 1.f / sk.y;
        }
        float b;
        phi_and_slope(mode, raw ? a * s : s, st.x, b, slope);
        const float base = fmaxf(b * st.y + st.z, 0.f);
        u = pe == 1 ? (base > 0.f ? 1.f : 0.f) : powi(base, pe - 1);
        w = pe == 1 ? base : u * base;
        dP = dot_row<D>(vb + (long long)j * D, sdo[warp]).x;
    };

    // pass 1: D_i, sum_j dP u, sum_j u
    float e_sum = 0.f, du_sum = 0.f, u_sum = 0.f;
    for (int j = lane; j < i; j += 32) {
        float slope, u, w, dP, ks;
        element(j, slope, u, w, dP, ks);
        e_sum = fmaf(w, dP, e_sum);
        du_sum = fmaf(dP, u, du_sum);
        u_sum += u;
    }
    const float Di = warp_sum(e_sum) / st.w;
    const float gsum = F * (warp_sum(du_sum) - Di * warp_sum(u_sum));
    const float o = (is_reweight(mode) && i > 3) ? 1.f : 0.f;
    const float dS1 = -(o / (float)i) * gsum;

    // pass 2: dqh = sum_j ds_ij kh_j
    float acc[D / 32];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) acc[c] = 0.f;
    for (int j0 = 0; j0 < i; j0 += 32) {
        const int j = j0 + lane;
        float ds = 0.f, kscale = 0.f;
        if (j < i) {
            float slope, u, w, dP;
            element(j, slope, u, w, dP, kscale);
            ds = a * slope * (F * (dP - Di) * u + dS1);
        }
        const int nj = min(32, i - j0);
        for (int t = 0; t < nj; ++t) {
            const float wt = __shfl_sync(0xffffffffu, ds, t) * __shfl_sync(0xffffffffu, kscale, t);
            const __nv_bfloat16 *kr = kb + (long long)(j0 + t) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) acc[c] = fmaf(wt, __bfloat162float(kr[lane + 32 * c]), acc[c]);
        }
    }
    float radial = 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) radial = fmaf(sq[warp][lane + 32 * c] / qn, acc[c], radial);
    radial = warp_sum(radial);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        float r = acc[c];
        if (!raw) r = (qss > 1e-24f) ? (r - sq[warp][lane + 32 * c] / qn * radial) / qn : r / 1e-12f;
        dq[qrow * D + lane + 32 * c] = __float2bfloat16_rn(r);
    }
    if (lane == 0) rowws[qrow] = make_float2(Di, dS1);
}

// dk and dv of one key row per warp.
template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
bwd_simt_cols(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
              const __nv_bfloat16 *__restrict__ v, const __nv_bfloat16 *__restrict__ dout,
              const float4 *__restrict__ stats, const float2 *__restrict__ rowws,
              __nv_bfloat16 *__restrict__ dk, __nv_bfloat16 *__restrict__ dv, long long rows_total,
              int L, int p, int mode, float qmul) {
    __shared__ float sk[kWarpsPerBlock][D];
    __shared__ float skh[kWarpsPerBlock][D];
    __shared__ float sv[kWarpsPerBlock][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long g = (long long)blockIdx.x * kWarpsPerBlock + warp;
    if (g >= rows_total) return;
    const long long bh = g / L;
    const int col = (int)(g % L);
    const long long krow = bh * L + col;
    const __nv_bfloat16 *qb = q + bh * (long long)L * D;
    const __nv_bfloat16 *db = dout + bh * (long long)L * D;
    const bool raw = !uses_normalised_qk(mode);
    const int pe = is_reweight(mode) ? p : 1;

    float kss = 0.f;
    for (int t = lane; t < D; t += 32) {
        const float x = __bfloat162float(k[krow * D + t]);
        sk[warp][t] = x;
        sv[warp][t] = __bfloat162float(v[krow * D + t]);
        kss = fmaf(x, x, kss);
    }
    kss = warp_sum(kss);
    const float kn = fmaxf(sqrtf(kss), 1e-12f);
    for (int t = lane; t < D; t += 32) skh[warp][t] = __half2float(__float2half_rn(sk[warp][t] * (1.f / kn)));
    __syncwarp();

    float dkh[D / 32], dva[D / 32];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) dkh[c] = dva[c] = 0.f;
    for (int i0 = col; i0 < L; i0 += 32) {
        const int r = i0 + lane;   // query row (0-based)
        float pw = 0.f, ds = 0.f, qscale = 0.f;
        if (r < L) {
            const int i = r + 1;
            float s;
            if (raw) {
                s = dot_row<D>(qb + (long long)r * D, sk[warp]).x;
                qscale = 1.f;
            } else {
                const float2 sq = dot_row_fp16<D>(qb + (long long)r * D, skh[warp], qmul * logf((float)(r + 1)));
                s = sq.x;   // z itself
                qscale = 1.f / sq.y;
            }
            const float a = score_scale(mode, D, i);
            const float4 st = stats[bh * L + r];
            const float2 rw = rowws[bh * L + r];
            float b, slope;
            phi_and_slope(mode, raw ? a * s : s, st.x, b, slope);
            const float base = fmaxf(b * st.y + st.z, 0.f);
            const float u = pe == 1 ? (base > 0.f ? 1.f : 0.f) : powi(base, pe - 1);
            const float w = pe == 1 ? base : u * base;
            pw = w / st.w;
            const float dP = dot_row<D>(db + (long long)r * D, sv[warp]).x;
            const float F = (float)pe * st.y / st.w;
            ds = a * slope * (F * (dP - rw.x) * u + rw.y);
        }
        const int ni = min(32, L - i0);
        for (int t = 0; t < ni; ++t) {
            const float w1 = __shfl_sync(0xffffffffu, pw, t);
            const float w2 = __shfl_sync(0xffffffffu, ds, t);
            const float qs = __shfl_sync(0xffffffffu, qscale, t);
            const __nv_bfloat16 *qr = qb + (long long)(i0 + t) * D;
            const __nv_bfloat16 *dr = db + (long long)(i0 + t) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                dva[c] = fmaf(w1, __bfloat162float(dr[lane + 32 * c]), dva[c]);
                dkh[c] = fmaf(w2 * qs, __bfloat162float(qr[lane + 32 * c]), dkh[c]);
            }
        }
    }
    float radial = 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) radial = fmaf(sk[warp][lane + 32 * c] / kn, dkh[c], radial);
    radial = warp_sum(radial);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        float r = dkh[c];
        if (!raw) r = (kss > 1e-24f) ? (r - sk[warp][lane + 32 * c] / kn * radial) / kn : r / 1e-12f;
        dk[krow * D + lane + 32 * c] = __float2bfloat16_rn(r);
        dv[krow * D + lane + 32 * c] = __float2bfloat16_rn(dva[c]);
    }
}

template <int D>
cudaError_t launch(const BwdProblem &pr, void *ws, cudaStream_t stream) {
    const long long rows = (long long)pr.B * pr.H * pr.L;
    const long long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const auto *q = static_cast<const __nv_bfloat16 *>(pr.q);
    const auto *k = static_cast<const __nv_bfloat16 *>(pr.k);
    const auto *v = static_cast<const __nv_bfloat16 *>(pr.v);
    const auto *dout = static_cast<const __nv_bfloat16 *>(pr.dout);
    const auto *st = reinterpret_cast<const float4 *>(pr.stats);
    auto *rowws = static_cast<float2 *>(ws);
    const float qmul = score_qmul(pr.d);
    bwd_simt_rows<D><<<(unsigned)blocks, kWarpsPerBlock * 32, 0, stream>>>(
        q, k, v, dout, st, static_cast<__nv_bfloat16 *>(pr.dq), rowws, rows, pr.L, pr.p, pr.mode, qmul);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    bwd_simt_cols<D><<<(unsigned)blocks, kWarpsPerBlock * 32, 0, stream>>>(
        q, k, v, dout, st, rowws, static_cast<__nv_bfloat16 *>(pr.dk), static_cast<__nv_bfloat16 *>(pr.dv),
        rows, pr.L, pr.p, pr.mode, qmul);
    return cudaGetLastError();
}

}  // namespace

size_t bwd_simt_workspace_bytes(const BwdProblem &pr) {
    return (size_t)pr.B * pr.H * pr.L * sizeof(float2);
}

cudaError_t launch_bwd_simt(const BwdProblem &pr, void *ws, cudaStream_t stream) {
    return pr.d == 64 ? launch<64>(pr, ws, stream) : launch<128>(pr, ws, stream);
}

}  // namespace lssar
