// Plain CUDA-core causal LSSAR / LSSA / softmax attention forward.
//
// One warp per query row, fp32 arithmetic, accurate libm softplus.  It is a
// second GPU implementation of the operation (Key designs 1-2 of the notes on
// "Softplus Attention with Re-weighting Boosts Length Extrapolation in Large
// Language Models"), independent of the tensor-core kernel and used to
// cross-check it.  Speed is not a goal here.
//
// Row i (1-based), keys j <= i:
//   x_ij = ln d ln i * (q_i.k_j) / (|q_i| |k_j|)        (LSSA / LSSAR)
//   x_ij = (q_i.k_j) / sqrt(d)                          (softmax)
//   pass 1: S1_i = sum_j softplus(x_ij), m_i = max_j x_ij
//   pass 2: weights w_ij, S2_i = sum_j w_ij, out_i = sum_j w_ij v_j / S2_i
//     LSSA:    w = softplus(x)
//     LSSAR:   w = max((softplus(x) - theta_i) / (softplus(m_i) - theta_i), 0)^p,
//              theta_i = O_i S1_i / i  (the common factor of the re-weighted row
//              cancels in the final L1 normalisation); a row with
//              softplus(m_i) <= theta_i is the all-zero 0/0 row: w = 1.
//     softmax: w = exp(x - m_i)
//   ablation modes, re-weighting of another normaliser phi (S1 = sum_j phi):
//     softmax normaliser: phi = exp(x - m_i), x = q.k/sqrt(d)
//     sigmoid normaliser: phi = 1/(1 + exp(-x)), x as in LSSA
//     w = max((phi(x) - theta_i) / (phi(m_i) - theta_i), 0)^p
#include <cuda_bf16.h>

#include "lssar_internal.cuh"

namespace lssar {
namespace {

constexpr int kWarpsPerBlock = 8;

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float softplus_libm(float x) {
    return fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
}

__device__ __forceinline__ float sigmoid_libm(float x) {
    return 1.f / (1.f + expf(-x));
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

template <int D>
__global__ void __launch_bounds__(kWarpsPerBlock * 32)
simt_fwd(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
         const __nv_bfloat16 *__restrict__ v, __nv_bfloat16 *__restrict__ out,
         long long rows_total, int L, int p, int mode) {
    __shared__ float sq[kWarpsPerBlock][D];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const long long g = (long long)blockIdx.x * kWarpsPerBlock + warp;
    if (g >= rows_total) return;
    // Longest rows first: within each head, row L-1 is handed out first.
    const long long bh = g / L;
    const int row = L - 1 - (int)(g % L);
    const int i = row + 1;
    const long long qrow = bh * L + row;
    const __nv_bfloat16 *kb = k + bh * (long long)L * D;
    const __nv_bfloat16 *vb = v + bh * (long long)L * D;

    float qss = 0.f;
    for (int t = lane; t < D; t += 32) {
        const float x = __bfloat162float(q[qrow * D + t]);
        sq[warp][t] = x;
        qss = fmaf(x, x, qss);
    }
    qss = warp_sum(qss);
    __syncwarp();
    const bool raw = !uses_normalised_qk(mode);
    const float qscale = raw ? rsqrtf((float)D)
                             : logf((float)D) * logf((float)i) / fmaxf(sqrtf(qss), 1e-12f);

    auto score = [&](int j) -> float {
        const uint4 *kr = reinterpret_cast<const uint4 *>(kb + (long long)j * D);
        float dot = 0.f, kss = 0.f;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
            uint4 u = __ldg(kr + c);
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(h[e]);
                dot = fmaf(f.x, sq[warp][8 * c + 2 * e], dot);
                dot = fmaf(f.y, sq[warp][8 * c + 2 * e + 1], dot);
                kss = fmaf(f.x, f.x, kss);
                kss = fmaf(f.y, f.y, kss);
            }
        }
        if (raw) return dot * qscale;
        return dot * qscale / fmaxf(sqrtf(kss), 1e-12f);
    };

    // Pass 1: row statistics (max, then the sum of the normaliser's values).
    float s1 = 0.f, m = -INFINITY;
    if (mode != kLssa) {
        for (int j = lane; j < i; j += 32) m = fmaxf(m, score(j));
        m = warp_max(m);
    }
    auto phi = [&](float x) -> float {
        if (mode == kSoftmaxRw) return expf(x - m);
        if (mode == kSigmoidRw) return sigmoid_libm(x);
        return softplus_libm(x);
    };
    if (is_reweight(mode)) {
        for (int j = lane; j < i; j += 32) s1 += phi(score(j));
        s1 = warp_sum(s1);
    }
    float theta = 0.f, kappa = 0.f;
    bool degenerate = false;
    if (is_reweight(mode)) {
        const float o = (i <= 3) ? 0.f : 1.f;
        theta = o * s1 / (float)i;
        const float den = phi(m) - theta;
        degenerate = !(den > 0.f);
        kappa = degenerate ? 0.f : 1.f / den;
    }

    // Pass 2: weights and the weighted sum of values.
    float acc[D / 32];
#pragma unroll
    for (int c = 0; c < D / 32; ++c) acc[c] = 0.f;
    float s2 = 0.f;
    for (int j0 = 0; j0 < i; j0 += 32) {
        const int j = j0 + lane;
        float w = 0.f;
        if (j < i) {
            const float x = score(j);
            if (mode == kSoftmax) {
                w = expf(x - m);
            } else if (mode == kLssa) {
                w = softplus_libm(x);
            } else {
                w = degenerate ? 1.f : powi(fmaxf((phi(x) - theta) * kappa, 0.f), p);
            }
        }
        s2 += w;
        const int nj = min(32, i - j0);
        for (int t = 0; t < nj; ++t) {
            const float wt = __shfl_sync(0xffffffffu, w, t);
            const __nv_bfloat16 *vr = vb + (long long)(j0 + t) * D;
#pragma unroll
            for (int c = 0; c < D / 32; ++c) acc[c] = fmaf(wt, __bfloat162float(vr[lane + 32 * c]), acc[c]);
        }
    }
    s2 = warp_sum(s2);
    const float inv = 1.f / s2;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) out[qrow * D + lane + 32 * c] = __float2bfloat16_rn(acc[c] * inv);
}

}  // namespace

cudaError_t launch_simt(const Problem &pr, cudaStream_t stream) {
    const long long rows = (long long)pr.B * pr.H * pr.L;
    const long long blocks = (rows + kWarpsPerBlock - 1) / kWarpsPerBlock;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const auto *q = static_cast<const __nv_bfloat16 *>(pr.q);
    const auto *k = static_cast<const __nv_bfloat16 *>(pr.k);
    const auto *v = static_cast<const __nv_bfloat16 *>(pr.v);
    auto *o = static_cast<__nv_bfloat16 *>(pr.out);
    if (pr.d == 64)
        simt_fwd<64><<<(unsigned)blocks, kWarpsPerBlock * 32, 0, stream>>>(q, k, v, o, rows, pr.L, pr.p, pr.mode);
    else
        simt_fwd<128><<<(unsigned)blocks, kWarpsPerBlock * 32, 0, stream>>>(q, k, v, o, rows, pr.L, pr.p, pr.mode);
    return cudaGetLastError();
}

}  // namespace lssar
