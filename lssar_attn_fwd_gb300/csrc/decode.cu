// Decode forward: one new query row (position i = L, 1-based) per head against
// a K/V cache of L rows, for every mode of the prefill kernel.  The same
// definitions apply (Key designs 1-2 of the notes on "Softplus Attention with
// Re-weighting Boosts Length Extrapolation in Large Language Models"; the
// ablation normalisers of its ablation table; the softmax of its Background),
// evaluated for the last row only.
//
// The work is a pair of matrix-vector products per head and is bound by HBM:
// every key and value row is read once.  Each head's L keys are split into
// chunks so that B*H*chunks CTAs fill the GPU:
//   dec_scores   z_j for the chunk (kept in a float scratch so that pass 2 does
//                not read K again), chunk max and chunk sum of the normaliser
//   dec_weights  combines the head's chunk statistics into the row constants,
//                computes the chunk's weights and its partial sum_j w_j v_j, S2
//   dec_combine  sums the partials of each head and divides
// Scores use log2 units as in the prefill kernel: z = log2(e) * x.
#include <cuda_bf16.h>

#include "lssar_internal.cuh"

namespace lssar {
namespace {

constexpr int kDecThreads = 256;
constexpr int kDecMaxPerThread = 16;   // keys per thread in a chunk (chunk <= 4096)

__device__ __forceinline__ float block_reduce(float x, bool is_max, float *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float y = __shfl_xor_sync(0xffffffffu, x, o);
        x = is_max ? fmaxf(x, y) : x + y;
    }
    __syncthreads();
    if (lane == 0) red[warp] = x;
    __syncthreads();
    float r = is_max ? -INFINITY : 0.f;
    for (int w = 0; w < kDecThreads / 32; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
    return r;
}

// log2(1 + 2^z) without overflow for any z
__device__ __forceinline__ float sp2_any(float z) {
    return fmaxf(z, 0.f) + log2f(1.f + exp2f(-fabsf(z)));
}

__device__ __forceinline__ float sigmoid2(float z) {   // 1 / (1 + 2^-z)
    return 1.f / (1.f + exp2f(-z));
}

// The normaliser value of a score (softmax modes: relative to the max m).
__device__ __forceinline__ float phi(int mode, float z, float m) {
    if (mode == kSoftmax || mode == kSoftmaxRw) return exp2f(z - m);
    if (mode == kSigmoidRw) return sigmoid2(z);
    return sp2_any(z);
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
__global__ void __launch_bounds__(kDecThreads)
dec_scores(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k, int L,
           int chunk, int mode, float *__restrict__ z_out, float2 *__restrict__ part) {
    __shared__ float qs[D];
    __shared__ float red[kDecThreads / 32];
    const int bh = blockIdx.y, c = blockIdx.x, nch = gridDim.x;
    const int j0 = c * chunk, j1 = min(L, j0 + chunk);
    const bool raw = !uses_normalised_qk(mode);
    // query row, L2-normalised for the LSSA family
    float qss = 0.f;
    for (int t = threadIdx.x; t < D; t += kDecThreads) {
        const float x = __bfloat162float(q[(size_t)bh * D + t]);
        qs[t] = x;
        qss += x * x;
    }
    qss = block_reduce(qss, false, red);
    const float log2e = 1.4426950408889634f;
    const float a = raw ? log2e * rsqrtf((float)D)
                        : log2e * logf((float)D) * logf((float)L) / fmaxf(sqrtf(qss), 1e-12f);
    // scores: a warp load covers KPW keys (16 bytes per lane, D/8 lanes per key),
    // kUnroll loads in flight per lane; the lanes of a key then add their parts
    constexpr int kParts = D / 8, KPW = 32 / kParts, kWarps = kDecThreads / 32, kUnroll = 4;
    __shared__ float zs[kDecMaxPerThread * kDecThreads];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / kParts, col8 = lane % kParts;
    const int n = j1 - j0;
    float qv[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) qv[e] = qs[col8 * 8 + e];
    const __nv_bfloat16 *kb = k + ((size_t)bh * L + j0) * D + col8 * 8;
    float m = -INFINITY;
    // The loop index is the same for every lane of the warp (the lane's key
    // offset `sub` is added inside), so the shuffles below are convergent.
    for (int base = warp * KPW; base < n; base += kWarps * KPW * kUnroll) {
        uint4 u[kUnroll];
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            const int jj = base + r * kWarps * KPW + sub;
            u[r] = jj < n ? __ldg(reinterpret_cast<const uint4 *>(kb + (size_t)jj * D))
                          : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u[r]);
            float dot = 0.f, kss = 0.f;
#pragma unroll
            for (int f = 0; f < 4; ++f) {
                const float2 v2 = __bfloat1622float2(h[f]);
                dot = fmaf(v2.x, qv[2 * f], dot);
                dot = fmaf(v2.y, qv[2 * f + 1], dot);
                kss = fmaf(v2.x, v2.x, kss);
                kss = fmaf(v2.y, v2.y, kss);
            }
#pragma unroll
            for (int o = kParts / 2; o > 0; o >>= 1) {
                dot += __shfl_xor_sync(0xffffffffu, dot, o);
                kss += __shfl_xor_sync(0xffffffffu, kss, o);
            }
            const int jj = base + r * kWarps * KPW + sub;
            if (col8 == 0 && jj < n) {
                const float z = raw ? a * dot : a * dot / fmaxf(sqrtf(kss), 1e-12f);
                zs[jj] = z;
                z_out[(size_t)bh * L + j0 + jj] = z;
                m = fmaxf(m, z);
            }
        }
    }
    m = block_reduce(m, true, red);   // its barriers also publish zs
    float s = 0.f;
    for (int jj = threadIdx.x; jj < n; jj += kDecThreads) s += phi(mode, zs[jj], m);
    s = block_reduce(s, false, red);
    if (threadIdx.x == 0) part[(size_t)bh * nch + c] = make_float2(m, s);
}

template <int D>
__global__ void __launch_bounds__(kDecThreads)
dec_weights(const __nv_bfloat16 *__restrict__ v, int L, int chunk, int mode, int p,
            const float *__restrict__ z_in, const float2 *__restrict__ part,
            float *__restrict__ opart /* [BH][nch][D+1] */) {
    __shared__ float wsm[kDecMaxPerThread * kDecThreads];
    __shared__ float accs[kDecThreads / 32][D];
    __shared__ float red[kDecThreads / 32];
    const int bh = blockIdx.y, c = blockIdx.x, nch = gridDim.x;
    const int j0 = c * chunk, j1 = min(L, j0 + chunk);
    // row statistics of the head from its chunks
    float m = -INFINITY;
    for (int u = 0; u < nch; ++u) m = fmaxf(m, part[(size_t)bh * nch + u].x);
    float s1 = 0.f;
    for (int u = 0; u < nch; ++u) {
        const float2 pu = part[(size_t)bh * nch + u];
        s1 += (mode == kSoftmax || mode == kSoftmaxRw) ? pu.y * exp2f(pu.x - m) : pu.y;
    }
    float kappa = 0.f, beta = 0.f;
    bool uniform = false;
    if (is_reweight(mode)) {
        const float o = (L <= 3) ? 0.f : 1.f;
        const float theta = o * s1 / (float)L;
        const float top = phi(mode, m, m);   // the normaliser at the row maximum
        const float den = top - theta;
        if (den > 1e-4f * top + 1e-6f) {
            kappa = 1.f / den;
            beta = -theta * kappa;
        } else {
            uniform = true;   // all-zero re-weighted row: uniform prefix mean
        }
    }
    for (int jj = threadIdx.x; jj < j1 - j0; jj += kDecThreads) {
        const float z = z_in[(size_t)bh * L + j0 + jj];
        float w;
        if (mode == kSoftmax) w = exp2f(z - m);
        else if (mode == kLssa) w = sp2_any(z);
        else w = uniform ? 1.f : powi(fmaxf(phi(mode, z, m) * kappa + beta, 0.f), p);
        wsm[jj] = w;
    }
    __syncthreads();
    // partial sum_j w_j v_j: a warp load covers KPW keys (16 bytes per lane,
    // D/8 lanes per key); each lane keeps kUnroll loads in flight
    constexpr int kParts = D / 8, KPW = 32 / kParts, kWarps = kDecThreads / 32, kUnroll = 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / kParts, col8 = lane % kParts;
    const int n = j1 - j0;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    const __nv_bfloat16 *vb = v + ((size_t)bh * L + j0) * D + col8 * 8;
    for (int base = warp * KPW; base < n; base += kWarps * KPW * kUnroll) {   // warp-uniform
        uint4 u[kUnroll];
        float w[kUnroll];
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            const int jj = base + r * kWarps * KPW + sub;
            if (jj < n) {
                u[r] = __ldg(reinterpret_cast<const uint4 *>(vb + (size_t)jj * D));
                w[r] = wsm[jj];
            } else {
                u[r] = make_uint4(0u, 0u, 0u, 0u);
                w[r] = 0.f;
            }
        }
#pragma unroll
        for (int r = 0; r < kUnroll; ++r) {
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u[r]);
#pragma unroll
            for (int f = 0; f < 4; ++f) {
                const float2 v2 = __bfloat1622float2(h[f]);
                acc[2 * f] = fmaf(w[r], v2.x, acc[2 * f]);
                acc[2 * f + 1] = fmaf(w[r], v2.y, acc[2 * f + 1]);
            }
        }
    }
    // the KPW key groups of a warp hold the same columns: fold them
#pragma unroll
    for (int o = kParts; o < 32; o <<= 1)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
    if (sub == 0)
#pragma unroll
        for (int e = 0; e < 8; ++e) accs[warp][col8 * 8 + e] = acc[e];
    float s2 = 0.f;
    for (int jj = threadIdx.x; jj < n; jj += kDecThreads) s2 += wsm[jj];
    s2 = block_reduce(s2, false, red);   // also orders the accs writes before the reads below
    float *dst = opart + ((size_t)bh * nch + c) * (D + 1);
    for (int t = threadIdx.x; t < D; t += kDecThreads) {
        float r = 0.f;
        for (int w2 = 0; w2 < kWarps; ++w2) r += accs[w2][t];
        dst[t] = r;
    }
    if (threadIdx.x == 0) dst[D] = s2;
}

template <int D>
__global__ void __launch_bounds__(D)
dec_combine(const float *__restrict__ opart, int nch, __nv_bfloat16 *__restrict__ out) {
    const int bh = blockIdx.x, t = threadIdx.x;
    float o = 0.f, s = 0.f;
    for (int c = 0; c < nch; ++c) {
        const float *src = opart + ((size_t)bh * nch + c) * (D + 1);
        o += src[t];
        s += src[D];
    }
    out[(size_t)bh * D + t] = __float2bfloat16_rn(o / s);
}

// Chunk length: a multiple of the block size, at most 16 keys per thread,
// and enough chunks for about four CTAs per SM.
int choose_chunk(int BH, int L, int sms) {
    const long long want_ctas = 4LL * sms;
    long long nch = (want_ctas + BH - 1) / BH;
    if (nch < 1) nch = 1;
    long long chunk = (L + nch - 1) / nch;
    chunk = ((chunk + kDecThreads - 1) / kDecThreads) * kDecThreads;
    if (chunk > (long long)kDecMaxPerThread * kDecThreads) chunk = (long long)kDecMaxPerThread * kDecThreads;
    if (chunk < kDecThreads) chunk = kDecThreads;
    return (int)chunk;
}

}  // namespace

size_t decode_workspace_bytes(int BH, int L, int d, int sms) {
    const int chunk = choose_chunk(BH, L, sms);
    const size_t nch = (L + chunk - 1) / chunk;
    const size_t z = ((size_t)BH * L * 4 + 255) & ~(size_t)255;
    const size_t part = ((size_t)BH * nch * 8 + 255) & ~(size_t)255;
    const size_t op = (size_t)BH * nch * (d + 1) * 4;
    return z + part + op;
}

cudaError_t launch_decode(const DecodeProblem &pr, void *ws, cudaStream_t stream) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int BH = pr.B * pr.H;
    const int chunk = choose_chunk(BH, pr.L, sms);
    const int nch = (pr.L + chunk - 1) / chunk;
    char *base = static_cast<char *>(ws);
    float *z = reinterpret_cast<float *>(base);
    const size_t zb = ((size_t)BH * pr.L * 4 + 255) & ~(size_t)255;
    float2 *part = reinterpret_cast<float2 *>(base + zb);
    const size_t pb = ((size_t)BH * nch * 8 + 255) & ~(size_t)255;
    float *opart = reinterpret_cast<float *>(base + zb + pb);
    const dim3 grid(nch, BH);
    const auto *q = static_cast<const __nv_bfloat16 *>(pr.q);
    const auto *k = static_cast<const __nv_bfloat16 *>(pr.k);
    const auto *v = static_cast<const __nv_bfloat16 *>(pr.v);
    auto *o = static_cast<__nv_bfloat16 *>(pr.out);
    if (pr.d == 64) {
        dec_scores<64><<<grid, kDecThreads, 0, stream>>>(q, k, pr.L, chunk, pr.mode, z, part);
        dec_weights<64><<<grid, kDecThreads, 0, stream>>>(v, pr.L, chunk, pr.mode, pr.p, z, part, opart);
        dec_combine<64><<<BH, 64, 0, stream>>>(opart, nch, o);
    } else {
        dec_scores<128><<<grid, kDecThreads, 0, stream>>>(q, k, pr.L, chunk, pr.mode, z, part);
        dec_weights<128><<<grid, kDecThreads, 0, stream>>>(v, pr.L, chunk, pr.mode, pr.p, z, part, opart);
        dec_combine<128><<<BH, 128, 0, stream>>>(opart, nch, o);
    }
    return cudaGetLastError();
}

}  // namespace lssar
