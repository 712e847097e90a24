// Decode forward: one new query row (position i = L, 1-based) per head against
// a K/V cache of L rows, for every mode of the prefill kernel.  The same
// definitions apply (Key designs 1-2 of the notes on "Softplus Attention with
// Re-weighting Boosts Length Extrapolation in Large Language Models"; the
// ablation normalisers of its ablation table; the softmax of its Background),
// evaluated for the last row only.
//
// The work is a pair of matrix-vector products per head and is bound by HBM:
// every key and value row is read once.  Each head's L keys are split into
// chunks so that B*H*chunks CTAs fill the GPU in one wave:
//   dec_scores   z_j for the chunk (kept in a float scratch so that pass 2 does
//                not read K again), chunk max and chunk sum of the normaliser
//   dec_weights  combines the head's chunk statistics into the row constants,
//                computes the chunk's weights and its partial sum_j w_j v_j, S2
//   dec_combine  sums the partials of each head and divides
// Scores use log2 units as in the prefill kernel: z = log2(e) * x.
//
// The K (V) rows of a chunk are contiguous, so a producer warp streams them
// with bulk copies (cp.async.bulk, 8 KB per stage) into a 4-stage shared-memory
// ring; eight consumer warps read the rows from shared memory.  The first
// stages are requested before the CTA's prologue, so the copy engine runs
// ahead of the arithmetic.  Every wait on the ring is bounded: after 2 s the
// kernel records a code in the device error word and leaves its loop.
#include <cstdlib>
#include <cstring>

#include <cuda_bf16.h>

#include "lssar_internal.cuh"
#include "tc_host.cuh"
#include "tc_ptx.cuh"

namespace lssar {
namespace {

constexpr int kDecWarps = 8;                    // consumer warps
constexpr int kDecThreads = kDecWarps * 32;     // consumer threads
constexpr int kDecBlock = kDecThreads + 32;     // + the producer warp
constexpr int kDecMaxChunk = 4096;              // keys per chunk (scores / weights in smem)
constexpr int kDecStages = 4;
constexpr int kDecStageBytes = 8192;
constexpr int kDecCtasPerSm = 4;
constexpr uint64_t kDecWaitLimitNs = 2000000000ull;
// device error word codes of the decode kernels
enum : unsigned { kErrDecFull = 41, kErrDecEmpty, kErrDecDrain, kErrDecGrid };

// Dynamic shared memory of the two streaming kernels.
struct alignas(16) DecSmem {
    uint8_t ring[kDecStages][kDecStageBytes];
    float row[kDecMaxChunk];           // scores (dec_scores) or weights (dec_weights)
    float red[kDecWarps + 1];
    uint64_t full[kDecStages], empty[kDecStages];
    int abort_flag;
};

// Bounded wait on an mbarrier phase.  With honour_abort it also gives up as
// soon as another role of the CTA has raised the abort flag.
__device__ __forceinline__ bool dec_wait(uint32_t bar, uint32_t parity, DecSmem *sm, unsigned *err,
                                         unsigned code, bool honour_abort) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t spin = 1;; ++spin) {
        if (ptx::mbar_try_wait_sleep(bar, parity, 200000)) return true;
        if ((spin & 15u) == 0) {
            if (honour_abort && *(volatile int *)&sm->abort_flag) return false;
            if (ptx::globaltimer_ns() - t0 > kDecWaitLimitNs) {
                atomicCAS(err, 0u, code);
                *(volatile int *)&sm->abort_flag = 1;
                return false;
            }
        }
    }
}

// Sum or max over all kDecBlock threads (every thread must call it).
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
    for (int w = 0; w < kDecWarps + 1; ++w) r = is_max ? fmaxf(r, red[w]) : r + red[w];
    return r;
}

// log2(1 + 2^z) without overflow for any z (MUFU ex2 / lg2, as in the
// prefill kernel)
__device__ __forceinline__ float sp2_any(float z) {
    return fmaxf(z, 0.f) + ptx::lg2(1.f + ptx::ex2(-fabsf(z)));
}

__device__ __forceinline__ float sigmoid2(float z) {   // 1 / (1 + 2^-z)
    return ptx::rcp(1.f + ptx::ex2(-z));
}

// The normaliser value of a score (softmax modes: relative to the max m).
__device__ __forceinline__ float phi(int mode, float z, float m) {
    if (mode == kSoftmax || mode == kSoftmaxRw) return ptx::ex2(z - m);
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

// The chunk's rows as a stream of stages of KT rows: row block `it` goes to
// the ring's stage sequence number base + it (slot (base + it) % kDecStages),
// so a second stream can follow a first one through the same ring.  The
// producer warp's lane 0 calls issue(0), issue(1), ...
template <int D>
struct Ring {
    static constexpr int KT = kDecStageBytes / (2 * D);   // rows per stage (64 or 32)
    DecSmem *sm;
    const __nv_bfloat16 *src;   // first row of the chunk
    int n;                      // rows in the chunk
    unsigned *err;
    int base = 0;               // stage sequence number of row block 0
    __device__ int stages() const { return (n + KT - 1) / KT; }
    __device__ int slot(int it) const { return (base + it) % kDecStages; }
    __device__ uint32_t parity(int it) const { return ((base + it) / kDecStages) & 1; }
    __device__ bool issue(int it) const {
        const int s = slot(it), use = (base + it) / kDecStages;
        if (use > 0 && !dec_wait(ptx::smem_u32(&sm->empty[s]), (use - 1) & 1, sm, err, kErrDecEmpty, true))
            return false;
        const int rows = min(KT, n - it * KT);
        const uint32_t bytes = (uint32_t)rows * D * 2;
        const uint32_t full = ptx::smem_u32(&sm->full[s]);
        ptx::mbar_arrive_expect_tx(full, bytes);
        // a block of 1..KT whole rows of this chunk, 16-byte aligned at both ends
        const __nv_bfloat16 *from = src + (size_t)it * KT * D;
        if (dcheck(rows >= 1 && rows <= KT && (bytes & 15u) == 0 &&
                       (reinterpret_cast<uintptr_t>(from) & 15u) == 0 && (ptx::smem_u32(sm->ring[s]) & 15u) == 0,
                   err, kDbgBulk))
            ptx::bulk_load(ptx::smem_u32(sm->ring[s]), from, bytes, full);
        return true;
    }
    // Issues row blocks [from, to) in order; returns the number issued in total
    // (fewer than `to` only after a wait gave up).
    __device__ int issue_upto(int from, int to) const {
        int it = from;
        while (it < to && issue(it)) ++it;
        return it;
    }
    // Before the CTA exits: every issued copy has landed (bounded wait, also
    // after an abort, so that no copy is in flight when the CTA ends).
    __device__ void drain(int issued) const {
        for (int it = max(0, issued - kDecStages); it < issued; ++it)
            dec_wait(ptx::smem_u32(&sm->full[slot(it)]), parity(it), sm, err, kErrDecDrain, false);
    }
};

__device__ __forceinline__ void init_ring(DecSmem *sm) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < kDecStages; ++s) {
            ptx::mbar_init(ptx::smem_u32(&sm->full[s]), 1);
            ptx::mbar_init(ptx::smem_u32(&sm->empty[s]), kDecWarps);
        }
        sm->abort_flag = 0;
        ptx::fence_mbar_init();
        ptx::fence_proxy_async_smem();
    }
    __syncthreads();
}

// Consumer warps (warps 0..7): the chunk's scores z_j into sm->row (and into
// z_out[j] when z_out is not null); returns this thread's running max of z.
// A warp load covers KPW rows (16 bytes per lane, D/8 lanes per row); warp w
// takes rows [2w KPW, 2(w+1) KPW) of each stage.  The loop index is
// warp-uniform, so the shuffles are convergent.
template <int D>
__device__ float consume_scores(const Ring<D> &ring, const float *qs, float a, bool raw, float *z_out) {
    constexpr int kParts = D / 8, KPW = 32 / kParts, KT = Ring<D>::KT;
    static_assert(KT == kDecWarps * 2 * KPW, "two loads per warp and stage");
    DecSmem *sm = ring.sm;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / kParts, col8 = lane % kParts;
    const int n = ring.n, n_st = ring.stages();
    float2 qv2[4];
#pragma unroll
    for (int f = 0; f < 4; ++f) qv2[f] = make_float2(qs[col8 * 8 + 2 * f], qs[col8 * 8 + 2 * f + 1]);
    float m = -INFINITY;
    for (int it = 0; it < n_st; ++it) {
        const int s = ring.slot(it);
        if (!__all_sync(0xffffffffu, dec_wait(ptx::smem_u32(&sm->full[s]), ring.parity(it), sm, ring.err,
                                              kErrDecFull, true)))
            break;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int kl = (2 * warp + r) * KPW + sub;   // row within the stage
            const int jj = it * KT + kl;                 // row within the chunk
            uint4 u = make_uint4(0u, 0u, 0u, 0u);
            if (jj < n) u = *reinterpret_cast<const uint4 *>(sm->ring[s] + kl * D * 2 + col8 * 16);
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
            float2 dot2 = make_float2(0.f, 0.f), kss2 = make_float2(0.f, 0.f);
#pragma unroll
            for (int f = 0; f < 4; ++f) {
                const float2 v2 = __bfloat1622float2(h[f]);
                dot2 = __ffma2_rn(v2, qv2[f], dot2);
                kss2 = __ffma2_rn(v2, v2, kss2);
            }
            float dot = dot2.x + dot2.y, kss = kss2.x + kss2.y;
#pragma unroll
            for (int o = kParts / 2; o > 0; o >>= 1) {
                dot += __shfl_xor_sync(0xffffffffu, dot, o);
                kss += __shfl_xor_sync(0xffffffffu, kss, o);
            }
            if (col8 == 0 && jj < n) {
                // |k| clamped at 1e-12 as everywhere: 1/max(|k|, eps) = rsqrt(max(|k|^2, eps^2))
                const float z = raw ? a * dot : a * dot * rsqrtf(fmaxf(kss, 1e-24f));
                sm->row[jj] = z;
                if (z_out) z_out[jj] = z;
                m = fmaxf(m, z);
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sm->empty[s]));
    }
    return m;
}

// Consumer warps: sum_j w_j v_j over the chunk's value rows, weights in
// sm->row; each warp's partial (D columns) goes to accs[warp].
template <int D>
__device__ void consume_pv(const Ring<D> &ring, float (*accs)[D]) {
    constexpr int kParts = D / 8, KPW = 32 / kParts, KT = Ring<D>::KT;
    DecSmem *sm = ring.sm;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int sub = lane / kParts, col8 = lane % kParts;
    const int n = ring.n, n_st = ring.stages();
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int it = 0; it < n_st; ++it) {
        const int s = ring.slot(it);
        if (!__all_sync(0xffffffffu, dec_wait(ptx::smem_u32(&sm->full[s]), ring.parity(it), sm, ring.err,
                                              kErrDecFull, true)))
            break;
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int kl = (2 * warp + r) * KPW + sub;
            const int jj = it * KT + kl;
            if (jj < n) {
                const uint4 u = *reinterpret_cast<const uint4 *>(sm->ring[s] + kl * D * 2 + col8 * 16);
                const float w = sm->row[jj];
                const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
                for (int f = 0; f < 4; ++f) {
                    const float2 r2 = __ffma2_rn(__bfloat1622float2(h[f]), make_float2(w, w),
                                                 make_float2(acc[2 * f], acc[2 * f + 1]));
                    acc[2 * f] = r2.x;
                    acc[2 * f + 1] = r2.y;
                }
            }
        }
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(&sm->empty[s]));
    }
    // the KPW row groups of a warp hold the same columns: fold them
#pragma unroll
    for (int o = kParts; o < 32; o <<= 1)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
    if (sub == 0)
#pragma unroll
        for (int e = 0; e < 8; ++e) accs[warp][col8 * 8 + e] = acc[e];
}

template <int D>
__global__ void __launch_bounds__(kDecBlock, kDecCtasPerSm)
dec_scores(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k, int L,
           int chunk, int mode, float *__restrict__ z_out, float2 *__restrict__ part, unsigned *err) {
    extern __shared__ __align__(128) uint8_t dsm[];
    DecSmem *sm = reinterpret_cast<DecSmem *>(dsm);
    __shared__ float qs[D];
    const int bh = blockIdx.y, c = blockIdx.x, nch = gridDim.x;
    const int j0 = c * chunk, j1 = min(L, j0 + chunk);
    const int n = j1 - j0;
    const bool raw = !uses_normalised_qk(mode);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool producer = warp == kDecWarps;
    const Ring<D> ring{sm, k + ((size_t)bh * L + j0) * D, n, err};
    const int n_st = ring.stages();
    init_ring(sm);
    int issued = 0;
    if (producer && lane == 0) issued = ring.issue_upto(0, min(n_st, kDecStages));
    // query row, L2-normalised for the LSSA family
    float qss = 0.f;
    for (int t = threadIdx.x; t < D; t += kDecBlock) {
        const float x = __bfloat162float(q[(size_t)bh * D + t]);
        qs[t] = x;
        qss += x * x;
    }
    qss = block_reduce(qss, false, sm->red);
    const float log2e = 1.4426950408889634f;
    const float a = raw ? log2e * rsqrtf((float)D)
                        : log2e * logf((float)D) * logf((float)L) / fmaxf(sqrtf(qss), 1e-12f);
    float m = -INFINITY;
    if (producer) {
        if (lane == 0) {
            issued = ring.issue_upto(issued, n_st);
            ring.drain(issued);
        }
        __syncwarp();
    } else {
        m = consume_scores<D>(ring, qs, a, raw, z_out + (size_t)bh * L + j0);
    }
    m = block_reduce(m, true, sm->red);   // its barriers also publish the scores
    float sum = 0.f;
    for (int jj = threadIdx.x; jj < n; jj += kDecBlock) sum += phi(mode, sm->row[jj], m);
    sum = block_reduce(sum, false, sm->red);
    if (threadIdx.x == 0) part[(size_t)bh * nch + c] = make_float2(m, sum);
}

// The head's row constants from its chunks' (max, sum of phi), then the
// weights of this chunk's n scores z[] into w[] (w may be z: in place).
// Every thread of the CTA takes part.
// The head's row maximum and normaliser sum from its chunks' (max, sum of
// phi) pairs, which `stat(u)` returns for chunk u (the softmax normalisers'
// sums are relative to each chunk's own max).
template <typename Stat>
__device__ float2 head_stats(Stat stat, int nch, int mode) {
    float m = -INFINITY;
    for (int u = 0; u < nch; ++u) m = fmaxf(m, stat(u).x);
    float s1 = 0.f;
    for (int u = 0; u < nch; ++u) {
        const float2 pu = stat(u);
        s1 += (mode == kSoftmax || mode == kSoftmaxRw) ? pu.y * exp2f(pu.x - m) : pu.y;
    }
    return make_float2(m, s1);
}

// The chunk's weights w_j from its scores z_j and the head's statistics.
__device__ void weights_from_stats(float2 hs, int L, int mode, int p, const float *z, float *w, int n) {
    const float m = hs.x, s1 = hs.y;
    float kappa = 0.f, beta = 0.f;
    bool uniform = false;
    if (is_reweight(mode)) {
        const float o = (L <= 3) ? 0.f : 1.f;
        const float theta = o * s1 / (float)L;
        const float top = phi(mode, m, m);   // the normaliser at the row maximum
        const float den = top - theta;
        if (den > 1e-5f * top + 2e-5f) {   // the prefill kernel's near-uniform band
            kappa = 1.f / den;
            beta = -theta * kappa;
        } else {
            uniform = true;   // all-zero re-weighted row: uniform prefix mean
        }
    }
    for (int jj = threadIdx.x; jj < n; jj += kDecBlock) {
        const float zj = z[jj];
        float wj;
        if (mode == kSoftmax) wj = exp2f(zj - m);
        else if (mode == kLssa) wj = sp2_any(zj);
        else wj = uniform ? 1.f : powi(fmaxf(phi(mode, zj, m) * kappa + beta, 0.f), p);
        w[jj] = wj;
    }
}

__device__ void chunk_weights(const float2 *__restrict__ part_head, int nch, int L, int mode, int p,
                              const float *z, float *w, int n) {
    // read through L2: other CTAs of the same launch may have written them
    const float2 hs = head_stats([&](int u) { return __ldcg(part_head + u); }, nch, mode);
    weights_from_stats(hs, L, mode, p, z, w, n);
}

template <int D>
__global__ void __launch_bounds__(kDecBlock, kDecCtasPerSm)
dec_weights(const __nv_bfloat16 *__restrict__ v, int L, int chunk, int mode, int p,
            const float *__restrict__ z_in, const float2 *__restrict__ part,
            float *__restrict__ opart /* [BH][nch][D+1] */, unsigned *err) {
    extern __shared__ __align__(128) uint8_t dsm[];
    DecSmem *sm = reinterpret_cast<DecSmem *>(dsm);
    __shared__ float accs[kDecWarps][D];
    const int bh = blockIdx.y, c = blockIdx.x, nch = gridDim.x;
    const int j0 = c * chunk, j1 = min(L, j0 + chunk);
    const int n = j1 - j0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool producer = warp == kDecWarps;
    const Ring<D> ring{sm, v + ((size_t)bh * L + j0) * D, n, err};
    const int n_st = ring.stages();
    init_ring(sm);
    int issued = 0;
    if (producer && lane == 0) issued = ring.issue_upto(0, min(n_st, kDecStages));
    chunk_weights(part + (size_t)bh * nch, nch, L, mode, p, z_in + (size_t)bh * L + j0, sm->row, n);
    __syncthreads();
    if (producer) {
        if (lane == 0) {
            issued = ring.issue_upto(issued, n_st);
            ring.drain(issued);
        }
        __syncwarp();
    } else {
        consume_pv<D>(ring, accs);
    }
    float s2 = 0.f;
    for (int jj = threadIdx.x; jj < n; jj += kDecBlock) s2 += sm->row[jj];
    s2 = block_reduce(s2, false, sm->red);   // also orders the accs writes before the reads below
    float *dst = opart + ((size_t)bh * nch + c) * (D + 1);
    for (int t = threadIdx.x; t < D; t += kDecBlock) {
        float r = 0.f;
        for (int w2 = 0; w2 < kDecWarps; ++w2) r += accs[w2][t];
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

// The whole decode step in one cooperative launch (every CTA resident):
// phase A streams the chunk's keys (scores stay in shared memory) and
// publishes the chunk's (max, sum of phi); the producer then already fetches
// the first value stages into the same ring while the CTAs meet at a grid
// barrier (bounded spin on a counter); phase B forms the weights from the
// head's statistics and streams the values; the last CTA of each head to
// finish (a per-head counter) sums the head's partials into the output.
// sync: [0] grid barrier, [1 + bh] per-head counters, zero at launch.
template <int D>
__global__ void __launch_bounds__(kDecBlock, kDecCtasPerSm)
dec_fused(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
          const __nv_bfloat16 *__restrict__ v, int L, int chunk, int mode, int p,
          float2 *__restrict__ part, float *__restrict__ opart, __nv_bfloat16 *__restrict__ out,
          unsigned *__restrict__ sync, unsigned *err, int withhold_copies) {
    extern __shared__ __align__(128) uint8_t dsm[];
    DecSmem *sm = reinterpret_cast<DecSmem *>(dsm);
    __shared__ float qs[D];
    __shared__ float accs[kDecWarps][D];
    __shared__ int last_of_head;
    const int bh = blockIdx.y, c = blockIdx.x, nch = gridDim.x;
    const int j0 = c * chunk, j1 = min(L, j0 + chunk);
    const int n = j1 - j0;
    const bool raw = !uses_normalised_qk(mode);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool producer = warp == kDecWarps;
    const Ring<D> rk{sm, k + ((size_t)bh * L + j0) * D, n, err, 0};
    const int n_st = rk.stages();
    const Ring<D> rv{sm, v + ((size_t)bh * L + j0) * D, n, err, n_st};
    init_ring(sm);
    // withhold_copies (self-test of the failure path only): the producer
    // issues nothing, so every consumer wait runs into its bound
    const int n_issue = withhold_copies ? 0 : n_st;
    int issued_k = 0, issued_v = 0;
    if (producer && lane == 0) issued_k = rk.issue_upto(0, min(n_issue, kDecStages));
    // phase A: scores
    float qss = 0.f;
    for (int t = threadIdx.x; t < D; t += kDecBlock) {
        const float x = __bfloat162float(q[(size_t)bh * D + t]);
        qs[t] = x;
        qss += x * x;
    }
    qss = block_reduce(qss, false, sm->red);
    const float log2e = 1.4426950408889634f;
    const float a = raw ? log2e * rsqrtf((float)D)
                        : log2e * logf((float)D) * logf((float)L) / fmaxf(sqrtf(qss), 1e-12f);
    float m = -INFINITY;
    if (producer) {
        if (lane == 0) {
            issued_k = rk.issue_upto(issued_k, n_issue);
            // the first value stages follow as the consumers free the ring
            if (issued_k == n_st) issued_v = rv.issue_upto(0, min(n_st, kDecStages));
        }
        __syncwarp();
    } else {
        m = consume_scores<D>(rk, qs, a, raw, nullptr);
    }
    m = block_reduce(m, true, sm->red);   // its barriers also publish the scores
    float sum = 0.f;
    for (int jj = threadIdx.x; jj < n; jj += kDecBlock) sum += phi(mode, sm->row[jj], m);
    sum = block_reduce(sum, false, sm->red);
    // grid barrier: every chunk's statistics are in `part`
    if (threadIdx.x == 0) {
        part[(size_t)bh * nch + c] = make_float2(m, sum);
        __threadfence();
        atomicAdd(sync, 1u);
        const unsigned total = gridDim.x * gridDim.y;
        const uint64_t t0 = ptx::globaltimer_ns();
        while (*(volatile unsigned *)sync < total) {
            __nanosleep(256);
            if (ptx::globaltimer_ns() - t0 > kDecWaitLimitNs) {
                atomicCAS(err, 0u, (unsigned)kErrDecGrid);
                *(volatile int *)&sm->abort_flag = 1;
                break;
            }
        }
        __threadfence();
    }
    __syncthreads();
    // phase B: weights in place of the scores, then the values
    chunk_weights(part + (size_t)bh * nch, nch, L, mode, p, sm->row, sm->row, n);
    __syncthreads();
    if (producer) {
        if (lane == 0) {
            if (issued_k == n_st) issued_v = rv.issue_upto(issued_v, n_st);
            // the last kDecStages copies of the K-then-V sequence have landed
            // (earlier ones were consumed, and their slots reused)
            const int total = issued_k + issued_v;
            for (int g = max(0, total - kDecStages); g < total; ++g)
                dec_wait(ptx::smem_u32(&sm->full[g % kDecStages]), (g / kDecStages) & 1, sm, err, kErrDecDrain,
                         false);
        }
        __syncwarp();
    } else {
        consume_pv<D>(rv, accs);
    }
    float s2 = 0.f;
    for (int jj = threadIdx.x; jj < n; jj += kDecBlock) s2 += sm->row[jj];
    s2 = block_reduce(s2, false, sm->red);   // also orders the accs writes before the reads below
    float *dst = opart + ((size_t)bh * nch + c) * (D + 1);
    for (int t = threadIdx.x; t < D; t += kDecBlock) {
        float r = 0.f;
        for (int w2 = 0; w2 < kDecWarps; ++w2) r += accs[w2][t];
        dst[t] = r;
    }
    if (threadIdx.x == 0) dst[D] = s2;
    // the last chunk of the head to finish writes the head's output row
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last_of_head = atomicAdd(sync + 1 + bh, 1u) == (unsigned)(nch - 1);
    __syncthreads();
    if (last_of_head) {
        __threadfence();
        for (int t = threadIdx.x; t < D; t += kDecBlock) {
            float o = 0.f, sw = 0.f;
            for (int u = 0; u < nch; ++u) {
                const volatile float *src = opart + ((size_t)bh * nch + u) * (D + 1);
                o += src[t];
                sw += src[D];
            }
            out[(size_t)bh * D + t] = __float2bfloat16_rn(o / sw);
        }
    }
}

// The whole step as one launch with one thread-block cluster per head (the
// cluster's CTAs are the head's chunks, rank = chunk): phase A streams the
// chunk's keys and keeps the scores in shared memory; the chunks' (max, sum
// of phi) meet through distributed shared memory at a cluster barrier; phase
// B forms the weights and streams the values (the producer has already
// fetched the first value stages); rank 0 sums the chunks' partial outputs
// from its partners' shared memory.  Heads never wait on one another, and no
// global memory beyond q, k, v and out is touched.  Every thread of every CTA
// reaches each cluster barrier (no path returns early; a timed-out copy wait
// only sets the error word and the abort flag).
template <int D>
__global__ void __launch_bounds__(kDecBlock, kDecCtasPerSm)
dec_cluster(const __nv_bfloat16 *__restrict__ q, const __nv_bfloat16 *__restrict__ k,
            const __nv_bfloat16 *__restrict__ v, int L, int chunk, int mode, int p,
            __nv_bfloat16 *__restrict__ out, unsigned *err, int withhold_copies) {
    extern __shared__ __align__(128) uint8_t dsm[];
    DecSmem *sm = reinterpret_cast<DecSmem *>(dsm);
    __shared__ float qs[D];
    __shared__ float accs[kDecWarps][D];
    __shared__ float2 stat;          // this chunk's (max, sum of phi)
    __shared__ float opart[D + 1];   // this chunk's sum_j w_j v_j and sum_j w_j
    const int bh = blockIdx.y, c = blockIdx.x, nch = gridDim.x;
    const int j0 = c * chunk, j1 = min(L, j0 + chunk);
    const int n = j1 - j0;
    const bool raw = !uses_normalised_qk(mode);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool producer = warp == kDecWarps;
    const Ring<D> rk{sm, k + ((size_t)bh * L + j0) * D, n, err, 0};
    const int n_st = rk.stages();
    const Ring<D> rv{sm, v + ((size_t)bh * L + j0) * D, n, err, n_st};
    init_ring(sm);
    // withhold_copies (self-test of the failure path only): the producer
    // issues nothing, so every consumer wait runs into its bound
    const int n_issue = withhold_copies ? 0 : n_st;
    int issued_k = 0, issued_v = 0;
    if (producer && lane == 0) issued_k = rk.issue_upto(0, min(n_issue, kDecStages));
    // phase A: scores
    float qss = 0.f;
    for (int t = threadIdx.x; t < D; t += kDecBlock) {
        const float x = __bfloat162float(q[(size_t)bh * D + t]);
        qs[t] = x;
        qss += x * x;
    }
    qss = block_reduce(qss, false, sm->red);
    const float log2e = 1.4426950408889634f;
    const float a = raw ? log2e * rsqrtf((float)D)
                        : log2e * logf((float)D) * logf((float)L) / fmaxf(sqrtf(qss), 1e-12f);
    float m = -INFINITY;
    if (producer) {
        if (lane == 0) {
            issued_k = rk.issue_upto(issued_k, n_issue);
            // the first value stages follow as the consumers free the ring
            if (issued_k == n_st) issued_v = rv.issue_upto(0, min(n_st, kDecStages));
        }
        __syncwarp();
    } else {
        m = consume_scores<D>(rk, qs, a, raw, nullptr);
    }
    m = block_reduce(m, true, sm->red);   // its barriers also publish the scores
    float sum = 0.f;
    for (int jj = threadIdx.x; jj < n; jj += kDecBlock) sum += phi(mode, sm->row[jj], m);
    sum = block_reduce(sum, false, sm->red);
    if (threadIdx.x == 0) stat = make_float2(m, sum);
    ptx::cluster_sync();   // every chunk's statistics are in its CTA's shared memory
    const uint32_t stat_addr = ptx::smem_u32(&stat);
    const float2 hs = head_stats(
        [&](int u) {
            const uint32_t r = ptx::cluster_map(stat_addr, (uint32_t)u);
            return make_float2(ptx::ld_cluster_f32(r), ptx::ld_cluster_f32(r + 4));
        },
        nch, mode);
    // phase B: weights in place of the scores, then the values
    weights_from_stats(hs, L, mode, p, sm->row, sm->row, n);
    __syncthreads();
    if (producer) {
        if (lane == 0) {
            if (issued_k == n_st) issued_v = rv.issue_upto(issued_v, n_st);
            // the last kDecStages copies of the K-then-V sequence have landed
            // (earlier ones were consumed, and their slots reused)
            const int total = issued_k + issued_v;
            for (int g = max(0, total - kDecStages); g < total; ++g)
                dec_wait(ptx::smem_u32(&sm->full[g % kDecStages]), (g / kDecStages) & 1, sm, err, kErrDecDrain,
                         false);
        }
        __syncwarp();
    } else {
        consume_pv<D>(rv, accs);
    }
    float s2 = 0.f;
    for (int jj = threadIdx.x; jj < n; jj += kDecBlock) s2 += sm->row[jj];
    s2 = block_reduce(s2, false, sm->red);   // also orders the accs writes before the reads below
    for (int t = threadIdx.x; t < D; t += kDecBlock) {
        float r = 0.f;
        for (int w2 = 0; w2 < kDecWarps; ++w2) r += accs[w2][t];
        opart[t] = r;
    }
    if (threadIdx.x == 0) opart[D] = s2;
    ptx::cluster_sync();   // every chunk's partial output is in its CTA's shared memory
    if (c == 0) {
        const uint32_t op_addr = ptx::smem_u32(opart);
        for (int t = threadIdx.x; t < D; t += kDecBlock) {
            float o = 0.f, sw = 0.f;
            for (int u = 0; u < nch; ++u) {
                const uint32_t r = ptx::cluster_map(op_addr, (uint32_t)u);
                o += ptx::ld_cluster_f32(r + 4u * (uint32_t)t);
                sw += ptx::ld_cluster_f32(r + 4u * D);
            }
            out[(size_t)bh * D + t] = __float2bfloat16_rn(o / sw);
        }
    }
    ptx::cluster_sync();   // the partners' shared memory stays in place until rank 0 has read it
}

// Chunk length: a multiple of 64 rows (whole stages at both head dimensions),
// at most kDecMaxChunk, and chunks for at most kDecCtasPerSm CTAs per SM (one
// wave) whenever the heads allow it.
int choose_chunk(int BH, int L, int sms) {
    const long long slots = (long long)kDecCtasPerSm * sms;
    long long nch = slots / BH;
    if (nch < 1) nch = 1;
    long long chunk = (L + nch - 1) / nch;
    chunk = ((chunk + 63) / 64) * 64;
    if (chunk > kDecMaxChunk) chunk = kDecMaxChunk;
    return (int)chunk;
}

constexpr int kDecMaxCluster = 16;   // CTAs per cluster (above 8: non-portable size)

// Chunks per head for the cluster path: about one wave of kDecCtasPerSm CTAs
// per SM when the heads allow it, at most kDecMaxCluster; 0 when a chunk would
// exceed kDecMaxChunk rows (the path is then not available).  (A rule that
// counted whole waves of CTAs, each as long as its chunk plus a fixed cost,
// split 768 heads of 2048 keys into three chunks and lost 7 %: the CTAs of
// a partial wave share the memory bandwidth rather than leave it idle.)
int cluster_chunks(int BH, int L, int sms, int *chunk_out) {
    long long nch = (long long)kDecCtasPerSm * sms / BH;
    if (nch < 1) nch = 1;
    if (nch > kDecMaxCluster) nch = kDecMaxCluster;
    long long chunk = (L + nch - 1) / nch;
    chunk = ((chunk + 63) / 64) * 64;
    if (chunk > kDecMaxChunk) return 0;
    *chunk_out = (int)chunk;
    return (int)((L + chunk - 1) / chunk);
}

// Launch configuration of dec_cluster: BH clusters of nch CTAs (attr is the
// caller's storage for the cluster-dimension attribute).
cudaLaunchConfig_t cluster_config(int BH, int nch, cudaStream_t stream, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nch, BH);
    cfg.blockDim = dim3(kDecBlock);
    cfg.dynamicSmemBytes = sizeof(DecSmem);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)nch;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// Whether this device can place a cluster of nch dec_cluster CTAs (checked
// once per size and device).
template <int D>
cudaError_t cluster_fits(int nch, bool *fits_out) {
    const int smem = (int)sizeof(DecSmem);
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = cluster_config(1, nch, nullptr, attr);
    static PerDeviceOnce once[kDecMaxCluster + 1];
    int fits = 0;
    cudaError_t e = per_device_once(once[nch], &fits, [&](int &v) {
        cudaError_t r = cudaFuncSetAttribute(dec_cluster<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (r == cudaSuccess && nch > 8)
            r = cudaFuncSetAttribute(dec_cluster<D>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (r != cudaSuccess) return r;
        int clusters = 0;
        r = cudaOccupancyMaxActiveClusters(&clusters, dec_cluster<D>, &cfg);
        if (r != cudaSuccess) {
            (void)cudaGetLastError();   // a size this device does not support: use the other path
            clusters = 0;
        }
        v = clusters > 0 ? 1 : 0;
        return cudaSuccess;
    });
    *fits_out = fits != 0;
    return e;
}

// Launch of dec_cluster with nch CTAs per cluster (a size cluster_fits accepted).
template <int D>
cudaError_t launch_cluster(const DecodeProblem &pr, int BH, int chunk, int nch, unsigned *err, int withhold,
                           cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = cluster_config(BH, nch, stream, attr);
    const auto *q = static_cast<const __nv_bfloat16 *>(pr.q);
    const auto *k = static_cast<const __nv_bfloat16 *>(pr.k);
    const auto *v = static_cast<const __nv_bfloat16 *>(pr.v);
    auto *o = static_cast<__nv_bfloat16 *>(pr.out);
    return cudaLaunchKernelEx(&cfg, dec_cluster<D>, q, k, v, pr.L, chunk, pr.mode, pr.p, o, err, withhold);
}

// One cooperative launch of dec_fused when every CTA of the grid can be
// resident at once; otherwise the three-kernel sequence.
// CTAs of dec_fused resident per SM (checked once per device; also sets the
// shared-memory attributes of the grid-path kernels).
template <int D>
cudaError_t grid_per_sm(int *per_sm) {
    const int smem = (int)sizeof(DecSmem);
    static PerDeviceOnce once;
    return per_device_once(once, per_sm, [&](int &v) {
        cudaError_t r = cudaFuncSetAttribute(dec_fused<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (r == cudaSuccess) r = cudaFuncSetAttribute(dec_scores<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (r == cudaSuccess) r = cudaFuncSetAttribute(dec_weights<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        return r != cudaSuccess ? r : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&v, dec_fused<D>, kDecBlock, smem);
    });
}

template <int D>
cudaError_t launch_d(const DecodeProblem &pr, int BH, int chunk, int nch, bool cooperative, float *z, float2 *part,
                     float *opart, unsigned *sync, unsigned *err, int withhold, cudaStream_t stream) {
    const int smem = (int)sizeof(DecSmem);
    cudaError_t e;
    if (withhold && !cooperative) return cudaErrorInvalidConfiguration;
    if (cooperative) {
        e = cudaMemsetAsync(sync, 0, (size_t)(1 + BH) * sizeof(unsigned), stream);
        if (e != cudaSuccess) return e;
        const auto *q = static_cast<const __nv_bfloat16 *>(pr.q);
        const auto *k = static_cast<const __nv_bfloat16 *>(pr.k);
        const auto *v = static_cast<const __nv_bfloat16 *>(pr.v);
        auto *o = static_cast<__nv_bfloat16 *>(pr.out);
        int L = pr.L, mode = pr.mode, p = pr.p;
        void *args[] = {&q, &k, &v, &L, &chunk, &mode, &p, &part, &opart, &o, &sync, &err, &withhold};
        return cudaLaunchCooperativeKernel((const void *)dec_fused<D>, dim3(nch, BH), dim3(kDecBlock), args,
                                           (size_t)smem, stream);
    }
    const dim3 grid(nch, BH);
    const auto *q = static_cast<const __nv_bfloat16 *>(pr.q);
    const auto *k = static_cast<const __nv_bfloat16 *>(pr.k);
    const auto *v = static_cast<const __nv_bfloat16 *>(pr.v);
    dec_scores<D><<<grid, kDecBlock, smem, stream>>>(q, k, pr.L, chunk, pr.mode, z, part, err);
    dec_weights<D><<<grid, kDecBlock, smem, stream>>>(v, pr.L, chunk, pr.mode, pr.p, z, part, opart, err);
    dec_combine<D><<<BH, D, 0, stream>>>(opart, nch, static_cast<__nv_bfloat16 *>(pr.out));
    return cudaGetLastError();
}

// Layout: [scores z: BH*L floats][chunk statistics][partials [BH][nch][d+1]]
// [sync counters: 1 + BH]; each part 256-byte aligned.
struct DecLayout {
    size_t part, opart, sync, total;
};

DecLayout dec_layout(int BH, int L, int d, int nch) {
    auto r = [](size_t x) { return (x + 255) & ~(size_t)255; };
    DecLayout l;
    l.part = r((size_t)BH * L * 4);
    l.opart = l.part + r((size_t)BH * nch * 8);
    l.sync = l.opart + r((size_t)BH * nch * (d + 1) * 4);
    l.total = l.sync + r((size_t)(1 + BH) * 4);
    return l;
}

}  // namespace

size_t decode_workspace_bytes(int BH, int L, int d, int sms) {
    const int chunk = choose_chunk(BH, L, sms);
    return dec_layout(BH, L, d, (L + chunk - 1) / chunk).total;
}

cudaError_t decode_route(int BH, int L, int d, DecodeRoute *route) {
    int sms = 0;
    cudaError_t e = device_sms(&sms);
    if (e != cudaSuccess) return e;
    // LSSAR_DECODE_PATH=grid | split steers the step away from the cluster
    // path (grid: the cooperative launch where possible; split: the three
    // launches), so that tests reach every path at small sizes.
    const char *force = getenv("LSSAR_DECODE_PATH");
    const bool no_cluster = force && (strcmp(force, "grid") == 0 || strcmp(force, "split") == 0);
    const bool split = force && strcmp(force, "split") == 0;
    int cchunk = 0;
    const int cnch = no_cluster ? 0 : cluster_chunks(BH, L, sms, &cchunk);
    if (cnch > 0) {
        bool fits = false;
        e = d == 64 ? cluster_fits<64>(cnch, &fits) : cluster_fits<128>(cnch, &fits);
        if (e != cudaSuccess) return e;
        if (fits) {
            *route = DecodeRoute{kDecodeCluster, cnch, cchunk};
            return cudaSuccess;
        }
    }
    const int chunk = choose_chunk(BH, L, sms);
    const int nch = (L + chunk - 1) / chunk;
    int per_sm = 0;
    e = d == 64 ? grid_per_sm<64>(&per_sm) : grid_per_sm<128>(&per_sm);
    if (e != cudaSuccess) return e;
    const bool coop = !split && (long long)nch * BH <= (long long)per_sm * sms;
    *route = DecodeRoute{coop ? kDecodeGrid : kDecodeSplit, nch, chunk};
    return cudaSuccess;
}

cudaError_t launch_decode(const DecodeProblem &pr, void *ws, cudaStream_t stream, bool withhold_copies) {
    unsigned *err = nullptr;
    cudaError_t e = error_word_ptr(&err);
    if (e != cudaSuccess) return e;
    const int BH = pr.B * pr.H;
    const int w = withhold_copies ? 1 : 0;
    DecodeRoute route;
    if ((e = decode_route(BH, pr.L, pr.d, &route)) != cudaSuccess) return e;
    if (route.path == kDecodeCluster)
        return pr.d == 64 ? launch_cluster<64>(pr, BH, route.chunk_rows, route.chunks, err, w, stream)
                          : launch_cluster<128>(pr, BH, route.chunk_rows, route.chunks, err, w, stream);
    const int chunk = route.chunk_rows, nch = route.chunks;
    const bool coop = route.path == kDecodeGrid;
    char *base = static_cast<char *>(ws);
    const DecLayout lay = dec_layout(BH, pr.L, pr.d, nch);
    float *z = reinterpret_cast<float *>(base);
    float2 *part = reinterpret_cast<float2 *>(base + lay.part);
    float *opart = reinterpret_cast<float *>(base + lay.opart);
    unsigned *sync = reinterpret_cast<unsigned *>(base + lay.sync);
    return pr.d == 64 ? launch_d<64>(pr, BH, chunk, nch, coop, z, part, opart, sync, err, w, stream)
                      : launch_d<128>(pr, BH, chunk, nch, coop, z, part, opart, sync, err, w, stream);
}

}  // namespace lssar
