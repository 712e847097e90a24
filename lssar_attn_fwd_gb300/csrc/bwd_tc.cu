// Host side of the tensor-core backward pass: workspace layout, the
// normalisation prologue (shared with the forward), the row and column passes
// and the final gradient of the L2 row normalisation.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bwd_dispatch.cuh"
#include "tc_host.cuh"

namespace lssar {
namespace {

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// [256 B: work counters of the two passes][rmax: BH floats][qh, kh: fp16
// (normalised modes)][query records: BH * n_tiles * 128 * 32 B][dqh, dkh: fp32]
struct Layout {
    size_t rmax, qh, kh, rowc, dqh, dkh, total;
};

Layout layout(const BwdProblem &pr) {
    const size_t BH = (size_t)pr.B * pr.H, elems = BH * pr.L * pr.d;
    const size_t n_tiles = (pr.L + tcb::kBN - 1) / tcb::kBN;
    Layout l;
    l.rmax = 256;
    size_t off = l.rmax + round256(BH * 4);
    const size_t half = uses_normalised_qk(pr.mode) ? round256(elems * 2) : 0;
    l.qh = off;
    off += half;
    l.kh = off;
    off += half;
    l.rowc = off;
    off += round256(BH * n_tiles * tcb::kBN * 32);
    l.dqh = off;
    off += round256(elems * 4);
    l.dkh = off;
    off += round256(elems * 4);
    l.total = off;
    return l;
}

// dq = (dqh - qh (qh . dqh)) / |q| for |q| > 1e-12 (else dqh / 1e-12) in the
// normalised modes, dq = dqh in the softmax modes; the same for k.  D/8
// threads per row, rows of q first, then rows of k.
template <int D>
__global__ void __launch_bounds__(256) finish_grad(const __nv_bfloat16 *__restrict__ q,
                                                   const __nv_bfloat16 *__restrict__ k,
                                                   const float *__restrict__ gq, const float *__restrict__ gk,
                                                   __nv_bfloat16 *__restrict__ dq, __nv_bfloat16 *__restrict__ dk,
                                                   long long rows, int normalised) {
    constexpr int G = D / 8;
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long r = tid / G;
    const int part = (int)(tid % G);
    const bool live = r < 2 * rows;
    const bool is_k = r >= rows;
    const long long rr = is_k ? r - rows : r;
    float x[8], g[8];
    float ss = 0.f, dot = 0.f;
    if (live) {
        const size_t off = (size_t)rr * D + part * 8;
        const uint4 u = *reinterpret_cast<const uint4 *>((is_k ? k : q) + off);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
        const float4 *gs = reinterpret_cast<const float4 *>((is_k ? gk : gq) + off);
        const float4 g0 = gs[0], g1 = gs[1];
        g[0] = g0.x; g[1] = g0.y; g[2] = g0.z; g[3] = g0.w;
        g[4] = g1.x; g[5] = g1.y; g[6] = g1.z; g[7] = g1.w;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(h[e]);
            x[2 * e] = f.x;
            x[2 * e + 1] = f.y;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            ss = fmaf(x[e], x[e], ss);
            dot = fmaf(x[e], g[e], dot);
        }
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, o);
        dot += __shfl_xor_sync(0xffffffffu, dot, o);
    }
    if (!live) return;
    float y[8];
    if (normalised) {
        const float n = sqrtf(ss);
        if (n > 1e-12f) {
            const float inv = 1.f / n, radial = dot * inv * inv;
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = (g[e] - x[e] * radial) * inv;
        } else {
#pragma unroll
            for (int e = 0; e < 8; ++e) y[e] = g[e] * 1e12f;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) y[e] = g[e];
    }
    uint4 o;
    __nv_bfloat162 *h = reinterpret_cast<__nv_bfloat162 *>(&o);
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(y[2 * e], y[2 * e + 1]);
    *reinterpret_cast<uint4 *>((is_k ? dk : dq) + (size_t)rr * D + part * 8) = o;
}

}  // namespace

size_t bwd_tc_workspace_bytes(const BwdProblem &pr) { return layout(pr).total; }

cudaError_t launch_bwd_tc(const BwdProblem &pr, void *ws, cudaStream_t stream) {
    const Layout lay = layout(pr);
    char *base = static_cast<char *>(ws);
    const int BH = pr.B * pr.H;
    const long long rows = (long long)BH * pr.L;
    const bool normalised = uses_normalised_qk(pr.mode);
    unsigned *counters = reinterpret_cast<unsigned *>(base);
    cudaError_t e = cudaMemsetAsync(base, 0, lay.qh, stream);   // counters and rmax
    if (e != cudaSuccess) return e;
    const void *qs = pr.q, *ks = pr.k;
    CUtensorMapDataType st = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (normalised) {
        // query rows as a_i qh_i in fp16, as the forward writes them (positive
        // orientation in every mode: the forward's negated sigmoid rows round
        // to exactly the negated values)
        e = launch_normalize_fp16(pr.q, pr.k, base + lay.qh, base + lay.kh, rows, pr.d, counters + 2, stream,
                                  pr.L, score_qmul(pr.d));
        if (e != cudaSuccess) return e;
        qs = base + lay.qh;
        ks = base + lay.kh;
        st = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    }
    CUtensorMap mq, mk, mv, mdo;
    if (!make_map(&mq, qs, st, BH, pr.L, pr.d) || !make_map(&mk, ks, st, BH, pr.L, pr.d) ||
        !make_map(&mv, pr.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, BH, pr.L, pr.d) ||
        !make_map(&mdo, pr.dout, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, BH, pr.L, pr.d))
        return cudaErrorInvalidValue;

    tcb::Params prm;
    prm.BH = BH;
    prm.L = pr.L;
    prm.n_tiles = (pr.L + tcb::kBN - 1) / tcb::kBN;
    prm.n_items = BH * prm.n_tiles;
    prm.ln_d = logf((float)pr.d);
    prm.p = pr.p;
    prm.H = pr.H;
    prm.per_head = pr.p_head ? 1 : 0;
    prm.exact_weights = exact_weights_requested() ? 1 : 0;
    for (int h = 0; h < 256; ++h) prm.p_head[h] = (pr.p_head && h < pr.H) ? pr.p_head[h] : pr.p;
    prm.stats = reinterpret_cast<const float4 *>(pr.stats);
    prm.rowc = reinterpret_cast<float *>(base + lay.rowc);
    prm.rmax = reinterpret_cast<unsigned *>(base + lay.rmax);
    prm.acc_out = reinterpret_cast<float *>(base + lay.dqh);
    prm.dv = nullptr;
    prm.counter = counters;
    if ((e = error_word_ptr(&prm.err)) != cudaSuccess) return e;
    int sms = 0;
    if ((e = device_sms(&sms)) != cudaSuccess) return e;
    const int grid = prm.n_items < sms ? prm.n_items : sms;

    // row pass: anchor (q, dout), streamed (k, v)
    tcb::Maps m{mq, mdo, mk, mv};
    e = pr.d == 64 ? tcb::dispatch_d64(pr, tcb::kRowPass, m, prm, grid, stream)
                   : tcb::dispatch_d128(pr, tcb::kRowPass, m, prm, grid, stream);
    if (e != cudaSuccess) return e;
    // column pass: anchor (k, v), streamed (q, dout)
    tcb::Params prc = prm;
    prc.acc_out = reinterpret_cast<float *>(base + lay.dkh);
    prc.dv = static_cast<__nv_bfloat16 *>(pr.dv);
    prc.counter = counters + 1;
    tcb::Maps mc{mk, mv, mq, mdo};
    e = pr.d == 64 ? tcb::dispatch_d64(pr, tcb::kColPass, mc, prc, grid, stream)
                   : tcb::dispatch_d128(pr, tcb::kColPass, mc, prc, grid, stream);
    if (e != cudaSuccess) return e;

    const long long threads = 2 * rows * (pr.d / 8);
    const long long blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const auto *q = static_cast<const __nv_bfloat16 *>(pr.q);
    const auto *k = static_cast<const __nv_bfloat16 *>(pr.k);
    const auto *gq = reinterpret_cast<const float *>(base + lay.dqh);
    const auto *gk = reinterpret_cast<const float *>(base + lay.dkh);
    auto *dq = static_cast<__nv_bfloat16 *>(pr.dq);
    auto *dk = static_cast<__nv_bfloat16 *>(pr.dk);
    if (pr.d == 64)
        finish_grad<64><<<(unsigned)blocks, 256, 0, stream>>>(q, k, gq, gk, dq, dk, rows, normalised);
    else
        finish_grad<128><<<(unsigned)blocks, 256, 0, stream>>>(q, k, gq, gk, dq, dk, rows, normalised);
    return cudaGetLastError();
}

}  // namespace lssar
