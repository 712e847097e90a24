// Host side of the tensor-core backward pass: workspace layout, the
// normalisation prologue (shared with the forward) and the row and column
// passes (whose epilogues apply the gradient of the L2 row normalisation).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "bwd_dispatch.cuh"
#include "tc_host.cuh"

namespace lssar {
namespace {

size_t round256(size_t x) { return (x + 255) & ~(size_t)255; }

// [256 B: work counters of the two passes][rmax: BH floats][qh, kh: fp16
// (normalised modes)][query records: BH * n_tiles * 128 * 32 B]
struct Layout {
    size_t rmax, qh, kh, rowc, total;
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
    l.total = off;
    return l;
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
    prm.xraw = static_cast<const __nv_bfloat16 *>(pr.q);
    prm.grad = static_cast<__nv_bfloat16 *>(pr.dq);
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
    prc.xraw = static_cast<const __nv_bfloat16 *>(pr.k);
    prc.grad = static_cast<__nv_bfloat16 *>(pr.dk);
    prc.dv = static_cast<__nv_bfloat16 *>(pr.dv);
    prc.counter = counters + 1;
    tcb::Maps mc{mk, mv, mq, mdo};
    e = pr.d == 64 ? tcb::dispatch_d64(pr, tcb::kColPass, mc, prc, grid, stream)
                   : tcb::dispatch_d128(pr, tcb::kColPass, mc, prc, grid, stream);
    return e;
}

}  // namespace lssar
