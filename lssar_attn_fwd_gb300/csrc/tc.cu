// Host side of the tensor-core path: the row-normalisation prologue, TMA
// tensor maps, template dispatch and launch, and the device error word.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <functional>
#include <map>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

#include "tc_kernel.cuh"
#include "tc_dispatch.cuh"
#include "tc_host.cuh"

namespace lssar {

namespace {

__device__ unsigned g_error_word;

// q_i / max(|q_i|, 1e-12) and k_j / max(|k_j|, 1e-12) rounded to fp16 (Key
// design 1 of the notes: rows are L2-normalised before the score product).
// With qmul != 0 query row i (1-based within its head) is also multiplied by
// qmul * ln i, so that the score product yields z = qmul ln i qh.kh directly
// (qmul = +-log2(e) ln d: the length scale in log2 units).  Each row is
// handled by D/16 consecutive threads, 16 elements each: both 16-byte loads
// of a thread are in flight together, so that enough bytes are in flight per
// SM to keep this HBM-bound pass near the copy bandwidth.  Thread 0 also
// zeroes the attention kernel's work counter.
constexpr int kNormElems = 16;   // elements per thread

template <int D>
__global__ void __launch_bounds__(256) normalize_rows_fp16(const __nv_bfloat16 *__restrict__ q,
                                                           const __nv_bfloat16 *__restrict__ k,
                                                           __half *__restrict__ qh,
                                                           __half *__restrict__ kh,
                                                           long long rows, unsigned *counter, int L,
                                                           float qmul) {
    constexpr int G = D / kNormElems;
    // the attention kernel may launch now; it waits for this grid's completion
    // before it reads anything written here
    ptx::launch_dependents();
    const long long tid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (tid == 0) *counter = 0u;
    const long long r = tid / G;
    const int part = (int)(tid % G);
    const bool live = r < 2 * rows;
    const bool is_k = r >= rows;
    const long long rr = is_k ? r - rows : r;
    float x[kNormElems];
    float ss = 0.f;
    if (live) {
        const uint4 *src = reinterpret_cast<const uint4 *>((is_k ? k : q) + rr * D + part * kNormElems);
        uint4 u[2];
        u[0] = src[0];
        u[1] = src[1];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u[c]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(h[e]);
                x[8 * c + 2 * e] = f.x;
                x[8 * c + 2 * e + 1] = f.y;
            }
        }
#pragma unroll
        for (int e = 0; e < kNormElems; ++e) ss = fmaf(x[e], x[e], ss);
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (!live) return;
    float inv = 1.f / fmaxf(sqrtf(ss), 1e-12f);
    if (!is_k && qmul != 0.f) inv *= qmul * logf((float)(rr % L + 1));
    uint4 *dst = reinterpret_cast<uint4 *>((is_k ? kh : qh) + rr * D + part * kNormElems);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
        uint4 u;
        __half2 *h = reinterpret_cast<__half2 *>(&u);
#pragma unroll
        for (int e = 0; e < 4; ++e)
            h[e] = __floats2half2_rn(x[8 * c + 2 * e] * inv, x[8 * c + 2 * e + 1] * inv);
        dst[c] = u;
    }
}

}  // namespace

cudaError_t launch_normalize_fp16(const void *q, const void *k, void *qh, void *kh, long long rows,
                                  int d, unsigned *counter, cudaStream_t stream, int L, float qmul) {
    const long long threads = 2 * rows * (d / kNormElems);
    const long long blocks = (threads + 255) / 256;
    if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    const auto *qb = static_cast<const __nv_bfloat16 *>(q);
    const auto *kb = static_cast<const __nv_bfloat16 *>(k);
    auto *qo = static_cast<__half *>(qh);
    auto *ko = static_cast<__half *>(kh);
    if (d == 64)
        normalize_rows_fp16<64><<<(unsigned)blocks, 256, 0, stream>>>(qb, kb, qo, ko, rows, counter, L, qmul);
    else
        normalize_rows_fp16<128><<<(unsigned)blocks, 256, 0, stream>>>(qb, kb, qo, ko, rows, counter, L, qmul);
    return cudaGetLastError();
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult qr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &qr) == cudaSuccess &&
            qr == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

// [BH, L, D] tensor of 16-bit elements, boxes of 64 elements x 128 rows,
// 128-byte swizzle; rows past L read as zero.
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int BH, int L, int D) {
    auto enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)L, (cuuint64_t)BH};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)L * D * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)tc::kBM, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
std::mutex g_sym_mutex;
unsigned *g_err_ptr[64] = {};
}  // namespace

cudaError_t error_word_ptr(unsigned **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_sym_mutex);
    if (!g_err_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_error_word);
        if (e != cudaSuccess) return e;
        g_err_ptr[dev] = static_cast<unsigned *>(p);
    }
    *out = g_err_ptr[dev];
    return cudaSuccess;
}

namespace {

// Work schedule of the attention kernel for BH heads of n_qtiles Q tiles on
// `grid` CTAs.  Item id i (longest first) is the Q-tile pair m = n_pairs-1 -
// i/BH of head i%BH; its cost is modelled as the K tiles its two Q tiles
// stream, (2m+1) + (2m+2) (one fewer tile when the second is past the end),
// plus one tile of fixed cost.  Two schedules are simulated and the one with
// the shorter makespan is used:
//   longest first: CTA c starts with item c, the rest from the counter;
//   complements:   CTA c starts with item c and its complement h0 - c, where
//                  h0 is the first item that fits next to item 0 within the
//                  mean load; items h0+1.. follow from the counter.
struct Schedule {
    int tail_base = 0;
    std::vector<int> first;   // 2 per CTA, -1 for none
};

Schedule plan_schedule(int BH, int n_qtiles, int grid) {
    const int n_pairs = (n_qtiles + 1) / 2;
    const long long N = (long long)BH * n_pairs;
    auto cost = [&](long long id) {
        const int m = n_pairs - 1 - (int)(id / BH);
        const int qa = 2 * m, qb = 2 * m + 1;
        return (double)(qa + 1) + (qb < n_qtiles ? qb + 1 : 0) + 1.0;
    };
    // makespan of: per-CTA preloaded work, then items [tail, N) longest first
    auto simulate = [&](std::vector<double> load, long long tail) {
        std::priority_queue<std::pair<double, int>, std::vector<std::pair<double, int>>,
                            std::greater<std::pair<double, int>>> heap;
        for (int c = 0; c < grid; ++c) heap.push({load[c], c});
        for (long long i = tail; i < N; ++i) {
            auto t = heap.top();
            heap.pop();
            t.first += cost(i);
            load[t.second] = t.first;
            heap.push(t);
        }
        return *std::max_element(load.begin(), load.end());
    };
    Schedule lpt;
    lpt.first.assign(2 * (size_t)grid, -1);
    std::vector<double> load(grid, 0.0);
    for (int c = 0; c < grid && c < N; ++c) {
        lpt.first[2 * c] = c;
        load[c] = cost(c);
    }
    lpt.tail_base = (int)std::min<long long>(grid, N);
    const double lpt_span = simulate(load, lpt.tail_base);
    double total = 0.0;
    for (long long i = 0; i < N; ++i) total += cost(i);
    const double mean = total / grid;
    long long h0 = -1;
    for (long long h = 1; h < N; ++h)
        if (cost(0) + cost(h) <= mean) {
            h0 = h;
            break;
        }
    if (h0 < 0 || (h0 + 2) / 2 > grid) return lpt;
    Schedule cmp;
    cmp.first.assign(2 * (size_t)grid, -1);
    std::fill(load.begin(), load.end(), 0.0);
    for (long long c = 0; c <= h0 - c; ++c) {
        cmp.first[2 * c] = (int)c;
        load[c] = cost(c);
        if (h0 - c != c) {
            cmp.first[2 * c + 1] = (int)(h0 - c);
            load[c] += cost(h0 - c);
        }
    }
    cmp.tail_base = (int)(h0 + 1);
    return simulate(load, cmp.tail_base) < lpt_span ? cmp : lpt;
}

// Schedules are computed once per (BH, n_qtiles, grid).
std::mutex g_plan_mutex;
std::map<std::tuple<int, int, int>, Schedule> g_plans;

const Schedule &schedule_for(int BH, int n_qtiles, int grid) {
    std::lock_guard<std::mutex> lock(g_plan_mutex);
    const auto key = std::make_tuple(BH, n_qtiles, grid);
    auto it = g_plans.find(key);
    if (it == g_plans.end()) it = g_plans.emplace(key, plan_schedule(BH, n_qtiles, grid)).first;
    return it->second;
}

constexpr size_t kCounterBytes = 256;

size_t qk_bytes(const Problem &pr) {
    return ((size_t)pr.B * pr.H * pr.L * pr.d * 2 + 255) & ~(size_t)255;
}
}  // namespace

// Layout: [work counter, 256 B][normalised q, fp16][normalised k, fp16]; the
// softmax mode needs only the counter.
size_t tc_workspace_bytes(const Problem &pr) {
    if (!uses_normalised_qk(pr.mode)) return kCounterBytes;
    return kCounterBytes + 2 * qk_bytes(pr);
}

cudaError_t launch_tc(const Problem &pr, void *ws, cudaStream_t stream, const Events &ev) {
    const int BH = pr.B * pr.H;
    const long long rows = (long long)BH * pr.L;
    const void *qsrc = pr.q, *ksrc = pr.k;
    CUtensorMapDataType qk_type = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (ev.start && cudaEventRecord(ev.start, stream) != cudaSuccess) return cudaGetLastError();
    unsigned *counter = static_cast<unsigned *>(ws);
    if (!uses_normalised_qk(pr.mode)) {
        cudaError_t e = cudaMemsetAsync(counter, 0, sizeof(unsigned), stream);
        if (e != cudaSuccess) return e;
    } else {
        const size_t half = qk_bytes(pr);
        __half *qh = reinterpret_cast<__half *>(static_cast<char *>(ws) + kCounterBytes);
        __half *kh = reinterpret_cast<__half *>(static_cast<char *>(ws) + kCounterBytes + half);
        // query rows pre-scaled by the length scale (negated for the sigmoid
        // normaliser, whose kernel registers hold -z)
        const float qmul = (pr.mode == kSigmoidRw ? -1.f : 1.f) * score_qmul(pr.d);
        cudaError_t e = launch_normalize_fp16(pr.q, pr.k, qh, kh, rows, pr.d, counter, stream, pr.L, qmul);
        if (e != cudaSuccess) return e;
        qsrc = qh;
        ksrc = kh;
        qk_type = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    }
    CUtensorMap mq, mk, mv;
    if (!make_map(&mq, qsrc, qk_type, BH, pr.L, pr.d) || !make_map(&mk, ksrc, qk_type, BH, pr.L, pr.d) ||
        !make_map(&mv, pr.v, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, BH, pr.L, pr.d))
        return cudaErrorInvalidValue;

    tc::Params prm;
    prm.BH = BH;
    prm.L = pr.L;
    prm.n_qtiles = (pr.L + tc::kBM - 1) / tc::kBM;
    prm.n_pairs = (prm.n_qtiles + 1) / 2;
    prm.n_items = BH * prm.n_pairs;
    prm.ln_d = logf((float)pr.d);
    prm.p = pr.p;
    prm.H = pr.H;
    prm.per_head = pr.p_head ? 1 : 0;
    // LSSAR_EXACT_WEIGHTS=1 keeps every row on the two-transcendental softplus
    // in pass 2 (a cross-check of the one-exponential weights)
    prm.exact_weights = exact_weights_requested() ? 1 : 0;
    for (int h = 0; h < tc::kMaxHeadsP; ++h) prm.p_head[h] = (pr.p_head && h < pr.H) ? pr.p_head[h] : pr.p;
    prm.out = static_cast<__nv_bfloat16 *>(pr.out);
    prm.stats = reinterpret_cast<float4 *>(pr.stats);
    prm.counter = counter;
    cudaError_t e = error_word_ptr(&prm.err);
    if (e != cudaSuccess) return e;
    int sms = 0;
    if ((e = device_sms(&sms)) != cudaSuccess) return e;
    int grid = prm.n_items < sms ? prm.n_items : sms;
    if (grid > tc::kMaxCtas) grid = tc::kMaxCtas;
    const Schedule &sch = schedule_for(BH, prm.n_qtiles, grid);
    prm.tail_base = sch.tail_base;
    for (int c = 0; c < tc::kMaxCtas; ++c) {
        prm.first_items[c][0] = c < grid ? sch.first[2 * c] : -1;
        prm.first_items[c][1] = c < grid ? sch.first[2 * c + 1] : -1;
    }
    if (ev.main && (e = cudaEventRecord(ev.main, stream)) != cudaSuccess) return e;
    e = pr.d == 64 ? tc::dispatch_d64(pr, mq, mk, mv, prm, grid, stream)
                   : tc::dispatch_d128(pr, mq, mk, mv, prm, grid, stream);
    if (e != cudaSuccess) return e;
    if (ev.end) e = cudaEventRecord(ev.end, stream);
    return e;
}

int schedule_plan(int BH, int n_qtiles, int grid, int *first, int *tail_base) {
    if (BH < 1 || n_qtiles < 1 || grid < 1 || grid > tc::kMaxCtas) return -1;
    const Schedule &sch = schedule_for(BH, n_qtiles, grid);
    for (int i = 0; i < 2 * grid; ++i) first[i] = sch.first[i];
    *tail_base = sch.tail_base;
    return 0;
}

bool exact_weights_requested() {
    const char *exact = getenv("LSSAR_EXACT_WEIGHTS");
    return exact != nullptr && exact[0] == '1';
}

cudaError_t read_and_clear_error_word(unsigned int *word) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(word, g_error_word, sizeof(unsigned));
    if (e != cudaSuccess) return e;
    const unsigned zero = 0;
    return cudaMemcpyToSymbol(g_error_word, &zero, sizeof(unsigned));
}

}  // namespace lssar
