// C ABI of liblssar_attn_fwd.so: argument validation, the stream-ordered
// scratch pool and dispatch to the kernels.  The declarations and the full
// contract are in include/lssar_attn_fwd.h.
#include <cstdint>
#include <mutex>

#include "lssar_attn_fwd.h"
#include "lssar_internal.cuh"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxP = 1024;
constexpr int kMaxHeadsP = 256;   // = tc::kMaxHeadsP

bool ranges_overlap(const void *a, size_t na, const void *b, size_t nb) {
    const auto x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Pure host checks; never touches the CUDA runtime.
int validate(const void *q, const void *k, const void *v, void *out, int B, int H, int L, int d,
             int p, int mode, lssar::Problem *pr) {
    if (!q || !k || !v || !out) return LSSAR_ERR_NULL;
    if (mode < LSSAR_MODE_SOFTMAX || mode > LSSAR_MODE_SIGMOID_RW) return LSSAR_ERR_MODE;
    if (B < 1 || H < 1 || L < 1 || L > (1 << 24)) return LSSAR_ERR_SHAPE;
    if (d != 64 && d != 128) return LSSAR_ERR_HEADDIM;
    const unsigned long long elems = (unsigned long long)B * H * L * d;
    if (elems > (1ULL << 40)) return LSSAR_ERR_SHAPE;
    const bool reweight = lssar::is_reweight(mode);
    if (reweight && (p < 1 || p > kMaxP)) return LSSAR_ERR_P;
    for (const void *ptr : {q, k, v, static_cast<const void *>(out)})
        if (reinterpret_cast<uintptr_t>(ptr) & 15u) return LSSAR_ERR_ALIGN;
    const size_t bytes = (size_t)elems * 2;
    if (ranges_overlap(out, bytes, q, bytes) || ranges_overlap(out, bytes, k, bytes) ||
        ranges_overlap(out, bytes, v, bytes))
        return LSSAR_ERR_ALIAS;
    *pr = lssar::Problem{q, k, v, out, B, H, L, d, reweight ? p : 1, mode};
    return LSSAR_OK;
}

// One memory pool per device, created on first use and kept for the life of
// the process.  Its release threshold is raised so that freed scratch stays
// cached in the pool instead of going back to the driver at every sync.
std::mutex g_pool_mutex;
cudaMemPool_t g_pools[kMaxDevices] = {};

cudaError_t device_pool(cudaMemPool_t *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_pool_mutex);
    if (!g_pools[dev]) {
        cudaMemPoolProps props = {};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool;
        e = cudaMemPoolCreate(&pool, &props);
        if (e != cudaSuccess) return e;
        uint64_t keep = UINT64_MAX;
        e = cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        if (e != cudaSuccess) {
            cudaMemPoolDestroy(pool);
            return e;
        }
        g_pools[dev] = pool;
    }
    *out = g_pools[dev];
    return cudaSuccess;
}

int run_tc(const void *q, const void *k, const void *v, void *out, int B, int H, int L, int d,
           int p, int mode, cudaStream_t stream, const lssar::Events &ev, float *stats = nullptr) {
    lssar::Problem pr;
    const int st = validate(q, k, v, out, B, H, L, d, p, mode, &pr);
    if (st != LSSAR_OK) return st;
    pr.stats = stats;
    const size_t ws_bytes = lssar::tc_workspace_bytes(pr);
    void *ws = nullptr;
    if (ws_bytes) {
        cudaMemPool_t pool;
        if (device_pool(&pool) != cudaSuccess) return LSSAR_ERR_CUDA;
        if (cudaMallocFromPoolAsync(&ws, ws_bytes, pool, stream) != cudaSuccess) return LSSAR_ERR_CUDA;
    }
    const cudaError_t e = lssar::launch_tc(pr, ws, stream, ev);
    if (ws && cudaFreeAsync(ws, stream) != cudaSuccess) return LSSAR_ERR_CUDA;
    return e == cudaSuccess ? LSSAR_OK : LSSAR_ERR_CUDA;
}

// Checks of a host array of per-head exponents (pure host).
int check_heads_p(const int *p_per_head, int H, int mode) {
    if (!p_per_head) return LSSAR_ERR_NULL;
    if (!lssar::is_reweight(mode)) {
        if (mode < LSSAR_MODE_SOFTMAX || mode > LSSAR_MODE_SIGMOID_RW) return LSSAR_ERR_MODE;
        return LSSAR_ERR_P;   // per-head exponents need a re-weighting mode
    }
    if (H < 1) return LSSAR_ERR_SHAPE;
    if (H > kMaxHeadsP) return LSSAR_ERR_P;
    for (int h = 0; h < H; ++h)
        if (p_per_head[h] < 1 || p_per_head[h] > kMaxP) return LSSAR_ERR_P;
    return LSSAR_OK;
}

// Checks of the backward's arguments (pure host).
int validate_bwd(const void *q, const void *k, const void *v, const void *dout, const float *stats,
                 void *dq, void *dk, void *dv, int B, int H, int L, int d, int p, int mode,
                 lssar::BwdProblem *bp) {
    if (!stats || !dq || !dk || !dv) return LSSAR_ERR_NULL;
    lssar::Problem pr;
    // the forward's checks cover q, k, v and dout (dout in the place of out)
    const int st = validate(q, k, v, const_cast<void *>(dout), B, H, L, d, p, mode, &pr);
    if (st != LSSAR_OK) return st;
    for (const void *ptr : {static_cast<const void *>(stats), static_cast<const void *>(dq),
                            static_cast<const void *>(dk), static_cast<const void *>(dv)})
        if (reinterpret_cast<uintptr_t>(ptr) & 15u) return LSSAR_ERR_ALIGN;
    const size_t bytes = (size_t)B * H * L * d * 2, sbytes = (size_t)B * H * L * 16;
    const void *outs[3] = {dq, dk, dv};
    for (int a = 0; a < 3; ++a) {
        for (const void *in : {q, k, v, dout})
            if (ranges_overlap(outs[a], bytes, in, bytes)) return LSSAR_ERR_ALIAS;
        if (ranges_overlap(outs[a], bytes, stats, sbytes)) return LSSAR_ERR_ALIAS;
        for (int b = a + 1; b < 3; ++b)
            if (ranges_overlap(outs[a], bytes, outs[b], bytes)) return LSSAR_ERR_ALIAS;
    }
    *bp = lssar::BwdProblem{q, k, v, dout, stats, dq, dk, dv, B, H, L, d, pr.p, mode};
    return LSSAR_OK;
}

}  // namespace

int lssar::validate_args(const void *q, const void *k, const void *v, void *out, int B, int H,
                         int L, int d, int p, int mode, lssar::Problem *pr) {
    return validate(q, k, v, out, B, H, L, d, p, mode, pr);
}

extern "C" {

int lssar_attn_fwd(const void *q, const void *k, const void *v, void *out, int B, int H, int L,
                   int d, int p, int mode, cudaStream_t stream) {
    return run_tc(q, k, v, out, B, H, L, d, p, mode, stream, lssar::Events());
}

int lssar_attn_fwd_profiled(const void *q, const void *k, const void *v, void *out, int B, int H,
                            int L, int d, int p, int mode, cudaStream_t stream,
                            cudaEvent_t ev_start, cudaEvent_t ev_main, cudaEvent_t ev_end) {
    lssar::Events ev;
    ev.start = ev_start;
    ev.main = ev_main;
    ev.end = ev_end;
    return run_tc(q, k, v, out, B, H, L, d, p, mode, stream, ev);
}

int lssar_attn_fwd_train(const void *q, const void *k, const void *v, void *out, float *stats,
                         int B, int H, int L, int d, int p, int mode, cudaStream_t stream) {
    if (!stats) return LSSAR_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(stats) & 15u) return LSSAR_ERR_ALIGN;
    if (B >= 1 && H >= 1 && L >= 1 && (d == 64 || d == 128)) {
        const size_t bytes = (size_t)B * H * L * d * 2, sbytes = (size_t)B * H * L * 16;
        for (const void *t : {q, k, v, static_cast<const void *>(out)})
            if (t && ranges_overlap(stats, sbytes, t, bytes)) return LSSAR_ERR_ALIAS;
    }
    return run_tc(q, k, v, out, B, H, L, d, p, mode, stream, lssar::Events(), stats);
}

int lssar_attn_bwd(const void *q, const void *k, const void *v, const void *dout, const float *stats,
                   void *dq, void *dk, void *dv, int B, int H, int L, int d, int p, int mode,
                   cudaStream_t stream) {
    lssar::BwdProblem bp;
    const int st = validate_bwd(q, k, v, dout, stats, dq, dk, dv, B, H, L, d, p, mode, &bp);
    if (st != LSSAR_OK) return st;
    cudaMemPool_t pool;
    if (device_pool(&pool) != cudaSuccess) return LSSAR_ERR_CUDA;
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, lssar::bwd_tc_workspace_bytes(bp), pool, stream) != cudaSuccess)
        return LSSAR_ERR_CUDA;
    const cudaError_t e = lssar::launch_bwd_tc(bp, ws, stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess) return LSSAR_ERR_CUDA;
    return e == cudaSuccess ? LSSAR_OK : LSSAR_ERR_CUDA;
}

int lssar_attn_fwd_train_heads_p(const void *q, const void *k, const void *v, void *out, float *stats,
                                 int B, int H, int L, int d, const int *p_per_head, int mode,
                                 cudaStream_t stream) {
    const int hst = check_heads_p(p_per_head, H, mode);
    if (hst != LSSAR_OK) return hst;
    if (!stats) return LSSAR_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(stats) & 15u) return LSSAR_ERR_ALIGN;
    lssar::Problem pr;
    const int st = validate(q, k, v, out, B, H, L, d, p_per_head[0], mode, &pr);
    if (st != LSSAR_OK) return st;
    const size_t bytes = (size_t)B * H * L * d * 2, sbytes = (size_t)B * H * L * 16;
    for (const void *t : {q, k, v, static_cast<const void *>(out)})
        if (ranges_overlap(stats, sbytes, t, bytes)) return LSSAR_ERR_ALIAS;
    pr.p_head = p_per_head;
    pr.stats = stats;
    cudaMemPool_t pool;
    if (device_pool(&pool) != cudaSuccess) return LSSAR_ERR_CUDA;
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, lssar::tc_workspace_bytes(pr), pool, stream) != cudaSuccess)
        return LSSAR_ERR_CUDA;
    const cudaError_t e = lssar::launch_tc(pr, ws, stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess) return LSSAR_ERR_CUDA;
    return e == cudaSuccess ? LSSAR_OK : LSSAR_ERR_CUDA;
}

int lssar_attn_bwd_heads_p(const void *q, const void *k, const void *v, const void *dout,
                           const float *stats, void *dq, void *dk, void *dv, int B, int H, int L,
                           int d, const int *p_per_head, int mode, cudaStream_t stream) {
    const int hst = check_heads_p(p_per_head, H, mode);
    if (hst != LSSAR_OK) return hst;
    lssar::BwdProblem bp;
    const int st = validate_bwd(q, k, v, dout, stats, dq, dk, dv, B, H, L, d, p_per_head[0], mode, &bp);
    if (st != LSSAR_OK) return st;
    bp.p_head = p_per_head;
    cudaMemPool_t pool;
    if (device_pool(&pool) != cudaSuccess) return LSSAR_ERR_CUDA;
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, lssar::bwd_tc_workspace_bytes(bp), pool, stream) != cudaSuccess)
        return LSSAR_ERR_CUDA;
    const cudaError_t e = lssar::launch_bwd_tc(bp, ws, stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess) return LSSAR_ERR_CUDA;
    return e == cudaSuccess ? LSSAR_OK : LSSAR_ERR_CUDA;
}

int lssar_attn_bwd_simt(const void *q, const void *k, const void *v, const void *dout,
                        const float *stats, void *dq, void *dk, void *dv, int B, int H, int L,
                        int d, int p, int mode, cudaStream_t stream) {
    lssar::BwdProblem bp;
    const int st = validate_bwd(q, k, v, dout, stats, dq, dk, dv, B, H, L, d, p, mode, &bp);
    if (st != LSSAR_OK) return st;
    cudaMemPool_t pool;
    if (device_pool(&pool) != cudaSuccess) return LSSAR_ERR_CUDA;
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, lssar::bwd_simt_workspace_bytes(bp), pool, stream) != cudaSuccess)
        return LSSAR_ERR_CUDA;
    const cudaError_t e = lssar::launch_bwd_simt(bp, ws, stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess) return LSSAR_ERR_CUDA;
    return e == cudaSuccess ? LSSAR_OK : LSSAR_ERR_CUDA;
}

int lssar_attn_fwd_heads_p(const void *q, const void *k, const void *v, void *out, int B, int H,
                           int L, int d, const int *p_per_head, int mode, cudaStream_t stream) {
    const int hst = check_heads_p(p_per_head, H, mode);
    if (hst != LSSAR_OK) return hst;
    lssar::Problem pr;
    const int st = validate(q, k, v, out, B, H, L, d, p_per_head[0], mode, &pr);
    if (st != LSSAR_OK) return st;
    pr.p_head = p_per_head;
    const size_t ws_bytes = lssar::tc_workspace_bytes(pr);
    void *ws = nullptr;
    cudaMemPool_t pool;
    if (device_pool(&pool) != cudaSuccess) return LSSAR_ERR_CUDA;
    if (cudaMallocFromPoolAsync(&ws, ws_bytes, pool, stream) != cudaSuccess) return LSSAR_ERR_CUDA;
    const cudaError_t e = lssar::launch_tc(pr, ws, stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess) return LSSAR_ERR_CUDA;
    return e == cudaSuccess ? LSSAR_OK : LSSAR_ERR_CUDA;
}

int lssar_attn_decode(const void *q, const void *k_cache, const void *v_cache, void *out, int B,
                      int H, int L, int d, int p, int mode, cudaStream_t stream) {
    if (!q || !k_cache || !v_cache || !out) return LSSAR_ERR_NULL;
    if (mode < LSSAR_MODE_SOFTMAX || mode > LSSAR_MODE_SIGMOID_RW) return LSSAR_ERR_MODE;
    if (B < 1 || H < 1 || L < 1 || L > (1 << 24)) return LSSAR_ERR_SHAPE;
    if (d != 64 && d != 128) return LSSAR_ERR_HEADDIM;
    const unsigned long long cache_elems = (unsigned long long)B * H * L * d;
    if (cache_elems > (1ULL << 40)) return LSSAR_ERR_SHAPE;
    const bool reweight = lssar::is_reweight(mode);
    if (reweight && (p < 1 || p > kMaxP)) return LSSAR_ERR_P;
    for (const void *ptr : {q, k_cache, v_cache, static_cast<const void *>(out)})
        if (reinterpret_cast<uintptr_t>(ptr) & 15u) return LSSAR_ERR_ALIGN;
    const size_t row_bytes = (size_t)B * H * d * 2, cache_bytes = (size_t)cache_elems * 2;
    if (ranges_overlap(out, row_bytes, q, row_bytes) || ranges_overlap(out, row_bytes, k_cache, cache_bytes) ||
        ranges_overlap(out, row_bytes, v_cache, cache_bytes))
        return LSSAR_ERR_ALIAS;
    lssar::DecodeProblem pr{q, k_cache, v_cache, out, B, H, L, d, reweight ? p : 1, mode};
    int sms = 0;
    if (lssar::device_sms(&sms) != cudaSuccess) return LSSAR_ERR_CUDA;
    cudaMemPool_t pool;
    if (device_pool(&pool) != cudaSuccess) return LSSAR_ERR_CUDA;
    void *ws = nullptr;
    if (cudaMallocFromPoolAsync(&ws, lssar::decode_workspace_bytes(B * H, L, d, sms), pool, stream) !=
        cudaSuccess)
        return LSSAR_ERR_CUDA;
    const cudaError_t e = lssar::launch_decode(pr, ws, stream);
    if (cudaFreeAsync(ws, stream) != cudaSuccess) return LSSAR_ERR_CUDA;
    return e == cudaSuccess ? LSSAR_OK : LSSAR_ERR_CUDA;
}

int lssar_decode_plan(int B, int H, int L, int d, int *path, int *launches, int *chunks, int *chunk_rows) {
    if (B < 1 || H < 1 || L < 1 || L > (1 << 24)) return LSSAR_ERR_SHAPE;
    if (d != 64 && d != 128) return LSSAR_ERR_HEADDIM;
    if ((unsigned long long)B * H * L * d > (1ULL << 40)) return LSSAR_ERR_SHAPE;
    lssar::DecodeRoute r;
    if (lssar::decode_route(B * H, L, d, &r) != cudaSuccess) return LSSAR_ERR_CUDA;
    if (path) *path = r.path;
    if (launches) *launches = r.path == lssar::kDecodeSplit ? 3 : 1;
    if (chunks) *chunks = r.chunks;
    if (chunk_rows) *chunk_rows = r.chunk_rows;
    return LSSAR_OK;
}

int lssar_attn_fwd_simt(const void *q, const void *k, const void *v, void *out, int B, int H,
                        int L, int d, int p, int mode, cudaStream_t stream) {
    lssar::Problem pr;
    const int st = validate(q, k, v, out, B, H, L, d, p, mode, &pr);
    if (st != LSSAR_OK) return st;
    return lssar::launch_simt(pr, stream) == cudaSuccess ? LSSAR_OK : LSSAR_ERR_CUDA;
}

int lssar_schedule_plan(int BH, int n_qtiles, int grid, int *first, int *tail_base) {
    if (!first || !tail_base) return LSSAR_ERR_NULL;
    return lssar::schedule_plan(BH, n_qtiles, grid, first, tail_base) == 0 ? LSSAR_OK : LSSAR_ERR_SHAPE;
}

int lssar_selftest_stall(cudaStream_t stream) {
    // B=1 H=4 L=512 d=64, zero inputs, from the pool
    const int B = 1, H = 4, L = 512, d = 64;
    const size_t cache = (size_t)B * H * L * d * 2;
    int sms = 0;
    if (lssar::device_sms(&sms) != cudaSuccess) return LSSAR_ERR_CUDA;
    const size_t ws_bytes = lssar::decode_workspace_bytes(B * H, L, d, sms);
    cudaMemPool_t pool;
    if (device_pool(&pool) != cudaSuccess) return LSSAR_ERR_CUDA;
    void *buf = nullptr;
    // [q: B*H*d bf16][k cache][v cache][out: B*H*d bf16][decode scratch], 1 KiB-aligned parts
    const size_t qbytes = (size_t)B * H * d * 2;
    const size_t off_k = 1024, off_v = off_k + cache, off_o = off_v + cache, off_ws = off_o + 1024;
    if (qbytes > 1024) return LSSAR_ERR_SHAPE;
    if (cudaMallocFromPoolAsync(&buf, off_ws + ws_bytes, pool, stream) != cudaSuccess) return LSSAR_ERR_CUDA;
    char *b = static_cast<char *>(buf);
    cudaError_t e = cudaMemsetAsync(b, 0, off_ws, stream);
    if (e == cudaSuccess) {
        lssar::DecodeProblem pr{b, b + off_k, b + off_v, b + off_o, B, H, L, d, 3, LSSAR_MODE_LSSAR};
        e = lssar::launch_decode(pr, b + off_ws, stream, true);
    }
    if (cudaFreeAsync(buf, stream) != cudaSuccess) return LSSAR_ERR_CUDA;
    return e == cudaSuccess ? LSSAR_OK : LSSAR_ERR_CUDA;
}

const char *lssar_status_string(int status) {
    switch (status) {
        case LSSAR_OK: return "ok";
        case LSSAR_ERR_NULL: return "null tensor pointer";
        case LSSAR_ERR_SHAPE: return "invalid shape (B, H >= 1, 1 <= L <= 2^24, B*H*L*d <= 2^40)";
        case LSSAR_ERR_HEADDIM: return "head dimension must be 64 or 128";
        case LSSAR_ERR_P: return "re-weighting exponent p must be in 1..1024";
        case LSSAR_ERR_MODE: return "unknown mode";
        case LSSAR_ERR_ALIGN: return "tensor pointer not 16-byte aligned";
        case LSSAR_ERR_CUDA: return "CUDA error";
        case LSSAR_ERR_ALIAS: return "an output overlaps an input or another output";
        case LSSAR_ERR_SCRATCH: return "problem needs more scratch than the fixed no-alloc array";
        default: return "unknown status";
    }
}

int lssar_device_error_word(unsigned int *word) {
    if (!word) return LSSAR_ERR_NULL;
    return lssar::read_and_clear_error_word(word) == cudaSuccess ? LSSAR_OK : LSSAR_ERR_CUDA;
}

int lssar_abi_version(void) { return 10000; }

}  // extern "C"
