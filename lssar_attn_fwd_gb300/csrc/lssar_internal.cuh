// Internal declarations shared by the translation units of liblssar_attn_fwd.so.
#pragma once

#include <cstdint>
#include <mutex>
#include <cuda_runtime.h>

namespace lssar {

enum Mode : int { kSoftmax = 0, kLssa = 1, kLssar = 2, kSoftmaxRw = 3, kSigmoidRw = 4 };

// Modes that end with the re-weighting step (and take the exponent p).
__host__ __device__ constexpr bool is_reweight(int mode) { return mode == kLssar || mode == kSoftmaxRw || mode == kSigmoidRw; }
// Modes whose scores use L2-normalised q, k (prepared by the prologue).
__host__ __device__ constexpr bool uses_normalised_qk(int mode) { return mode == kLssa || mode == kLssar || mode == kSigmoidRw; }

// Device-side checks of the debug build (compiled with -DLSSAR_DEBUG_CHECKS;
// in the default build they compile to nothing): a failed check records its
// code in the device error word and returns false, and the caller skips the
// access it guards (a skipped copy makes its wait run out, which the bounded
// waits turn into an error code; nothing traps).
enum : unsigned {
    kDbgTma = 101,      // a tensor-copy coordinate outside the tensor or misaligned
    kDbgTmem = 102,     // a TMEM lane or column range outside the allocation
    kDbgGlobal = 103,   // a global load or store index outside its tensor
    kDbgItem = 104,     // a work item outside the schedule
    kDbgBulk = 105      // a bulk copy outside its source or misaligned
};

__device__ __forceinline__ bool dcheck(bool ok, unsigned *err, unsigned code) {
#ifdef LSSAR_DEBUG_CHECKS
    if (!ok) atomicCAS(err, 0u, code);
    return ok;
#else
    (void)ok;
    (void)err;
    (void)code;
    return true;
#endif
}

// TMEM address (lane << 16 | column) of a `width`-column access relative to an
// allocation of `alloc` columns at `base`: lane below 128, columns inside.
__device__ __forceinline__ bool tmem_in_range(uint32_t addr, uint32_t base, uint32_t width, uint32_t alloc) {
    const uint32_t lane = addr >> 16, col = (addr & 0xFFFFu) - (base & 0xFFFFu);
    return lane < 128u && col + width <= alloc;
}

// Problem description after validation.  Tensors are [B, H, L, d] bf16.
struct Problem {
    const void *q;
    const void *k;
    const void *v;
    void *out;
    int B, H, L, d, p, mode;
    const int *p_head = nullptr;   // host array of H exponents, or null (one p for all heads)
    float *stats = nullptr;        // [B, H, L, 4] row statistics for the backward pass, or null
};

// Host-side argument checks of the C ABI (no CUDA call); LSSAR_OK or a
// negative status.  Fills *pr on success (p_head left null).
int validate_args(const void *q, const void *k, const void *v, void *out, int B, int H, int L,
                  int d, int p, int mode, Problem *pr);

// Plain CUDA-core kernel (one warp per query row).  Returns a cudaError_t.
cudaError_t launch_simt(const Problem &pr, cudaStream_t stream);

// Optional events recorded around the kernels of one call (NULL = skipped).
struct Events {
    cudaEvent_t start = nullptr;  // before the normalisation prologue
    cudaEvent_t main = nullptr;   // before the attention kernel
    cudaEvent_t end = nullptr;    // after the attention kernel
};

// Tensor-core path (tcgen05 + TMEM + TMA).  `ws` is device scratch of at
// least tc_workspace_bytes(pr) bytes, 256-byte aligned.
size_t tc_workspace_bytes(const Problem &pr);
cudaError_t launch_tc(const Problem &pr, void *ws, cudaStream_t stream, const Events &ev = Events());

// Backward pass: gradients of sum(dout * out) for q, k, v, from the forward's
// per-row statistics {m, kappa, beta, W} (float4 per row).
struct BwdProblem {
    const void *q, *k, *v, *dout;
    const float *stats;
    void *dq, *dk, *dv;
    int B, H, L, d, p, mode;
    const int *p_head = nullptr;   // host array of H exponents, or null (one p for all heads)
};
// Plain CUDA-core backward; ws holds bwd_simt_workspace_bytes(pr) bytes.
size_t bwd_simt_workspace_bytes(const BwdProblem &pr);
cudaError_t launch_bwd_simt(const BwdProblem &pr, void *ws, cudaStream_t stream);
// Tensor-core backward (row pass, column pass, normalisation gradient); ws
// holds bwd_tc_workspace_bytes(pr) bytes, 256-byte aligned.
size_t bwd_tc_workspace_bytes(const BwdProblem &pr);
cudaError_t launch_bwd_tc(const BwdProblem &pr, void *ws, cudaStream_t stream);
// Decode: one query row per head (position L) against a K/V cache of L rows.
struct DecodeProblem {
    const void *q;   // [B, H, d]
    const void *k;   // [B, H, L, d]
    const void *v;   // [B, H, L, d]
    void *out;       // [B, H, d]
    int B, H, L, d, p, mode;
};
size_t decode_workspace_bytes(int BH, int L, int d, int sms);
// The path a decode step takes on the current device: one launch with a
// thread-block cluster per head, one cooperative launch, or three launches;
// each head's cache in `chunks` pieces of `chunk_rows` keys (the last one
// shorter).
enum { kDecodeCluster = 0, kDecodeGrid = 1, kDecodeSplit = 2 };
struct DecodeRoute {
    int path, chunks, chunk_rows;
};
cudaError_t decode_route(int BH, int L, int d, DecodeRoute *route);
// withhold_copies: self-test of the failure path (the one-launch kernel issues
// no copies, every wait of the launch runs into its bound).
cudaError_t launch_decode(const DecodeProblem &pr, void *ws, cudaStream_t stream, bool withhold_copies = false);

// Launch-time setup that only has to happen once per device (function
// attributes, occupancy queries): `fn(v)` returns a cudaError_t and stores
// what it found in v; the first successful result is kept.
struct PerDeviceOnce {
    static constexpr int kMaxDevices = 64;
    std::mutex mu;
    bool done[kMaxDevices] = {};
    int value[kMaxDevices] = {};
};

template <class F>
cudaError_t per_device_once(PerDeviceOnce &once, int *value, F &&fn) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= PerDeviceOnce::kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(once.mu);
    if (!once.done[dev]) {
        int v = 0;
        e = fn(v);
        if (e != cudaSuccess) return e;
        once.value[dev] = v;
        once.done[dev] = true;
    }
    if (value) *value = once.value[dev];
    return cudaSuccess;
}

// Number of SMs of the current device (queried once per device).
inline cudaError_t device_sms(int *sms) {
    static PerDeviceOnce once;
    return per_device_once(once, sms, [](int &v) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        return e != cudaSuccess ? e : cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    });
}

// The attention kernel's work schedule for BH heads of n_qtiles Q tiles on
// `grid` CTAs (host only): first[2c], first[2c+1] = the fixed items of CTA c
// (-1: none), *tail_base = the first item handed out by the counter.
int schedule_plan(int BH, int n_qtiles, int grid, int *first, int *tail_base);

// Reads and clears the device error word of the current device.
cudaError_t read_and_clear_error_word(unsigned int *word);

}  // namespace lssar
