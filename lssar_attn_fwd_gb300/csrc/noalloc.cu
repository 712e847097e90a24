// lssar_attn_fwd_noalloc: the tensor-core forward with its scratch in a fixed
// device array instead of a stream-ordered allocation, for callers that
// cannot allow device memory allocation during a call (see the header).
#include <mutex>

#include "lssar_attn_fwd.h"
#include "lssar_internal.cuh"

namespace {

constexpr size_t kScratchBytes = LSSAR_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// One copy per device, held for the life of the process.  Host code must not
// use this name as a device address: the device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mutex;
void *g_scratch[kMaxDevices] = {};

// Device address of the current device's copy of the array, looked up once per
// device with that device current.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LSSAR_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return LSSAR_ERR_CUDA;
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return LSSAR_OK;
}

}  // namespace

extern "C" int lssar_attn_fwd_noalloc(const void *q, const void *k, const void *v, void *out,
                                      int B, int H, int L, int d, int p, int mode,
                                      cudaStream_t stream) {
    lssar::Problem pr;
    int st = lssar::validate_args(q, k, v, out, B, H, L, d, p, mode, &pr);
    if (st != LSSAR_OK) return st;
    if (lssar::tc_workspace_bytes(pr) > kScratchBytes) return LSSAR_ERR_SCRATCH;
    void *ws = nullptr;
    st = scratch_address(&ws);
    if (st != LSSAR_OK) return st;
    // launch_tc zeroes the work counter on `stream` and overwrites the rest.
    return lssar::launch_tc(pr, ws, stream) == cudaSuccess ? LSSAR_OK : LSSAR_ERR_CUDA;
}
