// Launch of the backward-kernel template instances, one translation unit per
// head dimension (bwd_d64.cu, bwd_d128.cu) so that they compile in parallel.
#pragma once

#include "bwd_kernel.cuh"

namespace lssar {
namespace tcb {

// The four tensor maps in the roles of the pass: anchor tiles X1 (score
// operand) and X2 (bf16), streamed tiles Y1 (score operand) and Y2 (bf16).
struct Maps {
    CUtensorMap x1, x2, y1, y2;
};

cudaError_t dispatch_d64(const BwdProblem &pr, int pass, const Maps &m, const Params &prm, int grid,
                         cudaStream_t s);
cudaError_t dispatch_d128(const BwdProblem &pr, int pass, const Maps &m, const Params &prm, int grid,
                          cudaStream_t s);

template <int D, int MODE, int PK, int PASS>
cudaError_t launch_kernel(const Maps &m, const Params &prm, int grid, cudaStream_t stream) {
    auto kern = lssar_bwd_kernel<D, MODE, PK, PASS>;
    constexpr int smem = Cfg<D>::kSmemBytes;
    static PerDeviceOnce once;
    cudaError_t e = per_device_once(once, nullptr, [&](int &) {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    // a programmatic dependent of the kernel before it (the prologue, or the
    // row pass for the column pass): the launch and the kernel's setup overlap
    // that kernel's tail (the kernel waits before it reads anything)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Tmem<D, PASS>::kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, m.x1, m.x2, m.y1, m.y2, prm);
}

// Re-weighting modes: fixed power chains for p = 3 and 15, square-and-multiply otherwise.
template <int D, int MODE, int PASS>
cudaError_t dispatch_p(const BwdProblem &pr, const Maps &m, const Params &prm, int grid, cudaStream_t s) {
    if (pr.p_head) return launch_kernel<D, MODE, 0, PASS>(m, prm, grid, s);   // per head
    switch (pr.p) {
        case 3: return launch_kernel<D, MODE, 3, PASS>(m, prm, grid, s);
        case 15: return launch_kernel<D, MODE, 15, PASS>(m, prm, grid, s);
        default: return launch_kernel<D, MODE, 0, PASS>(m, prm, grid, s);
    }
}

template <int D, int PASS>
cudaError_t dispatch_mode(const BwdProblem &pr, const Maps &m, const Params &prm, int grid, cudaStream_t s) {
    switch (pr.mode) {
        case kSoftmax: return launch_kernel<D, kSoftmax, 0, PASS>(m, prm, grid, s);
        case kLssa: return launch_kernel<D, kLssa, 0, PASS>(m, prm, grid, s);
        case kLssar: return dispatch_p<D, kLssar, PASS>(pr, m, prm, grid, s);
        case kSoftmaxRw: return dispatch_p<D, kSoftmaxRw, PASS>(pr, m, prm, grid, s);
        default: return dispatch_p<D, kSigmoidRw, PASS>(pr, m, prm, grid, s);
    }
}

template <int D>
cudaError_t dispatch(const BwdProblem &pr, int pass, const Maps &m, const Params &prm, int grid,
                     cudaStream_t s) {
    return pass == kRowPass ? dispatch_mode<D, kRowPass>(pr, m, prm, grid, s)
                            : dispatch_mode<D, kColPass>(pr, m, prm, grid, s);
}

}  // namespace tcb
}  // namespace lssar
