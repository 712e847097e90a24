// Launch of the attention-kernel template instances, one translation unit
// per head dimension (tc_d64.cu, tc_d128.cu) so that they compile in parallel.
#pragma once

#include "tc_kernel.cuh"

namespace lssar {
namespace tc {

cudaError_t dispatch_d64(const Problem &pr, const CUtensorMap &mq, const CUtensorMap &mk,
                         const CUtensorMap &mv, const Params &prm, int grid, cudaStream_t s);
cudaError_t dispatch_d128(const Problem &pr, const CUtensorMap &mq, const CUtensorMap &mk,
                          const CUtensorMap &mv, const Params &prm, int grid, cudaStream_t s);

template <int D, int MODE, int PK>
cudaError_t launch_kernel(const CUtensorMap &mq, const CUtensorMap &mk, const CUtensorMap &mv,
                          const Params &prm, int grid, cudaStream_t stream) {
    auto kern = lssar_tc_kernel<D, MODE, PK>;
    constexpr int smem = Cfg<D>::kSmemBytes;
    static PerDeviceOnce once;
    cudaError_t e = per_device_once(once, nullptr, [&](int &) {
        // the kernel moves registers from its control warpgroup to its score
        // warpgroups (setmaxnreg): that split adds up only for a launch at
        // exactly kLaunchRegs registers per thread, so any other allocation
        // is refused here rather than launched
        cudaFuncAttributes attr;
        cudaError_t a = cudaFuncGetAttributes(&attr, kern);
        if (a != cudaSuccess) return a;
        if (attr.numRegs != kLaunchRegs) return cudaErrorInvalidConfiguration;
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    });
    if (e != cudaSuccess) return e;
    // a programmatic dependent of the prologue: the launch and the kernel's
    // setup overlap the prologue's tail (the kernel waits before reading)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(Cfg<D>::kThreads);
    cfg.dynamicSmemBytes = (size_t)smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, prm);
}

// Re-weighting modes: compile-time power chains for p in {1, 2, 3, 15},
// square-and-multiply for any other p.
template <int D, int MODE>
cudaError_t dispatch_p(const Problem &pr, const CUtensorMap &mq, const CUtensorMap &mk,
                       const CUtensorMap &mv, const Params &prm, int grid, cudaStream_t s) {
    if (pr.p_head) return launch_kernel<D, MODE, 0>(mq, mk, mv, prm, grid, s);   // per head
    switch (pr.p) {
        case 1: return launch_kernel<D, MODE, 1>(mq, mk, mv, prm, grid, s);
        case 2: return launch_kernel<D, MODE, 2>(mq, mk, mv, prm, grid, s);
        case 3: return launch_kernel<D, MODE, 3>(mq, mk, mv, prm, grid, s);
        case 15: return launch_kernel<D, MODE, 15>(mq, mk, mv, prm, grid, s);
        default: return launch_kernel<D, MODE, 0>(mq, mk, mv, prm, grid, s);
    }
}

template <int D>
cudaError_t dispatch(const Problem &pr, const CUtensorMap &mq, const CUtensorMap &mk,
                     const CUtensorMap &mv, const Params &prm, int grid, cudaStream_t s) {
    switch (pr.mode) {
        case kSoftmax: return launch_kernel<D, kSoftmax, 0>(mq, mk, mv, prm, grid, s);
        case kLssa: return launch_kernel<D, kLssa, 0>(mq, mk, mv, prm, grid, s);
        case kLssar: return dispatch_p<D, kLssar>(pr, mq, mk, mv, prm, grid, s);
        case kSoftmaxRw: return dispatch_p<D, kSoftmaxRw>(pr, mq, mk, mv, prm, grid, s);
        default: return dispatch_p<D, kSigmoidRw>(pr, mq, mk, mv, prm, grid, s);
    }
}

}  // namespace tc
}  // namespace lssar
