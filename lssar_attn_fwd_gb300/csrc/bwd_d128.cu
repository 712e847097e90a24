// Backward-kernel instances for head dimension 128.
#include "bwd_dispatch.cuh"

namespace lssar {
namespace tcb {

cudaError_t dispatch_d128(const BwdProblem &pr, int pass, const Maps &m, const Params &prm, int grid,
                         cudaStream_t s) {
    return dispatch<128>(pr, pass, m, prm, grid, s);
}

}  // namespace tcb
}  // namespace lssar
