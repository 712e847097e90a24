// Backward-kernel instances for head dimension 64.
#include "bwd_dispatch.cuh"

namespace lssar {
namespace tcb {

cudaError_t dispatch_d64(const BwdProblem &pr, int pass, const Maps &m, const Params &prm, int grid,
                         cudaStream_t s) {
    return dispatch<64>(pr, pass, m, prm, grid, s);
}

}  // namespace tcb
}  // namespace lssar
