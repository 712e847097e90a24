// Attention-kernel instances for head dimension 128.
#include "tc_dispatch.cuh"

namespace lssar {
namespace tc {

cudaError_t dispatch_d128(const Problem &pr, const CUtensorMap &mq, const CUtensorMap &mk,
                         const CUtensorMap &mv, const Params &prm, int grid, cudaStream_t s) {
    return dispatch<128>(pr, mq, mk, mv, prm, grid, s);
}

}  // namespace tc
}  // namespace lssar
