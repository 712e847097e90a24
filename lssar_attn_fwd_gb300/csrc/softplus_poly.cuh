// Softplus in log2 units with the log2 of the small part taken by a
// polynomial on the FMA pipe instead of the MUFU lg2, shared by the forward and
// backward tensor-core kernels.
#pragma once

#include <cuda_runtime.h>

#include "tc_ptx.cuh"

namespace lssar {

// sp2(z) = log2(1 + 2^z) = max(z, 0) + log2(1 + u), u = 2^-|z| in [0, 1], with
// log2(1 + u) ~= u (c1 + u (c2 + ... + u c6)).  The coefficients were fitted
// for this code by minimax (Lawson-weighted least squares) on [0, 1] with the
// constant term fixed at 0, so that a masked column (z = -inf: u = 0) still
// gives exactly 0; the largest error is 2.2e-6 in fp32 Horner arithmetic.
// fit_softplus_poly.py beside this file reproduces them (and fits other degrees).
__device__ __forceinline__ float2 sp2x2_poly(float2 z) {
    const float2 u = make_float2(ptx::ex2(-fabsf(z.x)), ptx::ex2(-fabsf(z.y)));
    float2 h = __ffma2_rn(u, make_float2(-0.02645743452012539f, -0.02645743452012539f),
                          make_float2(0.12345144152641296f, 0.12345144152641296f));
    h = __ffma2_rn(h, u, make_float2(-0.279538094997406f, -0.279538094997406f));
    h = __ffma2_rn(h, u, make_float2(0.458270788192749f, 0.458270788192749f));
    h = __ffma2_rn(h, u, make_float2(-0.7182819247245789f, -0.7182819247245789f));
    h = __ffma2_rn(h, u, make_float2(1.442553162574768f, 1.442553162574768f));
    return __ffma2_rn(h, u, make_float2(fmaxf(z.x, 0.f), fmaxf(z.y, 0.f)));
}

// Whether element pair `idx` (0..15 within a 32-column chunk) takes the
// polynomial path when `k` of every 16 pairs do, spread evenly.
__host__ __device__ constexpr bool poly_pair(int idx, int k) { return (idx * k) % 16 < k; }

}  // namespace lssar
