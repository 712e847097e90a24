// The one-exponential softplus of the LSSAR weights and the per-row error
// bound that admits it, shared by the forward and the backward tensor-core
// kernels (Key design 1's Softplus, Key design 2's ReLU^p re-weighting).
#pragma once

#include <cuda_runtime.h>

#include "tc_ptx.cuh"

namespace lssar {

// LSSAR weights with one exponential per element.  For z >= 0,
// sp2(z) = z + log2(1 + u) with u = 2^-z, and log2(1 + u) <= u / ln 2 with a
// gap of at most u^2 / (2 ln 2); so z + u / ln 2 overestimates sp2 by at most
// C u^2, C = 1 / (2 ln 2), and never by more than that.  For z < 0 the same
// expression (u = 2^z) stays below 1 / ln 2 < 1.5, so on a row whose threshold
// theta is at least 1.5 those columns get weight 0, as they do exactly
// (sp2(z) < 1 <= theta).  The weight of a column above the threshold with
// exact value y = (sp2(z) - theta) kappa in (0, 1] then moves by at most
// p min(1, y + eta)^(p-1) C kappa u^2, where u <= 2^-(theta + y/kappa - 1)
// (because sp2(z) <= z + 1) and eta = C kappa 2^(-2 (theta - 1)) bounds the
// overestimate; the largest value of that bound over y is taken at
// y* = min(1, (p - 1) kappa / (2 ln 2)).  Columns below the threshold with
// z >= 0 get at most (C kappa)^p.  With at most i columns and a row maximum
// weight of 1 (so sum_j w_j >= 1), the row's weights change in sum by at most
//   R = i p C kappa 2^(2 eta / kappa) y*^(p-1) 2^(-2 (theta + y*/kappa - 1)) + i (C kappa)^p
// relative to their total.  A row takes the one-exponential weights when
// R <= kFastBound; the output then moves by at most 2 R max_j |v_j|.  The
// argument holds for any power of y, so the backward, which also needs
// y^(p-1), asks for the bound at both p and p - 1.
constexpr float kFastBound = 2e-4f;
constexpr float kHalfInvLn2 = 0.72134752044448170f;   // 1 / (2 ln 2)

__device__ __forceinline__ bool fast_weights_ok(float theta, float kappa, float fi, int p) {
    if (!(theta >= 1.5f) || p < 4) return false;
    const float ys = fminf(1.f, (float)(p - 1) * kappa * kHalfInvLn2);
    const float two_eta_k = 2.f * kHalfInvLn2 * ptx::ex2(-2.f * (theta - 1.f));   // 2 eta / kappa
    const float l_i = ptx::lg2(fi);
    const float l_r = l_i + ptx::lg2((float)p * kHalfInvLn2 * kappa) + two_eta_k + (float)(p - 1) * ptx::lg2(ys) -
                      2.f * (theta + ys / kappa - 1.f);
    const float l_c = l_i + (float)p * ptx::lg2(kHalfInvLn2 * kappa);
    return ptx::ex2(l_r) + ptx::ex2(l_c) <= kFastBound;
}

// Whether the one-exponential weights are switched off for every row
// (LSSAR_EXACT_WEIGHTS=1 in the environment, read at each call).
bool exact_weights_requested();

}  // namespace lssar
