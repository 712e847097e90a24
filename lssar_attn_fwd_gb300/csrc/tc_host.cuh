// Host helpers of the tensor-core path shared by the forward and backward
// launchers (implemented in tc.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>

namespace lssar {

// q_i / max(|q_i|, 1e-12) and k_j likewise, rounded to fp16, for `rows` rows of
// d elements each; also zeroes *counter.  With qmul != 0 query row i (1-based
// within its head of L rows) is also multiplied by qmul * ln i.
cudaError_t launch_normalize_fp16(const void *q, const void *k, void *qh, void *kh, long long rows,
                                  int d, unsigned *counter, cudaStream_t stream, int L = 1, float qmul = 0.f);

// log2(e) * ln d: the query-row multiplier of the normalised modes' scores in
// log2 units (times ln i); the forward, the backward and the CUDA-core
// backward all take it from here so that their fp16 operands agree.
inline float score_qmul(int d) { return 1.4426950408889634f * logf((float)d); }

// TMA map of a [BH, L, D] tensor of 16-bit elements: boxes of 64 elements x
// 128 rows, 128-byte swizzle, rows past L read as zero.
bool make_map(CUtensorMap *m, const void *base, CUtensorMapDataType dt, int BH, int L, int D);

// Device address of the library's error word on the current device.
cudaError_t error_word_ptr(unsigned **out);

}  // namespace lssar
