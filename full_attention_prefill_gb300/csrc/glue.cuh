// Internal launchers of the memory-bound glue kernels (not part of the C ABI).
#pragma once
#include "common.cuh"

namespace clef {

// x [M, 4096] fp32 = table[ids] (fp16 rows widened); ids outside [0, vocab) give zero rows and
// set the device status to DEV_BAD_TOKEN.
clef_status embed_launch(const int32_t* ids, const __half* table, int64_t vocab, float* x,
                         int64_t M, cudaStream_t stream);

// y [M, 4096] fp16 = x * rsqrt(mean(x^2) + 1e-6) * w.
clef_status rmsnorm_launch(const float* x, const __half* w, __half* y, int64_t M,
                           cudaStream_t stream);

// [a | b] = xn [M, 4096] . W_ab^T, W_ab [64, 4096] fp16 (tensor cores), then the GDN gates
// g [M, 32] = log(alpha) = -exp(A_log) softplus(a + dt_bias) (>= -30), beta [M, 32] = sigmoid(b).
clef_status ab_proj_launch(const __half* xn, const __half* w_ab, const __half* A_log,
                           const __half* dt_bias, float* g, float* beta, int64_t M,
                           cudaStream_t stream);

}  // namespace clef
