// Internal launchers of the memory-bound glue kernels (not part of the C ABI).
#pragma once
#include "common.cuh"

namespace clef {

// x [M, 4096] fp32 = table[ids] (fp16 rows widened); ids outside [0, vocab) give zero rows and
// set the device status to DEV_BAD_TOKEN.
clef_status embed_launch(const int32_t* ids, const __half* table, int64_t vocab, float* x,
                         int64_t M, cudaStream_t stream);

// Picture rows: rows start .. start + n - 1 of each of B requests of L tokens in the fp32 residual
// x take rows [b][0 .. n) of `rows` (fp16 [B][n][4096]) in place of the embedding rows.
clef_status image_rows_launch(const __half* rows, float* x, int64_t B, int64_t L, int64_t start,
                              int64_t n, cudaStream_t stream);

// y [M, 4096] fp16 = x * rsqrt(mean(x^2) + 1e-6) * w.  With check_finite (the final norm), rows
// whose residual or output is not finite are reported (DEV_NONFINITE_HIDDEN, lowest row kept).
clef_status rmsnorm_launch(const float* x, const __half* w, __half* y, int64_t M,
                           cudaStream_t stream, bool check_finite = false);

// Rows of an fp16 [rows, cols] array (cols % 8 == 0) holding an inf or a NaN: flags[row] = 1 / 0
// (flags may be NULL), the lowest such row reported as by the final norm.
clef_status check_finite_launch(const __half* x, int64_t rows, int64_t cols, uint8_t* flags,
                                cudaStream_t stream);

// [a | b] = xn [M, 4096] . W_ab^T, W_ab [64, 4096] fp16 (tensor cores), then the GDN gates
// g [M, 32] = log(alpha) = -exp(A_log) softplus(a + dt_bias) (>= -30), beta [M, 32] = sigmoid(b).
// When M is small the K dimension is split over up to kAbMaxSlices CTAs per token block; their
// partial sums go to `part` (ab_proj_scratch_bytes(M) bytes) and are added in a fixed order.
constexpr int kAbMaxSlices = 8;
size_t ab_proj_scratch_bytes(int64_t M);
clef_status ab_proj_launch(const __half* xn, const __half* w_ab, const __half* A_log,
                           const __half* dt_bias, float* g, float* beta, float* part, int64_t M,
                           cudaStream_t stream);

}  // namespace clef
