// Internal launchers of the LUT-6 kernels (not part of the C ABI).
#pragma once
#include "common.cuh"

namespace clef {

enum Epilogue : int {
  EPI_F16 = 0,        // y fp16 = acc
  EPI_F32 = 1,        // y fp32 = acc
  EPI_ADD_F32 = 2,    // y fp32 += acc (residual add, in place)
  EPI_SWIGLU_F16 = 3, // y fp16 [m, n/2] = SiLU(gate) * up, gate/up rows interleaved by 16
  EPI_PART_F32 = 4,   // (internal) k-part p of a split residual add: part[p][m][n] fp32 = acc
};

// Token tiles per group of the GEMM's tile walk for a reduction length K, epilogue mode and
// tile width (256 or 512 tokens).
int lut6_group_m(int64_t K, int mode, int tile_tokens);

// Whether a launch of M tokens x N channels (no K split) takes the 512-token tiles.
bool lut6_use_wide(int64_t M, int64_t N);

// The number of k-parts a residual-add launch of this shape is split into (1: no split).
int lut6_add_split(int64_t M, int64_t N, int64_t K);

// y[m, n] (row stride ldy elements) = x[m, k] . W^T with W in the tiled layout
// (clef_lut6_tile).  Requires n % 16 == 0, k % 64 == 0 (n % 32 == 0 for EPI_SWIGLU_F16), x packed
// [m, k], lut 16-byte aligned.
// In EPI_ADD_F32 mode with part_ws set and a split launch, the k-parts write their partial
// sums to part_ws ([parts][M][N] fp32, lut6_add_split parts) and one more kernel adds them to y in
// part order: the result is then the same bits on every run (without part_ws the parts add
// straight into y in whatever order they finish).
clef_status lut6_gemm_launch(const __half* x, const uint8_t* tiled, const __half* lut, void* y,
                             int64_t ldy, int64_t M, int64_t N, int64_t K, int mode,
                             cudaStream_t stream, float* part_ws = nullptr);

// canonical packed [n, k*3/4] -> tiled layout of the GEMM (same size)
clef_status lut6_tile_launch(const uint8_t* packed, int64_t n, int64_t k, uint8_t* tiled,
                             cudaStream_t stream);

clef_status lut6_dequant_launch(const uint8_t* packed, const __half* lut, int64_t n, int64_t k,
                                __half* w, cudaStream_t stream);

}  // namespace clef
