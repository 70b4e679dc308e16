// Internal launchers of the LUT-6 kernels (not part of the C ABI).
#pragma once
#include "common.cuh"

namespace clef {

enum Epilogue : int {
  EPI_F16 = 0,        // y fp16 = acc
  EPI_F32 = 1,        // y fp32 = acc
  EPI_ADD_F32 = 2,    // y fp32 += acc (residual add, in place)
  EPI_SWIGLU_F16 = 3, // y fp16 [m, n/2] = SiLU(gate) * up, gate/up rows interleaved by 16
};

// Workspace of the stream-K part of a launch (see lut6_gemm_launch), on the current device:
// partial sums (fp32, 3 tiles per SM) and the per-tile piece counters (zeroed before first use;
// every launch leaves them zero again).
int64_t lut6_split_part_bytes();
int64_t lut6_split_count_bytes();

// y[m, n] (row stride ldy elements) = x[m, k] . W^T with W in the tiled layout
// (clef_lut6_tile).  Requires n % 16 == 0, k % 64 == 0 (n % 32 == 0 for EPI_SWIGLU_F16), x packed
// [m, k], lut 16-byte aligned.
// With part and counts given (lut6_split_part_bytes / lut6_split_count_bytes, counters zero), a
// launch whose tiles leave the last wave of SMs partly idle runs its full waves data-parallel
// and shares the k-steps of the remaining tiles evenly among all SMs (stream-K): each share
// stores its partial sums and the SM that finishes a tile last adds the tile's pieces in a fixed
// order, so every run gives the same bits.  Without them every tile runs whole on one SM.
clef_status lut6_gemm_launch(const __half* x, const uint8_t* tiled, const __half* lut, void* y,
                             int64_t ldy, int64_t M, int64_t N, int64_t K, int mode,
                             cudaStream_t stream, float* part = nullptr, unsigned* counts = nullptr);

// canonical packed [n, k*3/4] -> tiled layout of the GEMM (same size)
clef_status lut6_tile_launch(const uint8_t* packed, int64_t n, int64_t k, uint8_t* tiled,
                             cudaStream_t stream);

clef_status lut6_dequant_launch(const uint8_t* packed, const __half* lut, int64_t n, int64_t k,
                                __half* w, cudaStream_t stream);

}  // namespace clef
