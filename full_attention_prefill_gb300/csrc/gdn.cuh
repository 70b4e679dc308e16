// Internal launchers of the Gated DeltaNet kernels (not part of the C ABI).
#pragma once
#include "common.cuh"

namespace clef {

namespace gdn {
constexpr int C = 64;          // chunk width
constexpr int D = 128;         // head size (key and value)
constexpr int HV = 32;         // value heads
constexpr int HK = 16;         // key heads
}  // namespace gdn

// conv(4) + SiLU + q/k L2 norm, for M tokens of request chunks of L positions.  Taps before a
// chunk's first position read conv_in [B][3][8192] (the carried last three rows of the conv
// input, oldest first), or zero when conv_in is NULL.
clef_status gdn_prep_launch(const __half* proj, int64_t ldp, const __half* conv_w,
                            const __half* conv_in, __half* q, __half* k, __half* v, int64_t M,
                            int64_t L, cudaStream_t stream);

// state [B][3][8192] <- the last three rows of the conv input (carried rows, then the chunk's L
// rows of proj q | k | v), in place.
clef_status conv_state_launch(const __half* proj, int64_t ldp, __half* state, int64_t B,
                              int64_t L, cudaStream_t stream);

// with_norm: room for o before the output gate (decoder layer path, z != NULL)
size_t gdn_scan_workspace_bytes(int64_t B, int64_t L, bool with_norm);
// Pieces a scan of B requests of L positions runs in (1: one chunk phase, one state pass).
int gdn_pieces(int64_t B, int64_t L);

// The chunked scan.  Exactly one of g (log alpha) / alpha is non-NULL.  With z != NULL the
// output is the z-gated RMSNorm (weight o_norm) of o; otherwise o itself.  out [M, ldo] fp16.
clef_status gdn_scan_launch(const __half* q, const __half* k, const __half* v, const float* g,
                            const float* alpha, const float* beta, const float* s0, float* s_out,
                            const __half* z, int64_t ldz, const __half* o_norm, __half* out,
                            int64_t ldo, int64_t B, int64_t L, void* ws, cudaStream_t stream);

// The sequential state pass on tcgen05 (gdn_state.cu).  Inputs are the chunk phase's outputs,
// one block per (chunk, head) in [B * nch, 32] order: W and decayed keys Kd [64][128] fp16, U'
// [64][128] fp32, Aqk^T [64][64] fp16 ([s][r]), ef [64] fp32 (exp of the in-chunk cumulative
// log alpha); and q [B, L, 16, 128] fp16.  out [B * L, ldo] fp16 (head h at columns 128 h ..).
// One launch walks chunks c0 .. c0 + ncl - 1 of every request (ncl < 0: to the end), entering
// from s0 (or zero) and leaving the state in s_out (may be s0).
clef_status gdn_state_launch(const __half* q, const __half* Kd, const __half* W, const float* U1,
                             const __half* Aqk, const float* ef, const float* s0, float* s_out,
                             __half* out, int64_t ldo, int64_t B, int64_t L, cudaStream_t stream,
                             int64_t c0 = 0, int64_t ncl = -1);

}  // namespace clef
