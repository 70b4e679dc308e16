// Internal launchers of the Gated DeltaNet kernels (not part of the C ABI).
#pragma once
#include "common.cuh"

namespace clef {

// conv(4) + SiLU + q/k L2 norm, for M tokens of requests of L positions.
clef_status gdn_prep_launch(const __half* proj, int64_t ldp, const __half* conv_w, __half* q,
                            __half* k, __half* v, int64_t M, int64_t L, cudaStream_t stream);

// with_norm: room for o before the output gate (decoder layer path, z != NULL)
size_t gdn_scan_workspace_bytes(int64_t B, int64_t L, bool with_norm);

// The chunked scan.  Exactly one of g (log alpha) / alpha is non-NULL.  With z != NULL the
// output is the z-gated RMSNorm (weight o_norm) of o; otherwise o itself.  out [M, ldo] fp16.
clef_status gdn_scan_launch(const __half* q, const __half* k, const __half* v, const float* g,
                            const float* alpha, const float* beta, const float* s0, float* s_out,
                            const __half* z, int64_t ldz, const __half* o_norm, __half* out,
                            int64_t ldo, int64_t B, int64_t L, void* ws, cudaStream_t stream);

}  // namespace clef
