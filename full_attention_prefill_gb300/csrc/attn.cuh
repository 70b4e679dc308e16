// Internal launchers of the attention kernels (not part of the C ABI).
#pragma once
#include "common.cuh"

namespace clef {

// Rotary on dims 0..63 of the 16 q heads and 4 k heads of M tokens (requests of L positions).
// In place when qout == qin and kout == kin; otherwise a rotated copy of all 256 dims.
clef_status rope_launch(const __half* qin, int64_t ldqi, __half* qout, int64_t ldqo,
                        const __half* kin, int64_t ldki, __half* kout, int64_t ldko, int64_t M,
                        int64_t L, cudaStream_t stream);

// Causal GQA flash attention on rotated q, k; gate may be NULL.  Row strides in elements.
clef_status flash_launch(const __half* q, int64_t ldq, const __half* k, int64_t ldk,
                         const __half* v, int64_t ldv, const __half* gate, int64_t ldg, __half* out,
                         int64_t ldo, int64_t B, int64_t L, cudaStream_t stream);

}  // namespace clef
