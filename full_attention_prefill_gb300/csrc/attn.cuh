// Internal launchers of the attention kernels (not part of the C ABI).
#pragma once
#include "common.cuh"

namespace clef {

// One picture block of a request for M-RoPE: h x w tokens from token index `start` (h * w == 0:
// text only, every plane at the token index).
struct MRope {
  int64_t start = 0, h = 0, w = 0;
};

// Rotary on dims 0..63 of the 16 q heads and 4 k heads of M tokens (request chunks of L
// tokens starting at token index pos0).  Pair j turns by the position of plane j mod 3 of the
// token's M-RoPE positions (all three equal the token index for text).  q rows stay in place
// (qout == qin) or go to the same rows of a copy; k rows go to row (request * kctx + pos0 + t)
// of kout (kctx = L, pos0 = 0: the same rows).  A copy carries all 256 dims.
clef_status rope_launch(const __half* qin, int64_t ldqi, __half* qout, int64_t ldqo,
                        const __half* kin, int64_t ldki, __half* kout, int64_t ldko, int64_t M,
                        int64_t L, int64_t pos0, int64_t kctx, cudaStream_t stream,
                        const MRope& mr = MRope());

// Causal GQA flash attention on rotated q, k; gate may be NULL.  Row strides in elements.
// Queries: positions pos0 .. pos0 + L - 1 of B requests (rows request * L + t of q, gate, out);
// keys and values: positions 0 .. pos0 + L - 1 (rows request * kv_req + p of k, v).  A whole
// prefill is pos0 = 0, kv_req = L.
clef_status flash_launch(const __half* q, int64_t ldq, const __half* k, int64_t ldk,
                         const __half* v, int64_t ldv, const __half* gate, int64_t ldg, __half* out,
                         int64_t ldo, int64_t B, int64_t L, int64_t pos0, int64_t kv_req,
                         cudaStream_t stream);

// Row (request * L + t) of src -> row (request * dctx + pos0 + t) of dst, `cols` fp16 each.
clef_status kv_store_launch(const __half* src, int64_t lds, __half* dst, int64_t ldd, int64_t M,
                            int64_t L, int64_t pos0, int64_t dctx, int cols, cudaStream_t stream);

}  // namespace clef
