// Memory-bound glue of the decoder: embedding gather, RMSNorm, and the small fp16 gate
// projections a, b of the Gated DeltaNet layers with the gates computed in their epilogue.
//
// "clef-flash-LiteRT" README, "Host contract" step 4: the input rows are the embedding table's
// rows at the request's ids; step 6: the output is the hidden state after the final RMSNorm.
// "Clef-Flash-ANE-LUT6" model card, "Weight precision": normalisation weights and the small gate
// projections are FP16.
#include "common.cuh"
#include "glue.cuh"
#include "mma.cuh"

namespace clef {
namespace glue {

constexpr int H = 4096;

// One picture row per CTA: fp16 row r = b * n + k of `rows` widens into row b * L + start + k of x.
__global__ void __launch_bounds__(256) image_rows_kernel(const __half* __restrict__ rows,
                                                         float* __restrict__ x, int64_t L,
                                                         int64_t start, int64_t n) {
  pdl_trigger();
  pdl_wait();
  const int64_t r = blockIdx.x, b = r / n, k = r % n;
  const int c0 = threadIdx.x * 16;
  const uint4* src = reinterpret_cast<const uint4*>(rows + r * H + c0);
  float4* dst = reinterpret_cast<float4*>(x + (b * L + start + k) * H + c0);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint4 u = src[i];
    const __half2* h2 = reinterpret_cast<const __half2*>(&u);
    const float2 a = __half22float2(h2[0]), c = __half22float2(h2[1]);
    const float2 d = __half22float2(h2[2]), e = __half22float2(h2[3]);
    dst[2 * i] = make_float4(a.x, a.y, c.x, c.y);
    dst[2 * i + 1] = make_float4(d.x, d.y, e.x, e.y);
  }
}

__global__ void __launch_bounds__(256) embed_kernel(const int32_t* __restrict__ ids,
                                                    const __half* __restrict__ table,
                                                    int64_t vocab, float* __restrict__ x,
                                                    unsigned* status) {
  pdl_trigger();
  pdl_wait();
  const int64_t tok = blockIdx.x;
  const int32_t id = ids[tok];
  const bool ok = id >= 0 && (int64_t)id < vocab;
  if (!ok && threadIdx.x == 0) report(status, DEV_BAD_TOKEN);
  const int c0 = threadIdx.x * 16;
  float4* dst = reinterpret_cast<float4*>(x + tok * H + c0);
  if (!ok) {
#pragma unroll
    for (int i = 0; i < 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const uint4* src = reinterpret_cast<const uint4*>(table + (int64_t)id * H + c0);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint4 u = src[i];
    const __half2* h2 = reinterpret_cast<const __half2*>(&u);
    const float2 a = __half22float2(h2[0]), b = __half22float2(h2[1]);
    const float2 c = __half22float2(h2[2]), d = __half22float2(h2[3]);
    dst[2 * i] = make_float4(a.x, a.y, b.x, b.y);
    dst[2 * i + 1] = make_float4(c.x, c.y, d.x, d.y);
  }
}

// With `status` set (the final norm) a row whose residual or normalised output is not finite
// (an fp16 overflow somewhere upstream, or inf / NaN in the inputs) is reported: the status word
// gets DEV_NONFINITE_HIDDEN and the lowest such row is kept in `bad_row`.
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float* __restrict__ x,
                                                      const __half* __restrict__ w,
                                                      __half* __restrict__ y, unsigned* status,
                                                      unsigned long long* bad_row) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[8];
  const int64_t tok = blockIdx.x;
  const int c0 = threadIdx.x * 16;
  const float4* src = reinterpret_cast<const float4*>(x + tok * H + c0);
  float v[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = src[i];
    v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) ss += v[i] * v[i];
#pragma unroll
  for (int off = 16; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) tot += red[i];
  const float r = rsqrtf(tot * (1.f / H) + 1e-6f);
  const uint4* wp = reinterpret_cast<const uint4*>(w + c0);
  uint4 out[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    uint4 wu = wp[i];
    const __half2* wh = reinterpret_cast<const __half2*>(&wu);
    uint32_t* o = reinterpret_cast<uint32_t*>(&out[i]);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 wf = __half22float2(wh[j]);
      o[j] = h2u(v[8 * i + 2 * j] * r * wf.x, v[8 * i + 2 * j + 1] * r * wf.y);
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(y + tok * H + c0);
  dst[0] = out[0];
  dst[1] = out[1];
  if (status) {
    // exponent all ones in an fp16 output (inf or NaN), or a sum of squares that is not finite
    // (which would make a huge but finite row come out as zeros)
    bool bad = !isfinite(tot);
    const uint32_t* o32 = reinterpret_cast<const uint32_t*>(out);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      bad |= ((o32[i] & 0x7C00u) == 0x7C00u) || ((o32[i] & 0x7C000000u) == 0x7C000000u);
    if (__syncthreads_or(bad) && threadIdx.x == 0) report_bad_row(status, bad_row, tok);
  }
}

// Rows of fp16 values with an inf or a NaN: flags[row] = 1 (0 otherwise) when flags is set, and
// the lowest such row is reported as for the final norm.  One warp per row, 8 values per load.
__global__ void check_finite_kernel(const __half* __restrict__ x, int64_t rows, int64_t cols,
                                    uint8_t* __restrict__ flags, unsigned* status,
                                    unsigned long long* bad_row) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t row = blockIdx.x * (int64_t)(blockDim.x >> 5) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const uint4* src = reinterpret_cast<const uint4*>(x + row * cols);
    bool bad = false;
    for (int64_t i = lane; i < cols / 8; i += 32) {
      const uint4 u = src[i];
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int j = 0; j < 4; ++j)
        bad |= ((w[j] & 0x7C00u) == 0x7C00u) || ((w[j] & 0x7C000000u) == 0x7C000000u);
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      if (flags) flags[row] = bad ? 1 : 0;
      if (bad) report_bad_row(status, bad_row, row);
    }
  }
}

// ab = xn . W_ab^T on the tensor cores: a CTA (128 threads) takes 128 tokens x the 64 outputs
// over its share of the 64 k blocks.  Both operands stream by TMA (128-byte swizzle, K-major)
// through a ring of AB_ST stages (X box 128 tokens x 64 k, W box 64 outputs x 64 k): one thread of
// warp 0 loads, one thread of warp 1 issues four MMAs per block (kind::f16, M = 128 tokens, N = 64
// outputs, K = 16, both operands from shared memory) into a 64-column fp32 accumulator and frees
// the stage with one commit.  Then warp w reads tensor-memory lanes 32w..32w+31 (one token per
// thread, its 64 sums) and writes that token's gates, or with a K split its partial sums.
constexpr int AB_T = 128, AB_K = 64, AB_ST = 6;
constexpr int AB_X_BYTES = AB_T * AB_K * 2;           // 16 KB
constexpr int AB_W_BYTES = 64 * AB_K * 2;             // 8 KB
constexpr int AB_STAGE = AB_X_BYTES + AB_W_BYTES;
constexpr int AB_OFF_BAR = AB_ST * AB_STAGE;
constexpr int AB_NUM_BARS = 2 * AB_ST + 1;
constexpr int AB_SMEM = AB_OFF_BAR + 8 * AB_NUM_BARS + 8 + 1024;   // + tensor-memory slot, alignment
static_assert(AB_STAGE % 1024 == 0, "stages keep the 1024-byte alignment of the swizzle atoms");

// Gates from the summed projections: g = -exp(A_log) softplus(a + dt_bias) (>= -30), beta = sigmoid(b).
__device__ __forceinline__ float gate_g(float v, int col, const __half* A_log, const __half* dt_bias) {
  const float a = v + __half2float(dt_bias[col]);
  const float sp = a > 20.f ? a : log1pf(__expf(a));
  return fmaxf(-__expf(__half2float(A_log[col])) * sp, -30.f);
}
__device__ __forceinline__ void write_gate(int64_t tok, int col, float v, const __half* A_log,
                                           const __half* dt_bias, float* g, float* beta) {
  if (col < 32)
    g[tok * 32 + col] = gate_g(v, col, A_log, dt_bias);
  else
    beta[tok * 32 + col - 32] = sigmoid_f(v);
}

// blockIdx.y = slice of K (gridDim.y slices, at most 64).  With one slice the epilogue computes
// the gates; otherwise it writes its partial sums to part [slice][M][64] for ab_gates_kernel.
__global__ void __launch_bounds__(128, 1) ab_proj_kernel(const __grid_constant__ CUtensorMap tmap_x,
                                                         const __grid_constant__ CUtensorMap tmap_w,
                                                         const __half* __restrict__ A_log,
                                                         const __half* __restrict__ dt_bias,
                                                         float* __restrict__ g,
                                                         float* __restrict__ beta,
                                                         float* __restrict__ part, int64_t M,
                                                         unsigned* status) {
  pdl_trigger();
  extern __shared__ uint8_t ab_smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ab_smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t t0 = (int64_t)blockIdx.x * AB_T;
  const int nkb_all = H / AB_K;
  const int kb0 = blockIdx.y * nkb_all / gridDim.y;
  const int nkb = (blockIdx.y + 1) * nkb_all / gridDim.y - kb0;
  const uint32_t bar_full = sb + AB_OFF_BAR;           // [AB_ST] stage landed (TMA bytes)
  const uint32_t bar_empty = bar_full + 8 * AB_ST;     // [AB_ST] stage read by its MMAs
  const uint32_t bar_done = bar_empty + 8 * AB_ST;     // every MMA completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + AB_OFF_BAR + 8 * AB_NUM_BARS);
  if (threadIdx.x == 0) {
    for (int s = 0; s < AB_ST; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_done, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();   // the barriers and tensor memory are set up; now the inputs

  if (warp == 0 && lane == 0) {
    int i = 0;
    for (; i < nkb; ++i) {
      const int s = i % AB_ST;
      // stage s was last read by the MMAs of block i - AB_ST
      if (i >= AB_ST && !mbar_wait(bar_empty + 8 * s, (uint32_t)(i / AB_ST - 1) & 1, status,
                                   DEV_TIMEOUT_TMA))
        break;
      const uint32_t fb = bar_full + 8 * s;
      mbar_arrive_expect_tx(fb, AB_STAGE);
      tma_load_2d(sb + s * AB_STAGE, &tmap_x, fb, (kb0 + i) * AB_K, (int)t0);   // rows >= M read 0
      tma_load_2d(sb + s * AB_STAGE + AB_X_BYTES, &tmap_w, fb, (kb0 + i) * AB_K, 0);
    }
    // copies still in flight land before the CTA may exit
    for (int h = i > AB_ST ? i - AB_ST : 0; h < i; ++h)
      mbar_wait(bar_full + 8 * (h % AB_ST), (uint32_t)(h / AB_ST) & 1, status, DEV_TIMEOUT_TMA);
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_f16_f32(AB_T, 64);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % AB_ST;
      // one descriptor per operand and stage; the four K slices are constant offsets of its
      // address field (32 bytes each)
      const uint64_t ad = sdesc_k_sw128(sb + s * AB_STAGE);
      const uint64_t bd = sdesc_k_sw128(sb + s * AB_STAGE + AB_X_BYTES);
      if (!mbar_wait(bar_full + 8 * s, (uint32_t)(i / AB_ST) & 1, status, DEV_TIMEOUT_MMA)) break;
      tc_fence_after();
      tc_mma_f16_ss(tmem, ad, bd, idesc, i != 0);
      tc_mma_f16_ss(tmem, ad + 2, bd + 2, idesc, 1);
      tc_mma_f16_ss(tmem, ad + 4, bd + 4, idesc, 1);
      tc_mma_f16_ss(tmem, ad + 6, bd + 6, idesc, 1);
      tc_commit(bar_empty + 8 * s);
    }
    // arrives once every MMA issued above has completed (also after a timed-out wait)
    tc_commit(bar_done);
  }
  __syncwarp();
  if (mbar_wait(bar_done, 0, status, DEV_TIMEOUT_EPILOGUE)) {
    tc_fence_after();
    uint32_t ra[32], rb[32];     // columns 0..31 (a) and 32..63 (b) of this thread's token
    const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16);
    tmem_ld_32x32b_x32(ta, ra);
    tmem_ld_32x32b_x32(ta + 32, rb);
    tc_wait_ld();
    const int64_t tok = t0 + warp * 32 + lane;
    if (tok < M) {
      if (gridDim.y == 1) {
        float4* gp = reinterpret_cast<float4*>(g + tok * 32);
        float4* bp = reinterpret_cast<float4*>(beta + tok * 32);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          gp[c / 4] = make_float4(gate_g(__uint_as_float(ra[c]), c, A_log, dt_bias),
                                  gate_g(__uint_as_float(ra[c + 1]), c + 1, A_log, dt_bias),
                                  gate_g(__uint_as_float(ra[c + 2]), c + 2, A_log, dt_bias),
                                  gate_g(__uint_as_float(ra[c + 3]), c + 3, A_log, dt_bias));
          bp[c / 4] = make_float4(sigmoid_f(__uint_as_float(rb[c])), sigmoid_f(__uint_as_float(rb[c + 1])),
                                  sigmoid_f(__uint_as_float(rb[c + 2])), sigmoid_f(__uint_as_float(rb[c + 3])));
        }
      } else {
        float4* pp = reinterpret_cast<float4*>(part + ((int64_t)blockIdx.y * M + tok) * 64);
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          pp[c / 4] = make_float4(__uint_as_float(ra[c]), __uint_as_float(ra[c + 1]),
                                  __uint_as_float(ra[c + 2]), __uint_as_float(ra[c + 3]));
          pp[8 + c / 4] = make_float4(__uint_as_float(rb[c]), __uint_as_float(rb[c + 1]),
                                      __uint_as_float(rb[c + 2]), __uint_as_float(rb[c + 3]));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

// Sums the K-slice partials in slice order (deterministic) and writes the gates.
__global__ void ab_gates_kernel(const float* __restrict__ part, int slices,
                                const __half* __restrict__ A_log, const __half* __restrict__ dt_bias,
                                float* __restrict__ g, float* __restrict__ beta, int64_t M) {
  pdl_trigger();
  pdl_wait();
  const int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  if (i >= M * 64) return;
  float v = 0.f;
  for (int sl = 0; sl < slices; ++sl) v += part[sl * M * 64 + i];
  write_gate(i / 64, (int)(i % 64), v, A_log, dt_bias, g, beta);
}

}  // namespace glue

clef_status embed_launch(const int32_t* ids, const __half* table, int64_t vocab, float* x,
                         int64_t M, cudaStream_t stream) {
  if (M == 0) return CLEF_OK;
  TraceScope ts(stream, "embed", 0.0, M * (4096.0 * 2 + 4096.0 * 4));
  CLEF_CUDA_CHECK(launch_pdl(glue::embed_kernel, dim3((unsigned)M), dim3(256), 0, stream,
       ids, table, vocab, x, status_word_ptr()));
  return CLEF_OK;
}

clef_status image_rows_launch(const __half* rows, float* x, int64_t B, int64_t L, int64_t start,
                              int64_t n, cudaStream_t stream) {
  if (B == 0 || n == 0) return CLEF_OK;
  TraceScope ts(stream, "image_rows", 0.0, B * n * (4096.0 * 2 + 4096.0 * 4));
  CLEF_CUDA_CHECK(launch_pdl(glue::image_rows_kernel, dim3((unsigned)(B * n)), dim3(256), 0, stream,
       rows, x, L, start, n));
  return CLEF_OK;
}

clef_status rmsnorm_launch(const float* x, const __half* w, __half* y, int64_t M,
                           cudaStream_t stream, bool check_finite) {
  if (M == 0) return CLEF_OK;
  TraceScope ts(stream, "rmsnorm", 0.0, M * (4096.0 * 4 + 4096.0 * 2));
  CLEF_CUDA_CHECK(launch_pdl(glue::rmsnorm_kernel, dim3((unsigned)M), dim3(256), 0, stream,
       x, w, y, check_finite ? status_word_ptr() : nullptr,
       check_finite ? bad_row_word_ptr() : nullptr));
  return CLEF_OK;
}

clef_status check_finite_launch(const __half* x, int64_t rows, int64_t cols, uint8_t* flags,
                                cudaStream_t stream) {
  if (rows == 0) return CLEF_OK;
  TraceScope ts(stream, "check_finite", 0.0, rows * cols * 2.0 + (flags ? rows : 0));
  const int64_t blocks = std::min<int64_t>((rows + 7) / 8, (int64_t)num_sms() * 16);
  glue::check_finite_kernel<<<(unsigned)blocks, 256, 0, stream>>>(x, rows, cols, flags,
                                                                  status_word_ptr(),
                                                                  bad_row_word_ptr());
  CLEF_LAUNCH_CHECK();
  return CLEF_OK;
}

size_t ab_proj_scratch_bytes(int64_t M) { return (size_t)kAbMaxSlices * M * 64 * 4; }

clef_status ab_proj_launch(const __half* xn, const __half* w_ab, const __half* A_log,
                           const __half* dt_bias, float* g, float* beta, float* part, int64_t M,
                           cudaStream_t stream) {
  if (M == 0) return CLEF_OK;
  const int64_t ctas = (M + glue::AB_T - 1) / glue::AB_T;
  // split K when there are too few token blocks to fill the GPU (partials summed in order)
  int slices = 1;
  while (slices < kAbMaxSlices && ctas * slices * 2 <= num_sms()) slices *= 2;
  TraceScope ts(stream, "ab_proj", 2.0 * M * 64 * 4096, M * (4096.0 * 2 + 64 * 4) + 64 * 4096 * 2.0);
  CUtensorMap tx, tw;
  if (tma_encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xn, (uint64_t)glue::H, (uint64_t)M,
                    (uint64_t)glue::H * 2, glue::AB_K, glue::AB_T, CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess ||
      tma_encode_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, w_ab, (uint64_t)glue::H, 64,
                    (uint64_t)glue::H * 2, glue::AB_K, 64, CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess)
    return CLEF_E_CUDA;
  static std::atomic<uint64_t> attr{0};
  CLEF_CUDA_CHECK(smem_opt_in((const void*)glue::ab_proj_kernel, glue::AB_SMEM, &attr));
  CLEF_CUDA_CHECK(launch_pdl(glue::ab_proj_kernel, dim3((unsigned)ctas, (unsigned)slices), dim3(128), glue::AB_SMEM, stream,
       tx, tw, A_log, dt_bias, g, beta, part, M, status_word_ptr()));
  if (slices > 1) {
    CLEF_CUDA_CHECK(launch_pdl(glue::ab_gates_kernel, dim3((unsigned)((M * 64 + 255) / 256)), dim3(256), 0, stream,
         part, slices, A_log,
         dt_bias, g, beta, M));
  }
  return CLEF_OK;
}

}  // namespace clef
