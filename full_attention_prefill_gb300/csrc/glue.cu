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

// ab = xn . W_ab^T: 64 tokens x 64 outputs per CTA, k streamed in blocks of 64 through a ring of
// AB_ST cp.async stages (three blocks in flight while one is multiplied), warp w owns tokens
// 16w..16w+15.
constexpr int AB_T = 64, AB_K = 64, AB_LD = AB_K + 8, AB_ST = 4;
struct AbSmem {
  __half X[AB_ST][AB_T][AB_LD];
  __half W[AB_ST][64][AB_LD];
};

// Gates from the summed projections: g = -exp(A_log) softplus(a + dt_bias) (>= -30), beta = sigmoid(b).
__device__ __forceinline__ void write_gate(int64_t tok, int col, float v, const __half* A_log,
                                           const __half* dt_bias, float* g, float* beta) {
  if (col < 32) {
    const float a = v + __half2float(dt_bias[col]);
    const float sp = a > 20.f ? a : log1pf(__expf(a));
    g[tok * 32 + col] = fmaxf(-__expf(__half2float(A_log[col])) * sp, -30.f);
  } else {
    beta[tok * 32 + col - 32] = sigmoid_f(v);
  }
}

// blockIdx.y = slice of K (gridDim.y slices).  With one slice the epilogue computes the gates;
// otherwise it writes its partial sums to part [slice][M][64] for ab_gates_kernel.
__global__ void __launch_bounds__(128) ab_proj_kernel(const __half* __restrict__ xn,
                                                      const __half* __restrict__ wab,
                                                      const __half* __restrict__ A_log,
                                                      const __half* __restrict__ dt_bias,
                                                      float* __restrict__ g,
                                                      float* __restrict__ beta,
                                                      float* __restrict__ part, int64_t M) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) uint8_t ab_smem[];
  AbSmem& s = *reinterpret_cast<AbSmem*>(ab_smem);
  const int64_t t0 = (int64_t)blockIdx.x * AB_T;
  const int nkb_all = H / AB_K;
  const int kb0 = blockIdx.y * nkb_all / gridDim.y;
  const int kb1 = (blockIdx.y + 1) * nkb_all / gridDim.y;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  auto load = [&](int buf, int kb) {
    for (int i = tid; i < AB_T * (AB_K / 8); i += 128) {
      const int r = i / (AB_K / 8), c8 = (i % (AB_K / 8)) * 8;
      const bool ok = t0 + r < M;
      cp_async16(smem_u32(&s.X[buf][r][c8]), xn + (ok ? t0 + r : 0) * H + kb * AB_K + c8, ok);
      cp_async16(smem_u32(&s.W[buf][r][c8]), wab + (int64_t)r * H + kb * AB_K + c8, true);
    }
    cp_async_commit();
  };
  float acc[8][4];
#pragma unroll
  for (int n = 0; n < 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
  for (int i = 0; i < AB_ST - 1; ++i) {
    if (kb0 + i < kb1) load(i, kb0 + i); else cp_async_commit();
  }
  for (int kb = kb0; kb < kb1; ++kb) {
    const int buf = (kb - kb0) % AB_ST;
    cp_async_wait<AB_ST - 2>();   // block kb has landed
    __syncthreads();              // ... for every thread, and the slot of kb - 1 is free again
    const int nxt = kb + AB_ST - 1;
    if (nxt < kb1) load((nxt - kb0) % AB_ST, nxt); else cp_async_commit();
    const uint32_t sX = smem_u32(&s.X[buf][0][0]), sW = smem_u32(&s.W[buf][0][0]);
#pragma unroll
    for (int ks = 0; ks < AB_K / 16; ++ks) {
      uint32_t a[4];
      ldsm_x4(a, a_addr(sX, AB_LD, warp * 16, ks * 16, lane));
#pragma unroll
      for (int n = 0; n < 8; n += 2) {
        uint32_t bq[4];
        ldsm_x4(bq, bn_addr(sW, AB_LD, n * 8, ks * 16, lane));
        mma16816(acc[n], a, bq[0], bq[1]);
        mma16816(acc[n + 1], a, bq[2], bq[3]);
      }
    }
  }
  cp_async_wait<0>();
  const int gq = lane >> 2, tq = lane & 3;
  // gates of the 32 value heads: columns 0..31 are a, 32..63 are b
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int64_t tok = t0 + warp * 16 + gq + hf * 8;
    if (tok >= M) continue;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int col = n * 8 + 2 * tq;
      if (gridDim.y == 1) {
        write_gate(tok, col, acc[n][2 * hf], A_log, dt_bias, g, beta);
        write_gate(tok, col + 1, acc[n][2 * hf + 1], A_log, dt_bias, g, beta);
      } else {
        *reinterpret_cast<float2*>(part + ((int64_t)blockIdx.y * M + tok) * 64 + col) =
            make_float2(acc[n][2 * hf], acc[n][2 * hf + 1]);
      }
    }
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
  static std::atomic<uint64_t> attr{0};
  CLEF_CUDA_CHECK(smem_opt_in((const void*)glue::ab_proj_kernel, sizeof(glue::AbSmem), &attr));
  CLEF_CUDA_CHECK(launch_pdl(glue::ab_proj_kernel, dim3(dim3((unsigned)ctas, (unsigned)slices)), dim3(128), sizeof(glue::AbSmem), stream,
       xn, w_ab, A_log, dt_bias, g, beta, part, M));
  if (slices > 1) {
    CLEF_CUDA_CHECK(launch_pdl(glue::ab_gates_kernel, dim3((unsigned)((M * 64 + 255) / 256)), dim3(256), 0, stream,
         part, slices, A_log,
         dt_bias, g, beta, M));
  }
  return CLEF_OK;
}

}  // namespace clef
