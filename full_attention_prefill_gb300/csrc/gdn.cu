// Gated DeltaNet: input preparation and the chunked scan.
//
// The recurrence ("Clef-Flash-ANE-LUT6" model card, "Model architecture"; "clef-flash - Core AI"
// README, "Core AI shape": a [32, 128, 128] state per GDN layer), for value head h reading key
// head h/2:
//     S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,   o_t = S_t q_t / sqrt(128)
// is evaluated in chunks of C = 64 positions ("clef-flash-LiteRT" README, "Provenance": there
// the recurrence is exported in 64-position chunks).  With g the cumulative
// log(alpha) inside a chunk and S0 the state entering it:
//     A = strict_tril(diag(beta) (exp(g_r - g_s)) o K K^T),   T = (I + A)^-1
//     W = T diag(beta exp(g)) K,   U' = T diag(beta) V,   U = U' - W S0^T
//     O = (diag(exp(g)) Q S0^T + (tril(Q K^T) o exp(g_r - g_s)) U) / sqrt(128)
//     S_C = exp(g_C) S0 + U^T diag(exp(g_C - g)) K
// Kernels:
//   gdn_chunk_wy    (parallel over chunks x heads): cumulative g, T by forward substitution,
//                   W, U', the decayed keys exp(g_C - g) k and the intra-chunk matrix
//                   Aqk = tril(Q K^T) o exp(g_r - g_s) / sqrt(128) (stored transposed)
//   gdn_state_tc    (gdn_state.cu; sequential over chunks, one CTA per value head): the state
//                   stays in tensor memory; per chunk U = U' - W S0^T, S <- exp(g_C) S + U^T Kd,
//                   O = exp(g) Q S0^T / sqrt(128) + Aqk U, all on tcgen05
//   gdn_gated_norm  (decoder layer only): y = RMSNorm_128(O) * w_o * SiLU(z)
// The chunk phase's products run on mma.sync (m16n8k16, fp16 inputs, fp32 accumulation); the
// state and the scalars stay fp32.  A long scan of one request runs in pieces of chunks:
// the chunk phase of the next piece on a low-priority stream beside the state pass of this one
// on a high-priority stream (events order them; the state crosses pieces in fp32).
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "gdn.cuh"
#include "mma.cuh"

namespace clef {
namespace gdn {

constexpr int LDH = D + 8;     // padded fp16 row (272 bytes) for conflict-free ldmatrix
constexpr float kLogAlphaMin = -30.0f;

// ------------------------------------------------------------------------------------------
// Prep for the decoder layer: causal depthwise conv (4 taps) + SiLU over the 8192 QKV channels and
// the per-head L2 norm of q and k.  Persistent: three CTAs (256 threads) per SM walk tiles of
// PREP_T tokens x 512 channels (tile t: channel block t mod 16, token block t / 16).  A tile's
// PREP_T + 3 rows (the conv's history included) are copied into shared memory with cp.async,
// double-buffered so that the next tile's copies are in flight while this one is computed; then
// thread (token half, 4 channels) walks its PREP_T / 2 tokens with the 3-row history in
// registers, fully unrolled when none of them lies within 3 positions of a request start.  A warp
// covers 128 channels, exactly one q or k head, so the norm is a warp reduction.  The gates
// come from the a/b projection's epilogue.  Token indices are 32-bit (the entry points refuse
// more than 2^22 tokens).
// proj [M, ldp] fp16: q 0..2047 | k 2048..4095 | v 4096..8191 (| z 8192..).
// ------------------------------------------------------------------------------------------
constexpr int PREP_T = 32;
constexpr int PREP_CH = 512;
constexpr int PREP_ROWS = PREP_T + 3;
constexpr int PREP_BUF = PREP_ROWS * PREP_CH * 2;
constexpr int PREP_SMEM = 2 * PREP_BUF;
constexpr int PREP_CTAS_PER_SM = 3;
// x * sigmoid(x) and 1 / sqrt(x) by the hardware's approximate exp2, reciprocal and reciprocal
// square root with subnormals flushed (PTX ex2.approx.ftz.f32, rcp.approx.ftz.f32,
// rsqrt.approx.ftz.f32): one instruction each, where the non-flushing forms add range handling.
// Large negative x: 2^(-x log2 e) overflows to +inf and the reciprocal to 0, so the result is -0.
__device__ __forceinline__ float silu_ftz(float x) {
  float e, r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(x * -1.4426950408889634f));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
  return x * r;
}
__device__ __forceinline__ float rsqrt_ftz(float x) {
  float r;
  asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}
// The 4 channels of a tile row as floats.
__device__ __forceinline__ void prep_row(const __half* p, float (&x)[4]) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
  x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
}
// One output token from its four taps (oldest first): conv, SiLU, and for q and k the head's L2
// norm (the warp's 32 lanes hold its 128 channels).
template <bool QK>
__device__ __forceinline__ void prep_token(const float (&w)[4][4], const float (&x0)[4],
                                           const float (&x1)[4], const float (&x2)[4],
                                           const float (&x3)[4], __half* out) {
  float y[4];
#pragma unroll
  for (int c = 0; c < 4; ++c)
    y[c] = silu_ftz(w[c][0] * x0[c] + w[c][1] * x1[c] + w[c][2] * x2[c] + w[c][3] * x3[c]);
  if (QK) {
    float ss = y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float r = rsqrt_ftz(ss + 1e-6f);
#pragma unroll
    for (int c = 0; c < 4; ++c) y[c] *= r;
  }
  *reinterpret_cast<uint2*>(out) = make_uint2(h2u(y[0], y[1]), h2u(y[2], y[3]));
}
// PREP_T / 2 consecutive tokens of one request whose taps all lie in the tile (rows j0 .. j0 +
// PREP_T / 2 + 2 at `row0`); q and k rows are 2048 apart, v rows 4096, so the stores take
// constant offsets from `out`.
template <bool QK>
__device__ __forceinline__ void prep_run(const __half* row0, const float (&w)[4][4], __half* out) {
  constexpr int LDD = QK ? 2048 : 4096;
  float h0[4], h1[4], h2[4];
  prep_row(row0, h0);
  prep_row(row0 + PREP_CH, h1);
  prep_row(row0 + 2 * PREP_CH, h2);
#pragma unroll
  for (int j = 0; j < PREP_T / 2; ++j) {
    float x3[4];
    prep_row(row0 + (j + 3) * PREP_CH, x3);
    prep_token<QK>(w, h0, h1, h2, x3, out + j * LDD);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      h0[c] = h1[c];
      h1[c] = h2[c];
      h2[c] = x3[c];
    }
  }
}

// The conv taps of channels ch0 .. ch0 + 3 as floats, [channel][tap].
__device__ __forceinline__ void prep_weights(const __half* conv_w, int ch0, float (&w)[4][4]) {
  const uint4* wp = reinterpret_cast<const uint4*>(conv_w + (int64_t)ch0 * 4);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint4 u = __ldg(wp + i);
    const __half* hh = reinterpret_cast<const __half*>(&u);
#pragma unroll
    for (int j = 0; j < 8; ++j) w[(i * 8 + j) / 4][(i * 8 + j) % 4] = __half2float(hh[j]);
  }
}

// Tokens of a thread's run that lie within 3 positions of a request start (their earlier taps
// read the carried conv input, or zero) or past M: one token at a time.
__device__ __noinline__ void prep_edge(const __half* row0, const __half* conv_w, bool is_qk,
                                       __half* dst, int64_t ldd, const __half* conv_in, int ch0,
                                       int tok_a, int pos, int64_t M, int L) {
  float w[4][4];
  prep_weights(conv_w, ch0, w);
  int req = tok_a / L;
  auto emit = [&](int tok, const float (&x0)[4], const float (&x1)[4], const float (&x2)[4],
                  const float (&x3)[4]) {
    if (is_qk)
      prep_token<true>(w, x0, x1, x2, x3, dst + (int64_t)tok * ldd);
    else
      prep_token<false>(w, x0, x1, x2, x3, dst + (int64_t)tok * ldd);
  };
  float h0[4], h1[4], h2[4];            // tokens t-3, t-2, t-1
  prep_row(row0, h0);
  prep_row(row0 + PREP_CH, h1);
  prep_row(row0 + 2 * PREP_CH, h2);
#pragma unroll 1
  for (int j = 0; j < PREP_T / 2 && tok_a + j < M; ++j) {
    float x3[4];
    prep_row(row0 + (j + 3) * PREP_CH, x3);
    if (pos >= 3) {
      emit(tok_a + j, h0, h1, h2, x3);
    } else {
      // taps reaching before the request's start read the carried conv input (its last
      // three rows, oldest first), or zero without one
      auto hist = [&](int r, float (&x)[4]) {   // carried row r = 0..2
        if (conv_in) {
          const uint2 u = __ldg(reinterpret_cast<const uint2*>(conv_in + ((int64_t)req * 3 + r) * 8192 + ch0));
          const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
          const float2 bb = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
          x[0] = a.x; x[1] = a.y; x[2] = bb.x; x[3] = bb.y;
        } else {
          x[0] = x[1] = x[2] = x[3] = 0.f;
        }
      };
      // tap j reads position pos - 3 + j, i.e. carried row pos + j when that is negative
      float x0[4], x1[4], x2[4];
      if (pos >= 3) { for (int c = 0; c < 4; ++c) x0[c] = h0[c]; } else hist(pos, x0);
      if (pos >= 2) { for (int c = 0; c < 4; ++c) x1[c] = h1[c]; } else hist(pos + 1, x1);
      if (pos >= 1) { for (int c = 0; c < 4; ++c) x2[c] = h2[c]; } else hist(pos + 2, x2);
      emit(tok_a + j, x0, x1, x2, x3);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      h0[c] = h1[c];
      h1[c] = h2[c];
      h2[c] = x3[c];
    }
    if (++pos == L) {
      pos = 0;
      ++req;
    }
  }
}

__global__ void __launch_bounds__(256, PREP_CTAS_PER_SM) gdn_prep_kernel(
    const __half* __restrict__ proj, int64_t ldp, const __half* __restrict__ conv_w,
    const __half* __restrict__ conv_in, __half* __restrict__ q, __half* __restrict__ k,
    __half* __restrict__ v, int64_t M, int L, int64_t n_tiles) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) uint8_t prep_smem[];
  const int tid = threadIdx.x;
  // copies of tile t into buffer b (row i = token tok0 - 3 + i; rows outside [0, M) zero-filled)
  // (thread tid copies 16 bytes at column (tid mod 64) * 8 of rows tid / 64, + 4, + 8, ...)
  auto load = [&](int64_t t, int b) {
    const int c8 = (tid % (PREP_CH / 8)) * 8;
    const int r0 = tid / (PREP_CH / 8);
    const int tok0 = (int)(t / (8192 / PREP_CH)) * PREP_T;
    const __half* src = proj + (int)(t % (8192 / PREP_CH)) * PREP_CH + c8;
    const uint32_t dst = smem_u32(prep_smem + b * PREP_BUF) + (uint32_t)(tid * 16);
    if (tok0 >= 3 && tok0 + PREP_T <= M) {
      const __half* p = src + (int64_t)(tok0 - 3 + r0) * ldp;
#pragma unroll
      for (int m = 0; m < PREP_ROWS / 4; ++m, p += 4 * ldp) cp_async16(dst + m * 4096, p, true);
      if (r0 + 4 * (PREP_ROWS / 4) < PREP_ROWS) cp_async16(dst + (PREP_ROWS / 4) * 4096, p, true);
    } else {
#pragma unroll 1
      for (int r = r0; r < PREP_ROWS; r += 4) {
        const int tk = tok0 - 3 + r;
        const bool ok = tk >= 0 && tk < M;
        cp_async16(dst + (r - r0) * 1024, src + (int64_t)(ok ? tk : 0) * ldp, ok);
      }
    }
  };
  const int cl = (tid & 127) * 4;           // this thread's 4 channels within the tile
  const int j0 = (tid >> 7) * (PREP_T / 2); // its first token within the tile
  int64_t t = blockIdx.x;
  if (t < n_tiles) load(t, 0);
  cp_async_commit();
  for (int n = 0; t < n_tiles; ++n, t += gridDim.x) {
    if (t + gridDim.x < n_tiles) load(t + gridDim.x, (n + 1) & 1);
    cp_async_commit();
    const int ch0 = (int)(t % (8192 / PREP_CH)) * PREP_CH + cl;
    const int tok_a = (int)(t / (8192 / PREP_CH)) * PREP_T + j0;   // this thread's first token
    float w[4][4];                          // [channel][tap]
    prep_weights(conv_w, ch0, w);
    const bool is_qk = ch0 < 4096;
    __half* dst = (ch0 < 2048 ? q + ch0 : (ch0 < 4096 ? k + (ch0 - 2048) : v + (ch0 - 4096)));
    const int64_t ldd = ch0 < 4096 ? 2048 : 4096;
    const __half* tile = reinterpret_cast<const __half*>(prep_smem + (n & 1) * PREP_BUF) + cl;
    cp_async_wait<1>();
    __syncthreads();
    int pos = tok_a % L;                    // position of the first token in its request
    if (pos >= 3 && pos + PREP_T / 2 <= L && tok_a + PREP_T / 2 <= M) {
      // the same for the whole warp (one token half): every tap lies in this request and the tile
      __half* out = dst + (int64_t)tok_a * ldd;
      if (is_qk)
        prep_run<true>(tile + j0 * PREP_CH, w, out);
      else
        prep_run<false>(tile + j0 * PREP_CH, w, out);
    } else {
      prep_edge(tile + j0 * PREP_CH, conv_w, is_qk, dst, ldd, conv_in, ch0, tok_a, pos, M, L);
    }
    __syncthreads();                        // buffer n & 1 is refilled by the next iteration
  }
}

// The conv input carried to the next chunk: for request b, the last three rows (oldest first)
// of the q | k | v projection over the carried rows and this chunk's L rows.  In place: each
// thread reads the old rows it needs before writing.
__global__ void conv_state_kernel(const __half* __restrict__ proj, int64_t ldp, __half* state,
                                  int64_t B, int L) {
  pdl_trigger();
  pdl_wait();
  const int64_t n = B * (8192 / 8);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t b = i / (8192 / 8);
    const int c8 = (int)(i % (8192 / 8)) * 8;
    uint4 r[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      const int p = L - 3 + j;               // position of the new row j within the chunk
      r[j] = p >= 0 ? *reinterpret_cast<const uint4*>(proj + (b * L + p) * ldp + c8)
                    : *reinterpret_cast<const uint4*>(state + (b * 3 + (3 + p)) * 8192 + c8);
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) *reinterpret_cast<uint4*>(state + (b * 3 + j) * 8192 + c8) = r[j];
  }
}

// g = log(alpha), clamped, for callers that pass alpha itself.
__global__ void log_alpha_kernel(const float* __restrict__ alpha, float* __restrict__ g, int64_t n) {
  pdl_trigger();
  pdl_wait();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float a = alpha[i];
    g[i] = a > 0.f ? fmaxf(logf(a), kLogAlphaMin) : kLogAlphaMin;
  }
}

// ------------------------------------------------------------------------------------------
// Phase 1: per (chunk, value head): cumulative g, A, T = (I + A)^-1, W = T diag(beta e^g) K,
// U' = T diag(beta) V, the decayed keys and Aqk.  128 threads; warp w owns rows 16w .. 16w+15
// of every 64-row product.  Outputs go to one contiguous block per (chunk, head): W [64][128]
// fp16, U' [64][128] fp32, Kd [64][128] fp16, Aqk^T [64][64] fp16, exp(g) [64] fp32.  Rows past
// the request's end come out zero (their beta, K and V are zero).
// T is formed blockwise: the four 16x16 diagonal blocks by forward substitution (one warp each),
// then the off-diagonal blocks by distance d = 1, 2, 3 from the diagonal:
//     T_ij = -T_ii (sum_{j <= k < i} A_ik T_kj),
// all in fp32.
// ------------------------------------------------------------------------------------------
struct WySmem {
  union {
    __half Q[C][LDH];                            // until Aqk is formed
    float A[C][C + 4];                           // then A (strictly lower triangular)
    struct {
      __half Tw[C][C + 8];                       // then T diag(beta e^g)
      __half Tu[C][C + 8];                       //  and T diag(beta), the products' A operands
    } t;
  } u;
  __half K[C][LDH];
  union {
    float Tf[C][C + 4];                          // T in fp32, until its scaled fp16 copies exist
    __half V[C][LDH];                            // then V (loaded behind the W product)
  } tv;
  float gc[C];
  float bt[C];
  float eb[C];                                   // beta_r exp(g_r)
  float ed[C];                                   // exp(g_C - g_r)
};

__global__ void __launch_bounds__(128) gdn_chunk_wy_kernel(
    const __half* __restrict__ qq, const __half* __restrict__ kk, const __half* __restrict__ vv,
    const float* __restrict__ g, const float* __restrict__ beta, float* __restrict__ ef,
    __half* __restrict__ Wout, float* __restrict__ Uout, __half* __restrict__ Kdout,
    __half* __restrict__ AqkT, int L, int nch, int c0, int ncl) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ __align__(16) uint8_t smraw[];
  WySmem& s = *reinterpret_cast<WySmem*>(smraw);
  // this launch covers chunks c0 .. c0 + ncl - 1 of every request
  const int b = blockIdx.x / ncl, c = c0 + (int)(blockIdx.x % ncl);
  const int cg = b * nch + c;          // global chunk index
  const int h = blockIdx.y;            // value head
  const int64_t t0 = (int64_t)b * L + (int64_t)c * C;
  const int64_t blk = (int64_t)cg * HV + h;   // output block
  const int nvalid = min(C, L - c * C);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  // Q and K (key head h/2) rows, zero past the request's end; V (head h) comes later, into the
  // space of the fp32 T once that is consumed
  for (int i = tid; i < C * (D / 8); i += 128) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    const bool ok = r < nvalid;
    const int64_t rr = ok ? t0 + r : t0;
    cp_async16(smem_u32(&s.u.Q[r][c8]), qq + rr * (HK * D) + (h >> 1) * D + c8, ok);
    cp_async16(smem_u32(&s.K[r][c8]), kk + rr * (HK * D) + (h >> 1) * D + c8, ok);
  }
  cp_async_commit();
  if (warp == 0) {
    // inclusive prefix sum of g over the chunk (2 rows per lane)
    const int r0 = 2 * lane, r1 = 2 * lane + 1;
    const float g0 = r0 < nvalid ? g[(t0 + r0) * HV + h] : 0.f;
    const float g1 = r1 < nvalid ? g[(t0 + r1) * HV + h] : 0.f;
    const float pair = g0 + g1;
    float incl = pair;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += o;
    }
    const float excl = incl - pair;
    s.gc[r0] = excl + g0;
    s.gc[r1] = incl;
    s.bt[r0] = r0 < nvalid ? beta[(t0 + r0) * HV + h] : 0.f;
    s.bt[r1] = r1 < nvalid ? beta[(t0 + r1) * HV + h] : 0.f;
  }
  cp_async_wait<0>();
  __syncthreads();
  const float gC = s.gc[C - 1];  // rows past the end add g = 0, so this is the chunk's last g
  if (tid < C) {
    const float e = __expf(s.gc[tid]);
    ef[blk * C + tid] = e;       // for the state pass
    s.eb[tid] = s.bt[tid] * e;
    s.ed[tid] = __expf(gC - s.gc[tid]);
  }
  __syncthreads();

  const uint32_t sK = smem_u32(&s.K[0][0]);
  // Aqk = tril(q_r . k_s e^{g_r - g_s}) / sqrt(128), stored transposed ([s][r])
  {
    const uint32_t sQ = smem_u32(&s.u.Q[0][0]);
    float acc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a[4];
      ldsm_x4(a, a_addr(sQ, LDH, warp * 16, ks * 16, lane));
#pragma unroll
      for (int n = 0; n < 8; n += 2) {
        uint32_t bq[4];
        ldsm_x4(bq, bn_addr(sK, LDH, n * 8, ks * 16, lane));
        mma16816(acc[n], a, bq[0], bq[1]);
        mma16816(acc[n + 1], a, bq[2], bq[3]);
      }
    }
    __half* at = AqkT + blk * C * C;
    const float scale = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = warp * 16 + gq + hf * 8;
        const int col = n * 8 + 2 * tq;
        const float v0 = (col <= r) ? __expf(s.gc[r] - s.gc[col]) * acc[n][2 * hf] * scale : 0.f;
        const float v1 =
            (col + 1 <= r) ? __expf(s.gc[r] - s.gc[col + 1]) * acc[n][2 * hf + 1] * scale : 0.f;
        at[col * C + r] = __float2half_rn(v0);
        at[(col + 1) * C + r] = __float2half_rn(v1);
      }
    }
  }
  // decayed keys exp(g_C - g_r) k_r, 16 bytes per store
  for (int i = tid; i < C * (D / 8); i += 128) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    const uint4 kv = *reinterpret_cast<const uint4*>(&s.K[r][c8]);
    const __half2* kh = reinterpret_cast<const __half2*>(&kv);
    const float e = s.ed[r];
    uint4 o;
    uint32_t* op = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __half22float2(kh[j]);
      op[j] = h2u(e * f.x, e * f.y);
    }
    *reinterpret_cast<uint4*>(Kdout + (blk * C + r) * D + c8) = o;
  }
  __syncthreads();  // Q is dead: A takes its place
  // A = strict_tril(beta_r e^{g_r - g_s} k_r . k_s)
  {
    float acc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a[4];
      ldsm_x4(a, a_addr(sK, LDH, warp * 16, ks * 16, lane));
#pragma unroll
      for (int n = 0; n < 8; n += 2) {
        uint32_t bq[4];
        ldsm_x4(bq, bn_addr(sK, LDH, n * 8, ks * 16, lane));
        mma16816(acc[n], a, bq[0], bq[1]);
        mma16816(acc[n + 1], a, bq[2], bq[3]);
      }
    }
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = warp * 16 + gq + hf * 8;
        const int col = n * 8 + 2 * tq;
        const float br = s.bt[r];
        s.u.A[r][col] = (col < r) ? br * __expf(s.gc[r] - s.gc[col]) * acc[n][2 * hf] : 0.f;
        s.u.A[r][col + 1] =
            (col + 1 < r) ? br * __expf(s.gc[r] - s.gc[col + 1]) * acc[n][2 * hf + 1] : 0.f;
      }
    }
  }
  __syncthreads();
  // T, diagonal blocks: warp w inverts I + A_ww, lane j < 16 owning column j of the block
  if (lane < 16) {
    const int base = 16 * warp;
    float t[16];
#pragma unroll
    for (int r = 0; r < 16; ++r) t[r] = (r == lane) ? 1.f : 0.f;
#pragma unroll
    for (int r = 1; r < 16; ++r) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int j = 0; j < r; ++j) {
        if (j & 1) a1 += s.u.A[base + r][base + j] * t[j];
        else a0 += s.u.A[base + r][base + j] * t[j];
      }
      if (r > lane) t[r] = -(a0 + a1);
    }
#pragma unroll
    for (int r = 0; r < 16; ++r) s.tv.Tf[base + r][base + lane] = t[r];
  }
  __syncthreads();
  // T, off-diagonal blocks at distance d: block (i, j = i - d); thread (block, column cc, row
  // half rh) forms column cc of X = sum_k A_ik T_kj, then rows 8 rh .. 8 rh + 7 of -T_ii X
#pragma unroll 1
  for (int d = 1; d < 4; ++d) {
    if (tid < (4 - d) * 32) {
      const int j = tid >> 5, i = j + d;
      const int cc = lane & 15, rh = lane >> 4;
      const int i0 = 16 * i, colg = 16 * j + cc;
      float x[16];
#pragma unroll
      for (int r = 0; r < 16; ++r) x[r] = 0.f;
      for (int kq = 4 * j; kq < 4 * i; ++kq) {   // 4 columns of A_i. (rows of T_.j) per step
        float tv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) tv[e] = s.tv.Tf[4 * kq + e][colg];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          const float4 av = *reinterpret_cast<const float4*>(&s.u.A[i0 + r][4 * kq]);
          x[r] += av.x * tv[0] + av.y * tv[1] + av.z * tv[2] + av.w * tv[3];
        }
      }
#pragma unroll
      for (int rr = 0; rr < 8; ++rr) {
        const int r = 8 * rh + rr;
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
          const float4 tvv = *reinterpret_cast<const float4*>(&s.tv.Tf[i0 + r][i0 + m]);
          acc += tvv.x * x[m] + tvv.y * x[m + 1] + tvv.z * x[m + 2] + tvv.w * x[m + 3];
        }
        s.tv.Tf[i0 + r][colg] = -acc;
      }
    }
    __syncthreads();
  }
  // A is dead: T diag(beta e^g) and T diag(beta) in fp16 (blocks above the diagonal are zero)
  for (int i = tid; i < C * C; i += 128) {
    const int r = i / C, sc = i % C;
    const float tv = (sc >> 4) > (r >> 4) ? 0.f : s.tv.Tf[r][sc];
    s.u.t.Tw[r][sc] = __float2half_rn(tv * s.eb[sc]);
    s.u.t.Tu[r][sc] = __float2half_rn(tv * s.bt[sc]);
  }
  __syncthreads();
  // the fp32 T is dead: V's rows into its space, landing while W = T diag(beta e^g) K runs
  for (int i = tid; i < C * (D / 8); i += 128) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    const bool ok = r < nvalid;
    const int64_t rr = ok ? t0 + r : t0;
    cp_async16(smem_u32(&s.tv.V[r][c8]), vv + rr * (HV * D) + h * D + c8, ok);
  }
  cp_async_commit();
  // W = T diag(beta e^g) K and U' = T diag(beta) V  (rows 16w.., all 128 columns)
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    if (which == 1) {
      cp_async_wait<0>();
      __syncthreads();   // V has landed for every thread
    }
    const uint32_t sT = smem_u32(which == 0 ? &s.u.t.Tw[0][0] : &s.u.t.Tu[0][0]);
    const uint32_t sB = smem_u32(which == 0 ? &s.K[0][0] : &s.tv.V[0][0]);
    float acc[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < C / 16; ++ks) {
      uint32_t a[4];
      ldsm_x4(a, a_addr(sT, C + 8, warp * 16, ks * 16, lane));
#pragma unroll
      for (int n = 0; n < 16; n += 2) {
        uint32_t bq[4];
        ldsm_x4_t(bq, bk_addr(sB, LDH, n * 8, ks * 16, lane));
        mma16816(acc[n], a, bq[0], bq[1]);
        mma16816(acc[n + 1], a, bq[2], bq[3]);
      }
    }
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = warp * 16 + gq + half * 8;
      const int64_t row = blk * C + r;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const int col = n * 8 + 2 * tq;
        if (which == 0) {
          *reinterpret_cast<uint32_t*>(Wout + row * D + col) = h2u(acc[n][2 * half], acc[n][2 * half + 1]);
        } else {
          *reinterpret_cast<float2*>(Uout + row * D + col) = make_float2(acc[n][2 * half], acc[n][2 * half + 1]);
        }
      }
    }
  }
}

// ------------------------------------------------------------------------------------------
// Output gate of the decoder layer: y[t, h*128 + i] = RMSNorm_128(o[t, h, :])_i * w_i * SiLU(z).
// One CTA (256 threads) per token; 8 threads x 16 values per head.
// ------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(256) gdn_gated_norm_kernel(const __half* __restrict__ o,
                                                             const __half* __restrict__ z,
                                                             int64_t ldz,
                                                             const __half* __restrict__ w,
                                                             __half* __restrict__ y, int64_t ldy) {
  pdl_trigger();
  pdl_wait();
  const int64_t tok = blockIdx.x;
  const int c0 = threadIdx.x * 16;            // 16 consecutive values of head c0 / 128
  float ov[16], zv[16];
  {
    const uint4* op = reinterpret_cast<const uint4*>(o + tok * (HV * D) + c0);
    const uint4* zp = reinterpret_cast<const uint4*>(z + tok * ldz + c0);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      uint4 a = op[i], bz = zp[i];
      const __half2* ah = reinterpret_cast<const __half2*>(&a);
      const __half2* zh = reinterpret_cast<const __half2*>(&bz);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 fa = __half22float2(ah[j]), fz = __half22float2(zh[j]);
        ov[8 * i + 2 * j] = fa.x; ov[8 * i + 2 * j + 1] = fa.y;
        zv[8 * i + 2 * j] = fz.x; zv[8 * i + 2 * j + 1] = fz.y;
      }
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) ss += ov[i] * ov[i];
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  ss += __shfl_xor_sync(0xffffffffu, ss, 4);
  const float inv = rsqrtf(ss * (1.f / D) + 1e-6f);
  const int wi = c0 % D;
  uint32_t pk[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const float2 wf = __half22float2(*reinterpret_cast<const __half2*>(w + wi + 2 * j));
    pk[j] = h2u(ov[2 * j] * inv * wf.x * silu_f(zv[2 * j]),
                ov[2 * j + 1] * inv * wf.y * silu_f(zv[2 * j + 1]));
  }
  uint4* yp = reinterpret_cast<uint4*>(y + tok * ldy + c0);
  yp[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  yp[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
}

}  // namespace gdn

static inline size_t al256g(size_t x) { return (x + 255) & ~size_t(255); }

// A long scan of one request runs in pieces of chunks: the chunk phase of piece p + 1 (many
// CTAs) overlaps the sequential state pass of piece p (one CTA per value head, which leaves most
// SMs idle), on two streams ordered by events.  Pieces of at least 32 chunks.
int gdn_pieces(int64_t B, int64_t L) {
  const int64_t nch = (L + gdn::C - 1) / gdn::C;
  if (B > 1 || nch < 64) return 1;
  return (int)std::min<int64_t>(8, nch / 32);
}

size_t gdn_scan_workspace_bytes(int64_t B, int64_t L, bool with_norm) {
  const int64_t M = B * L;
  const int64_t nch = (L + gdn::C - 1) / gdn::C;
  size_t n = 0;
  n += al256g(M * gdn::HV * 4);                          // g (from alpha)
  n += al256g(B * nch * gdn::HV * gdn::C * 4);           // exp(g) per chunk row
  const int64_t rows = B * nch * gdn::C;                 // whole chunks
  n += al256g(rows * gdn::HV * gdn::D * 2);              // W
  n += al256g(rows * gdn::HV * gdn::D * 4);              // U'
  n += al256g(rows * gdn::HV * gdn::D * 2);              // decayed keys
  n += al256g(B * nch * gdn::HV * gdn::C * gdn::C * 2);  // Aqk
  if (gdn_pieces(B, L) > 1) n += al256g(B * gdn::HV * gdn::D * gdn::D * 4);   // carried state
  if (with_norm) n += al256g(M * gdn::HV * gdn::D * 2);  // o before the output gate (last)
  return n;
}

struct GdnWs {
  float* g;
  float* ef;
  __half* W;
  float* U1;
  __half* Kt;
  __half* Aqk;
  __half* o;
  float* state;
};
static GdnWs carve(void* ws, int64_t B, int64_t L) {
  const int64_t M = B * L;
  const int64_t nch = (L + gdn::C - 1) / gdn::C;
  uint8_t* p = static_cast<uint8_t*>(ws);
  GdnWs w;
  w.g = reinterpret_cast<float*>(p); p += al256g(M * gdn::HV * 4);
  w.ef = reinterpret_cast<float*>(p); p += al256g(B * nch * gdn::HV * gdn::C * 4);
  const int64_t rows = B * nch * gdn::C;
  w.W = reinterpret_cast<__half*>(p); p += al256g(rows * gdn::HV * gdn::D * 2);
  w.U1 = reinterpret_cast<float*>(p); p += al256g(rows * gdn::HV * gdn::D * 4);
  w.Kt = reinterpret_cast<__half*>(p); p += al256g(rows * gdn::HV * gdn::D * 2);
  w.Aqk = reinterpret_cast<__half*>(p); p += al256g(B * nch * gdn::HV * gdn::C * gdn::C * 2);
  // same order as gdn_scan_workspace_bytes: the carried state only when the scan runs in pieces,
  // o (only with the gated norm) last
  w.state = nullptr;
  if (gdn_pieces(B, L) > 1) {
    w.state = reinterpret_cast<float*>(p);
    p += al256g(B * gdn::HV * gdn::D * gdn::D * 4);
  }
  w.o = reinterpret_cast<__half*>(p);
  return w;
}

static clef_status gdn_set_attrs() {
  static std::atomic<uint64_t> attr{0};
  CLEF_CUDA_CHECK(smem_opt_in((const void*)gdn::gdn_chunk_wy_kernel, sizeof(gdn::WySmem), &attr));
  return CLEF_OK;
}

clef_status gdn_prep_launch(const __half* proj, int64_t ldp, const __half* conv_w,
                            const __half* conv_in, __half* q, __half* k, __half* v, int64_t M,
                            int64_t L, cudaStream_t stream) {
  if (M == 0) return CLEF_OK;
  TraceScope ts(stream, "gdn_prep", 0.0, M * (8192.0 * 2 + 8192 * 2));
  static std::atomic<uint64_t> attr{0};
  CLEF_CUDA_CHECK(smem_opt_in((const void*)gdn::gdn_prep_kernel, gdn::PREP_SMEM, &attr));
  const int64_t n_tiles = (8192 / gdn::PREP_CH) * ((M + gdn::PREP_T - 1) / gdn::PREP_T);
  const int64_t grid = std::min<int64_t>(n_tiles, (int64_t)gdn::PREP_CTAS_PER_SM * num_sms());
  CLEF_CUDA_CHECK(launch_pdl(gdn::gdn_prep_kernel, dim3((unsigned)grid), dim3(256), gdn::PREP_SMEM, stream,
       proj, ldp, conv_w, conv_in, q, k, v,
       M, (int)L, n_tiles));
  return CLEF_OK;
}

clef_status conv_state_launch(const __half* proj, int64_t ldp, __half* state, int64_t B,
                              int64_t L, cudaStream_t stream) {
  if (B == 0) return CLEF_OK;
  TraceScope ts(stream, "conv_state", 0.0, (double)B * 3 * 8192 * 2 * 2);
  const int64_t n = B * (8192 / 8);
  CLEF_CUDA_CHECK(launch_pdl(gdn::conv_state_kernel, dim3((unsigned)std::min<int64_t>((n + 255) / 256, 4096)), dim3(256), 0, stream,
       proj, ldp, state, B, (int)L));
  return CLEF_OK;
}

// Two internal streams per device (high priority for the latency-bound state pass, low for the
// chunk phase) and the events that order them, created on first use and kept for the process.
// The caller holds `lock` while it enqueues, so the events are never re-recorded by another
// thread before the waits on them have been enqueued.
struct SideStreams {
  cudaStream_t hi = nullptr, lo = nullptr;
  cudaEvent_t ev[12] = {};
};
static std::mutex g_side_mu;
static clef_status side_streams(SideStreams** out, std::unique_lock<std::mutex>* lock) {
  static SideStreams per_dev[64];
  static bool made[64] = {};
  int dev = 0;
  CLEF_CUDA_CHECK(cudaGetDevice(&dev));
  if (dev < 0 || dev >= 64) {
    set_error("device index %d out of range", dev);
    return CLEF_E_CUDA;
  }
  *lock = std::unique_lock<std::mutex>(g_side_mu);
  if (!made[dev]) {
    int least = 0, greatest = 0;
    CLEF_CUDA_CHECK(cudaDeviceGetStreamPriorityRange(&least, &greatest));
    SideStreams& s = per_dev[dev];
    CLEF_CUDA_CHECK(cudaStreamCreateWithPriority(&s.hi, cudaStreamNonBlocking, greatest));
    CLEF_CUDA_CHECK(cudaStreamCreateWithPriority(&s.lo, cudaStreamNonBlocking, least));
    for (auto& e : s.ev) CLEF_CUDA_CHECK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));
    made[dev] = true;
  }
  *out = &per_dev[dev];
  return CLEF_OK;
}

clef_status gdn_scan_launch(const __half* q, const __half* k, const __half* v, const float* g,
                            const float* alpha, const float* beta, const float* s0, float* s_out,
                            const __half* z, int64_t ldz, const __half* o_norm, __half* out,
                            int64_t ldo, int64_t B, int64_t L, void* ws, cudaStream_t stream) {
  if (B == 0 || L == 0) return CLEF_OK;
  clef_status st = gdn_set_attrs();
  if (st != CLEF_OK) return st;
  GdnWs w = carve(ws, B, L);
  const int64_t M = B * L;
  const int nch = (int)((L + gdn::C - 1) / gdn::C);
  if (!g) {
    const int64_t n = M * gdn::HV;
    CLEF_CUDA_CHECK(launch_pdl(gdn::log_alpha_kernel, dim3((unsigned)std::min<int64_t>((n + 255) / 256, 4096)), dim3(256), 0, stream,
         alpha, w.g, n));
    g = w.g;
  }
  __half* o = z ? w.o : out;
  const int64_t ldo_pass = z ? (int64_t)gdn::HV * gdn::D : ldo;
  auto chunk_phase = [&](int64_t c0, int64_t ncl, cudaStream_t s) -> clef_status {
    const double C = gdn::C, D = gdn::D, HVd = gdn::HV, nchunks = (double)B * ncl;
    TraceScope ts(s, "gdn_chunk_wy", nchunks * HVd * 8.0 * C * C * D,
                  nchunks * C * HVd * D * (2 + 2 + 2 + 2 + 4) + nchunks * HVd * C * C * 2);
    CLEF_CUDA_CHECK(launch_pdl(gdn::gdn_chunk_wy_kernel, dim3(dim3((unsigned)(B * ncl), gdn::HV)), dim3(128), sizeof(gdn::WySmem), s,
         q, k, v, g, beta, w.ef, w.W, w.U1, w.Kt, w.Aqk, (int)L, nch, (int)c0, (int)ncl));
    return CLEF_OK;
  };
  const int pieces = gdn_pieces(B, L);
  if (pieces <= 1) {
    st = chunk_phase(0, nch, stream);
    if (st != CLEF_OK) return st;
    st = gdn_state_launch(q, w.Kt, w.W, w.U1, w.Aqk, w.ef, s0, s_out, o, ldo_pass, B, L, stream);
    if (st != CLEF_OK) return st;
  } else {
    SideStreams* ss = nullptr;
    std::unique_lock<std::mutex> lock;
    st = side_streams(&ss, &lock);
    if (st != CLEF_OK) return st;
    float* s_eff = s_out ? s_out : w.state;
    // fork: both side streams start after everything already queued on `stream`
    CLEF_CUDA_CHECK(cudaEventRecord(ss->ev[0], stream));
    CLEF_CUDA_CHECK(cudaStreamWaitEvent(ss->lo, ss->ev[0], 0));
    CLEF_CUDA_CHECK(cudaStreamWaitEvent(ss->hi, ss->ev[0], 0));
    auto run_pieces = [&]() -> clef_status {
      for (int p = 0; p < pieces; ++p) {
        const int64_t c0 = (int64_t)p * nch / pieces, c1 = (int64_t)(p + 1) * nch / pieces;
        clef_status ps = chunk_phase(c0, c1 - c0, ss->lo);
        if (ps != CLEF_OK) return ps;
        CLEF_CUDA_CHECK(cudaEventRecord(ss->ev[1 + p], ss->lo));
        CLEF_CUDA_CHECK(cudaStreamWaitEvent(ss->hi, ss->ev[1 + p], 0));
        ps = gdn_state_launch(q, w.Kt, w.W, w.U1, w.Aqk, w.ef, p == 0 ? s0 : s_eff, s_eff, o,
                              ldo_pass, B, L, ss->hi, c0, c1 - c0);
        if (ps != CLEF_OK) return ps;
        if (z) {
          // the z-gated norm of this piece's rows, in the state stream's wait for the next
          // chunk phase
          const int64_t t0 = c0 * gdn::C, t1 = std::min<int64_t>(c1 * gdn::C, L);
          for (int64_t b = 0; b < B; ++b) {
            const int64_t r0 = b * L + t0;
            TraceScope ts(ss->hi, "gdn_gated_norm", 0.0, (double)(t1 - t0) * 4096 * 2 * 3);
            CLEF_CUDA_CHECK(launch_pdl(gdn::gdn_gated_norm_kernel, dim3((unsigned)(t1 - t0)), dim3(256), 0, ss->hi,
                 o + r0 * ldo_pass, z + r0 * ldz, ldz, o_norm, out + r0 * ldo, ldo));
          }
        }
      }
      return CLEF_OK;
    };
    st = run_pieces();
    // join, also after an error part way: whatever was queued on the side streams is ordered
    // before later work on the caller's stream (which may free or reuse the workspace)
    CLEF_CUDA_CHECK(cudaEventRecord(ss->ev[1 + pieces], ss->hi));
    CLEF_CUDA_CHECK(cudaEventRecord(ss->ev[2 + pieces], ss->lo));
    CLEF_CUDA_CHECK(cudaStreamWaitEvent(stream, ss->ev[1 + pieces], 0));
    CLEF_CUDA_CHECK(cudaStreamWaitEvent(stream, ss->ev[2 + pieces], 0));
    if (st != CLEF_OK) return st;
  }
  if (z && pieces <= 1) {
    TraceScope ts(stream, "gdn_gated_norm", 0.0, (double)M * 4096 * 2 * 3);
    CLEF_CUDA_CHECK(launch_pdl(gdn::gdn_gated_norm_kernel, dim3((unsigned)M), dim3(256), 0, stream,
         o, z, ldz, o_norm, out, ldo));
  }
  return CLEF_OK;
}

}  // namespace clef

// Host only: where the scan's workspace regions start (bytes from the workspace base), for
// checking the carving against the size query without a GPU.
extern "C" clef_status clef_debug_gdn_workspace_layout(int64_t B, int64_t L, int32_t with_norm,
                                                       int64_t* offsets, int64_t* total) {
  using namespace clef;
  if (!offsets || !total || B < 1 || L < 1) return CLEF_E_INVALID;
  uint8_t* const base = reinterpret_cast<uint8_t*>(uintptr_t(1) << 20);   // never dereferenced
  const GdnWs w = carve(base, B, L);
  const void* regions[8] = {w.g, w.ef, w.W, w.U1, w.Kt, w.Aqk, w.state, w.o};
  for (int i = 0; i < 8; ++i)
    offsets[i] = regions[i] ? (int64_t)(static_cast<const uint8_t*>(regions[i]) - base) : -1;
  if (!with_norm) offsets[7] = -1;
  *total = (int64_t)gdn_scan_workspace_bytes(B, L, with_norm != 0);
  return CLEF_OK;
}

