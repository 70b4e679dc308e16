// Gated DeltaNet: input preparation and the chunked scan.
//
// The recurrence ("Clef-Flash-ANE-LUT6" model card, "Model architecture"; "clef-flash - Core AI"
// README, "Core AI shape": a [32, 128, 128] state per GDN layer), for value head h reading key
// head h/2:
//     S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,   o_t = S_t q_t / sqrt(128)
// is evaluated in chunks of C = 64 positions ("clef-flash-LiteRT" README, "Provenance": the
// recurrence re-expressed as a chunked kernel of 64 positions).  With g the cumulative
// log(alpha) inside a chunk and S0 the state entering it:
//     A = strict_tril(diag(beta) (exp(g_r - g_s)) o K K^T),   T = (I + A)^-1
//     W = T diag(beta exp(g)) K,   U' = T diag(beta) V,   U = U' - W S0^T
//     O = (diag(exp(g)) Q S0^T + (tril(Q K^T) o exp(g_r - g_s)) U) / sqrt(128)
//     S_C = exp(g_C) S0 + U^T diag(exp(g_C - g)) K
// Kernels:
//   gdn_chunk_wy    (parallel over chunks x heads): cumulative g, T by forward substitution,
//                   W, U', the decayed keys exp(g_C - g) k and the intra-chunk matrix
//                   Aqk = tril(Q K^T) o exp(g_r - g_s) / sqrt(128)
//   gdn_state_pass  (sequential over chunks; one warp per 16 value rows of a head): the state
//                   slice stays in mma accumulators and is reused in registers as the fp16
//                   operand S0^T; per chunk U = U' - W S0^T, O = exp(g) Q S0^T / sqrt(128) + Aqk U,
//                   S <- exp(g_C) S + U^T Kd, with U transposed in registers (movmatrix)
//   gdn_gated_norm  (decoder layer only): y = RMSNorm_128(O) * w_o * SiLU(z)
// All products run on tensor cores (mma.sync m16n8k16, fp16 inputs, fp32 accumulation); the
// state and the scalars stay fp32.
#include <algorithm>

#include "common.cuh"
#include "gdn.cuh"
#include "mma.cuh"

namespace clef {
namespace gdn {

constexpr int C = 64;          // chunk width
constexpr int D = 128;         // head size (key and value)
constexpr int HV = 32;         // value heads
constexpr int HK = 16;         // key heads
constexpr int LDH = D + 8;     // padded fp16 row (272 bytes) for conflict-free ldmatrix
constexpr float kLogAlphaMin = -30.0f;

// ------------------------------------------------------------------------------------------
// Prep for the decoder layer: causal depthwise conv (4 taps) + SiLU over the 8192 QKV channels and
// the per-head L2 norm of q and k.  A CTA covers 16 consecutive tokens for 1024 channels (128
// threads x 8 channels); each thread issues the loads of all 19 rows it needs at once and keeps
// them in registers.  The gates come from the a/b projection's epilogue.
// proj [M, ldp] fp16: q 0..2047 | k 2048..4095 | v 4096..8191 (| z 8192..).
// ------------------------------------------------------------------------------------------
constexpr int PREP_T = 16;
__global__ void __launch_bounds__(128) gdn_prep_kernel(
    const __half* __restrict__ proj, int64_t ldp, const __half* __restrict__ conv_w,
    __half* __restrict__ q, __half* __restrict__ k, __half* __restrict__ v, int64_t M, int L) {
  const int tid = threadIdx.x;
  const int ch0 = blockIdx.x * 1024 + tid * 8;
  const int64_t tok0 = (int64_t)blockIdx.y * PREP_T;
  float w[8][4];
  {
    const uint4* wp = reinterpret_cast<const uint4*>(conv_w + (int64_t)ch0 * 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      uint4 u = wp[i];
      const __half* hh = reinterpret_cast<const __half*>(&u);
#pragma unroll
      for (int j = 0; j < 8; ++j) w[(i * 8 + j) / 4][(i * 8 + j) % 4] = __half2float(hh[j]);
    }
  }
  // rows tok0 - 3 .. tok0 + PREP_T - 1, all loads in flight at once; rows before the start of
  // their request or past M are zero
  uint4 xr[PREP_T + 3];
  const int pos0 = (int)(tok0 % L);
#pragma unroll
  for (int i = 0; i < PREP_T + 3; ++i) {
    const int64_t tok = tok0 - 3 + i;
    const bool ok = (i >= 3 || pos0 >= 3 - i) && tok < M;
    xr[i] = ok ? *reinterpret_cast<const uint4*>(proj + tok * ldp + ch0) : make_uint4(0, 0, 0, 0);
  }
#pragma unroll
  for (int i = 0; i < PREP_T; ++i) {
    const int64_t tok = tok0 + i;
    if (tok >= M) break;
    const int pos = (int)(tok % L);
    float y[8];
#pragma unroll
    for (int c2 = 0; c2 < 4; ++c2) {
      float2 xs[4];
#pragma unroll
      for (int tap = 0; tap < 4; ++tap) {
        // tap j multiplies x[t - 3 + j]; positions before the request's start are zero
        const uint4 u = xr[i + tap];
        const __half2 hv = reinterpret_cast<const __half2*>(&u)[c2];
        xs[tap] = (pos - 3 + tap >= 0) ? __half22float2(hv) : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int c = 2 * c2 + e;
        const float pre = w[c][0] * (e ? xs[0].y : xs[0].x) + w[c][1] * (e ? xs[1].y : xs[1].x) +
                          w[c][2] * (e ? xs[2].y : xs[2].x) + w[c][3] * (e ? xs[3].y : xs[3].x);
        y[c] = silu_f(pre);
      }
    }
    __half* dst;
    if (ch0 < 4096) {
      // q or k: a head is 128 channels = 16 consecutive threads
      float ss = 0.f;
#pragma unroll
      for (int c = 0; c < 8; ++c) ss += y[c] * y[c];
#pragma unroll
      for (int off = 1; off < 16; off <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      const float r = rsqrtf(ss + 1e-6f);
#pragma unroll
      for (int c = 0; c < 8; ++c) y[c] *= r;
      dst = ch0 < 2048 ? q + tok * 2048 + ch0 : k + tok * 2048 + (ch0 - 2048);
    } else {
      dst = v + tok * 4096 + (ch0 - 4096);
    }
    *reinterpret_cast<uint4*>(dst) =
        make_uint4(h2u(y[0], y[1]), h2u(y[2], y[3]), h2u(y[4], y[5]), h2u(y[6], y[7]));
  }
}

// g = log(alpha), clamped, for callers that pass alpha itself.
__global__ void log_alpha_kernel(const float* __restrict__ alpha, float* __restrict__ g, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float a = alpha[i];
    g[i] = a > 0.f ? fmaxf(logf(a), kLogAlphaMin) : kLogAlphaMin;
  }
}

// ------------------------------------------------------------------------------------------
// Phase 1: per (chunk, value head): cumulative g, T = (I + A)^-1, W = T diag(beta e^g) K,
// U' = T diag(beta) V.  128 threads; warp w owns rows 16w .. 16w+15 of every 64-row product.
// ------------------------------------------------------------------------------------------
struct WySmem {
  __half Q[C][LDH];
  __half K[C][LDH];    // K, then beta * exp(g) * K in place
  __half V[C][LDH];    // V, then beta * V in place
  __half T[C][C + 8];  // (I + A)^-1 in fp16 for the products
  float A[C][C + 4];   // 16-byte aligned rows for broadcast float4 reads
  float gc[C];
  float bt[C];
  float eb[C];         // beta_r exp(g_r)
  float ed[C];         // exp(g_C - g_r)
};

__global__ void __launch_bounds__(128) gdn_chunk_wy_kernel(
    const __half* __restrict__ qq, const __half* __restrict__ kk, const __half* __restrict__ vv,
    const float* __restrict__ g, const float* __restrict__ beta, float* __restrict__ gcum,
    __half* __restrict__ Wout, float* __restrict__ Uout, __half* __restrict__ Ktout,
    __half* __restrict__ Aqk, int L, int nch) {
  extern __shared__ __align__(16) uint8_t smraw[];
  WySmem& s = *reinterpret_cast<WySmem*>(smraw);
  const int cg = blockIdx.x;           // global chunk index = b * nch + c
  const int h = blockIdx.y;            // value head
  const int b = cg / nch, c = cg % nch;
  const int64_t t0 = (int64_t)b * L + (int64_t)c * C;
  const int nvalid = min(C, L - c * C);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  // Q, K (key head h/2) and V (head h) rows, zero past the request's end
  for (int i = tid; i < C * (D / 8); i += 128) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    const bool ok = r < nvalid;
    const int64_t rr = ok ? t0 + r : t0;
    cp_async16(smem_u32(&s.Q[r][c8]), qq + rr * (HK * D) + (h >> 1) * D + c8, ok);
    cp_async16(smem_u32(&s.K[r][c8]), kk + rr * (HK * D) + (h >> 1) * D + c8, ok);
    cp_async16(smem_u32(&s.V[r][c8]), vv + rr * (HV * D) + h * D + c8, ok);
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
  if (tid < C && tid < nvalid) gcum[(t0 + tid) * HV + h] = s.gc[tid];
  const float gC = s.gc[C - 1];  // rows past the end add g = 0, so this is the chunk's last g
  if (tid < C) {
    s.eb[tid] = s.bt[tid] * __expf(s.gc[tid]);
    s.ed[tid] = __expf(gC - s.gc[tid]);
  }

  const uint32_t sK = smem_u32(&s.K[0][0]);
  const uint32_t sQ = smem_u32(&s.Q[0][0]);
  // A = strict_tril(beta_r e^{g_r - g_s} k_r . k_s) and Aqk = tril(q_r . k_s e^{g_r - g_s}) / sqrt(128)
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    const uint32_t sA = which == 0 ? sK : sQ;
    float acc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a[4];
      ldsm_x4(a, a_addr(sA, LDH, warp * 16, ks * 16, lane));
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
        const float d0 = __expf(s.gc[r] - s.gc[col]), d1 = __expf(s.gc[r] - s.gc[col + 1]);
        if (which == 0) {
          s.A[r][col] = (col < r) ? s.bt[r] * d0 * acc[n][2 * hf] : 0.f;
          s.A[r][col + 1] = (col + 1 < r) ? s.bt[r] * d1 * acc[n][2 * hf + 1] : 0.f;
        } else {
          const float scale = 0.08838834764831845f;  // 1 / sqrt(128)
          const float v0 = (col <= r) ? d0 * acc[n][2 * hf] * scale : 0.f;
          const float v1 = (col + 1 <= r) ? d1 * acc[n][2 * hf + 1] * scale : 0.f;
          *reinterpret_cast<uint32_t*>(Aqk + (((int64_t)cg * HV + h) * C + r) * C + col) = h2u(v0, v1);
        }
      }
    }
  }
  __syncthreads();
  // decayed keys to global; K -> beta e^g K and V -> beta V in place
  for (int i = tid; i < C * (D / 2); i += 128) {
    const int r = i / (D / 2), c2 = (i % (D / 2)) * 2;
    const float eb = s.eb[r], ed = s.ed[r];
    const float2 kf = __half22float2(*reinterpret_cast<const __half2*>(&s.K[r][c2]));
    const float2 vf = __half22float2(*reinterpret_cast<const __half2*>(&s.V[r][c2]));
    *reinterpret_cast<__half2*>(&s.K[r][c2]) = __floats2half2_rn(eb * kf.x, eb * kf.y);
    *reinterpret_cast<__half2*>(&s.V[r][c2]) = __floats2half2_rn(s.bt[r] * vf.x, s.bt[r] * vf.y);
    if (r < nvalid)
      *reinterpret_cast<__half2*>(Ktout + ((t0 + r) * HV + h) * D + c2) =
          __floats2half2_rn(ed * kf.x, ed * kf.y);
  }
  __syncthreads();
  // T = (I + A)^-1 by forward substitution: T[r][sc] = -sum_{j<r} A[r][j] T[j][sc] (r > sc).
  // Column sc depends only on earlier rows of the same column: thread sc keeps its column in
  // registers and all 64 threads read each A row as the same (broadcast) float4s.  A is zero on
  // and above the diagonal, so whole float4s can be read past j = r.
  if (tid < C) {
    const int sc = tid;
    float tcol[C];
#pragma unroll
    for (int r = 0; r < C; ++r) tcol[r] = (r == sc) ? 1.f : 0.f;
#pragma unroll
    for (int r = 1; r < C; ++r) {
      float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
      for (int j = 0; j < r; j += 4) {
        const float4 av = *reinterpret_cast<const float4*>(&s.A[r][j]);
        a0 += av.x * tcol[j];
        a1 += av.y * tcol[j + 1];
        a2 += av.z * tcol[j + 2];
        a3 += av.w * tcol[j + 3];
      }
      const float val = -((a0 + a1) + (a2 + a3));
      tcol[r] = (r > sc) ? val : tcol[r];
    }
#pragma unroll
    for (int r = 0; r < C; ++r) s.T[r][sc] = __float2half_rn(tcol[r]);
  }
  __syncthreads();
  // W = T KB and U' = T VB  (rows 16w.., all 128 columns)
  const uint32_t sT = smem_u32(&s.T[0][0]);
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    const uint32_t sB = smem_u32(which == 0 ? &s.K[0][0] : &s.V[0][0]);
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
      if (r >= nvalid) continue;
      const int64_t row = (t0 + r) * HV + h;
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
// Phase 2: the fused state pass.  CTA = (request, value head, 32 value rows); warp w owns value
// rows 16w.. of that slice.  Per chunk (all data prefetched by cp.async one chunk ahead):
//   SB   = fp16 B fragments of S0^T, taken straight from the fp32 state accumulators
//   U    = U' - W S0^T                               (rows past the end set to zero)
//   UT   = U transposed in registers (movmatrix): A fragments of U^T, B fragments of U
//   O    = exp(g) / sqrt(128) * (Q S0^T) + Aqk U     -> out
//   S   <- exp(g_C) S + U^T Kd
// One barrier per chunk (the two warps share the prefetched tiles).
// ------------------------------------------------------------------------------------------
constexpr int SW = 2;              // warps (16-row value slices) per CTA
struct PassBuf {
  __half W[C][LDH];
  __half Q[C][LDH];
  __half K[C][LDH];       // decayed keys
  __half Aq[C][C + 8];
  float U[SW][C][16 + 4];
  float gc[C];
};
struct PassSmem {
  PassBuf buf[2];
};

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

__device__ __forceinline__ void pass_prefetch(PassBuf& pb, const __half* __restrict__ Wg,
                                              const __half* __restrict__ qq,
                                              const __half* __restrict__ Kt,
                                              const __half* __restrict__ Aqk,
                                              const float* __restrict__ Ug,
                                              const float* __restrict__ gcum, int64_t t0,
                                              int64_t cgi, int nvalid, int h, int dv0, int tid) {
  for (int i = tid; i < C * (D / 8); i += 32 * SW) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    const bool ok = r < nvalid;
    const int64_t rr = ok ? (t0 + r) : t0;
    cp_async16(smem_u32(&pb.W[r][c8]), Wg + (rr * HV + h) * D + c8, ok);
    cp_async16(smem_u32(&pb.Q[r][c8]), qq + rr * (HK * D) + (h >> 1) * D + c8, ok);
    cp_async16(smem_u32(&pb.K[r][c8]), Kt + (rr * HV + h) * D + c8, ok);
  }
  for (int i = tid; i < C * (C / 8); i += 32 * SW) {
    const int r = i / (C / 8), c8 = (i % (C / 8)) * 8;
    cp_async16(smem_u32(&pb.Aq[r][c8]), Aqk + ((cgi * HV + h) * C + r) * C + c8, true);
  }
  for (int i = tid; i < SW * C * 4; i += 32 * SW) {
    const int w = i / (C * 4), r = (i / 4) % C, c4 = (i % 4) * 4;
    const bool ok = r < nvalid;
    const int64_t rr = ok ? (t0 + r) : t0;
    cp_async16(smem_u32(&pb.U[w][r][c4]), Ug + (rr * HV + h) * D + dv0 + 16 * w + c4, ok);
  }
  if (tid < C) {
    // rows past the end repeat the last valid g
    const int64_t rr = t0 + min(tid, nvalid - 1);
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(&pb.gc[tid])),
                 "l"(gcum + rr * HV + h)
                 : "memory");
  }
  cp_async_commit();
}

__global__ void __launch_bounds__(32 * SW) gdn_state_pass_kernel(
    const __half* __restrict__ qq, const __half* __restrict__ Kt, const __half* __restrict__ Wg,
    const float* __restrict__ Ug, const __half* __restrict__ Aqk, const float* __restrict__ gcum,
    const float* __restrict__ s0, __half* __restrict__ out, int64_t ldo,
    float* __restrict__ s_out, int L, int nch) {
  extern __shared__ __align__(16) uint8_t smraw[];
  PassSmem& s = *reinterpret_cast<PassSmem*>(smraw);
  constexpr int NSL = D / (16 * SW);     // CTAs per head
  const int sl = blockIdx.x % NSL;
  const int h = (blockIdx.x / NSL) % HV;
  const int b = blockIdx.x / (NSL * HV);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int dv0 = sl * 16 * SW;          // first value row of the CTA
  const int dvw = dv0 + 16 * warp;       // first value row of this warp

  // state slice [16 value rows x 128 key cols]: n-tile nt covers key columns 8nt..8nt+7
  float S[16][4];
#pragma unroll
  for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v0 = 0.f;
      if (s0) {
        const int r = dvw + gq + (e >= 2 ? 8 : 0);
        const int col = nt * 8 + 2 * tq + (e & 1);
        v0 = s0[(((int64_t)b * HV + h) * D + r) * D + col];
      }
      S[nt][e] = v0;
    }
  }
  const int64_t tb = (int64_t)b * L;
  pass_prefetch(s.buf[0], Wg, qq, Kt, Aqk, Ug, gcum, tb, (int64_t)b * nch, min(C, L), h, dv0, tid);
  const float inv_sqrt_d = 0.08838834764831845f;

  for (int c = 0; c < nch; ++c) {
    const int64_t t0 = tb + (int64_t)c * C;
    const int nvalid = min(C, L - c * C);
    PassBuf& pb = s.buf[c & 1];
    cp_async_wait<0>();
    __syncthreads();  // chunk c landed for both warps; both are done with chunk c-1's buffer
    if (c + 1 < nch)
      pass_prefetch(s.buf[(c + 1) & 1], Wg, qq, Kt, Aqk, Ug, gcum, t0 + C, (int64_t)b * nch + c + 1,
                    min(C, L - (c + 1) * C), h, dv0, tid);
    // SB[ks][nv]: B fragments of S0^T for key step ks (16 columns) and value n-tile nv
    uint32_t SB[8][2][2];
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      SB[ks][0][0] = h2u(S[2 * ks][0], S[2 * ks][1]);
      SB[ks][0][1] = h2u(S[2 * ks + 1][0], S[2 * ks + 1][1]);
      SB[ks][1][0] = h2u(S[2 * ks][2], S[2 * ks][3]);
      SB[ks][1][1] = h2u(S[2 * ks + 1][2], S[2 * ks + 1][3]);
    }
    const uint32_t sW = smem_u32(&pb.W[0][0]), sQ = smem_u32(&pb.Q[0][0]);
    const uint32_t sK = smem_u32(&pb.K[0][0]), sA = smem_u32(&pb.Aq[0][0]);
    // U = U' - W S0^T, transposed into UT[mt][nv][2] (fp16): rows tok 16mt.., value rows 8nv..
    uint32_t UT[4][2][2];
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      float acc[2][4];
#pragma unroll
      for (int nv = 0; nv < 2; ++nv) acc[nv][0] = acc[nv][1] = acc[nv][2] = acc[nv][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, a_addr(sW, LDH, mt * 16, ks * 16, lane));
        mma16816(acc[0], a, SB[ks][0][0], SB[ks][0][1]);
        mma16816(acc[1], a, SB[ks][1][0], SB[ks][1][1]);
      }
#pragma unroll
      for (int nv = 0; nv < 2; ++nv) {
        const int r0 = mt * 16 + gq, r1 = r0 + 8;
        const int col = nv * 8 + 2 * tq;
        const float u00 = r0 < nvalid ? pb.U[warp][r0][col] - acc[nv][0] : 0.f;
        const float u01 = r0 < nvalid ? pb.U[warp][r0][col + 1] - acc[nv][1] : 0.f;
        const float u10 = r1 < nvalid ? pb.U[warp][r1][col] - acc[nv][2] : 0.f;
        const float u11 = r1 < nvalid ? pb.U[warp][r1][col + 1] - acc[nv][3] : 0.f;
        UT[mt][nv][0] = movmatrix_t(h2u(u00, u01));
        UT[mt][nv][1] = movmatrix_t(h2u(u10, u11));
      }
    }
    // O = e^g / sqrt(128) * (Q S0^T) + Aqk U
#pragma unroll
    for (int mt = 0; mt < 4; ++mt) {
      float acc[2][4];
#pragma unroll
      for (int nv = 0; nv < 2; ++nv) acc[nv][0] = acc[nv][1] = acc[nv][2] = acc[nv][3] = 0.f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, a_addr(sQ, LDH, mt * 16, ks * 16, lane));
        mma16816(acc[0], a, SB[ks][0][0], SB[ks][0][1]);
        mma16816(acc[1], a, SB[ks][1][0], SB[ks][1][1]);
      }
      const int r0 = mt * 16 + gq, r1 = r0 + 8;
      const float f0 = __expf(pb.gc[r0]) * inv_sqrt_d, f1 = __expf(pb.gc[r1]) * inv_sqrt_d;
#pragma unroll
      for (int nv = 0; nv < 2; ++nv) {
        acc[nv][0] *= f0; acc[nv][1] *= f0; acc[nv][2] *= f1; acc[nv][3] *= f1;
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks) {
        uint32_t a[4];
        ldsm_x4(a, a_addr(sA, C + 8, mt * 16, ks * 16, lane));
        mma16816(acc[0], a, UT[ks][0][0], UT[ks][0][1]);
        mma16816(acc[1], a, UT[ks][1][0], UT[ks][1][1]);
      }
#pragma unroll
      for (int nv = 0; nv < 2; ++nv) {
        const int col = dvw + nv * 8 + 2 * tq;
        if (r0 < nvalid)
          *reinterpret_cast<uint32_t*>(out + (t0 + r0) * ldo + h * D + col) = h2u(acc[nv][0], acc[nv][1]);
        if (r1 < nvalid)
          *reinterpret_cast<uint32_t*>(out + (t0 + r1) * ldo + h * D + col) = h2u(acc[nv][2], acc[nv][3]);
      }
    }
    // S <- e^{g_C} S + U^T Kd
    const float eC = __expf(pb.gc[C - 1]);
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      S[nt][0] *= eC; S[nt][1] *= eC; S[nt][2] *= eC; S[nt][3] *= eC;
    }
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      const uint32_t a[4] = {UT[ks][0][0], UT[ks][1][0], UT[ks][0][1], UT[ks][1][1]};
#pragma unroll
      for (int nt = 0; nt < 16; nt += 2) {
        uint32_t bq[4];
        ldsm_x4_t(bq, bk_addr(sK, LDH, nt * 8, ks * 16, lane));
        mma16816(S[nt], a, bq[0], bq[1]);
        mma16816(S[nt + 1], a, bq[2], bq[3]);
      }
    }
  }
  if (s_out) {
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = dvw + gq + (e >= 2 ? 8 : 0);
        const int col = nt * 8 + 2 * tq + (e & 1);
        s_out[(((int64_t)b * HV + h) * D + r) * D + col] = S[nt][e];
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

size_t gdn_scan_workspace_bytes(int64_t B, int64_t L, bool with_norm) {
  const int64_t M = B * L;
  const int64_t nch = (L + gdn::C - 1) / gdn::C;
  size_t n = 0;
  n += al256g(M * gdn::HV * 4);                          // g (from alpha)
  n += al256g(M * gdn::HV * 4);                          // gcum
  n += al256g(M * gdn::HV * gdn::D * 2);                 // W
  n += al256g(M * gdn::HV * gdn::D * 4);                 // U'
  n += al256g(M * gdn::HV * gdn::D * 2);                 // decayed keys
  n += al256g(B * nch * gdn::HV * gdn::C * gdn::C * 2);  // Aqk
  if (with_norm) n += al256g(M * gdn::HV * gdn::D * 2);  // o before the output gate
  return n;
}

struct GdnWs {
  float* g;
  float* gcum;
  __half* W;
  float* U1;
  __half* Kt;
  __half* Aqk;
  __half* o;
};
static GdnWs carve(void* ws, int64_t B, int64_t L) {
  const int64_t M = B * L;
  const int64_t nch = (L + gdn::C - 1) / gdn::C;
  uint8_t* p = static_cast<uint8_t*>(ws);
  GdnWs w;
  w.g = reinterpret_cast<float*>(p); p += al256g(M * gdn::HV * 4);
  w.gcum = reinterpret_cast<float*>(p); p += al256g(M * gdn::HV * 4);
  w.W = reinterpret_cast<__half*>(p); p += al256g(M * gdn::HV * gdn::D * 2);
  w.U1 = reinterpret_cast<float*>(p); p += al256g(M * gdn::HV * gdn::D * 4);
  w.Kt = reinterpret_cast<__half*>(p); p += al256g(M * gdn::HV * gdn::D * 2);
  w.Aqk = reinterpret_cast<__half*>(p); p += al256g(B * nch * gdn::HV * gdn::C * gdn::C * 2);
  w.o = reinterpret_cast<__half*>(p);
  return w;
}

static bool g_gdn_attr = false;
static clef_status gdn_set_attrs() {
  if (g_gdn_attr) return CLEF_OK;
  CLEF_CUDA_CHECK(cudaFuncSetAttribute(gdn::gdn_chunk_wy_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, sizeof(gdn::WySmem)));
  CLEF_CUDA_CHECK(cudaFuncSetAttribute(gdn::gdn_state_pass_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, sizeof(gdn::PassSmem)));
  g_gdn_attr = true;
  return CLEF_OK;
}

clef_status gdn_prep_launch(const __half* proj, int64_t ldp, const __half* conv_w, __half* q,
                            __half* k, __half* v, int64_t M, int64_t L, cudaStream_t stream) {
  if (M == 0) return CLEF_OK;
  TraceScope ts(stream, "gdn_prep", 0.0, M * (8192.0 * 2 + 8192 * 2));
  dim3 grid(8, (unsigned)((M + gdn::PREP_T - 1) / gdn::PREP_T));
  gdn::gdn_prep_kernel<<<grid, 128, 0, stream>>>(proj, ldp, conv_w, q, k, v, M, (int)L);
  CLEF_LAUNCH_CHECK();
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
    gdn::log_alpha_kernel<<<(unsigned)std::min<int64_t>((n + 255) / 256, 4096), 256, 0, stream>>>(
        alpha, w.g, n);
    CLEF_LAUNCH_CHECK();
    g = w.g;
  }
  dim3 g1((unsigned)(B * nch), gdn::HV);
  const double C = gdn::C, D = gdn::D, HVd = gdn::HV, nchunks = (double)B * nch;
  {
    TraceScope ts(stream, "gdn_chunk_wy", nchunks * HVd * 8.0 * C * C * D,
                  (double)M * HVd * D * (2 + 2 + 2 + 2 + 4) + nchunks * HVd * C * C * 2);
    gdn::gdn_chunk_wy_kernel<<<g1, 128, sizeof(gdn::WySmem), stream>>>(
        q, k, v, g, beta, w.gcum, w.W, w.U1, w.Kt, w.Aqk, (int)L, nch);
    CLEF_LAUNCH_CHECK();
  }
  __half* o = z ? w.o : out;
  const int64_t ldo_pass = z ? (int64_t)gdn::HV * gdn::D : ldo;
  {
    TraceScope ts(stream, "gdn_state_pass",
                  nchunks * HVd * (6.0 * C * D * D + 2.0 * C * C * D),
                  (double)M * HVd * D * (2 + 2 + 4 + 2) + (double)M * 16 * D * 2 +
                      nchunks * HVd * C * C * 2);
    constexpr int nsl = gdn::D / (16 * gdn::SW);
    gdn::gdn_state_pass_kernel<<<(unsigned)(B * gdn::HV * nsl), 32 * gdn::SW,
                                 sizeof(gdn::PassSmem), stream>>>(q, w.Kt, w.W, w.U1, w.Aqk, w.gcum,
                                                                  s0, o, ldo_pass, s_out, (int)L,
                                                                  nch);
    CLEF_LAUNCH_CHECK();
  }
  if (z) {
    TraceScope ts(stream, "gdn_gated_norm", 0.0, (double)M * 4096 * 2 * 3);
    gdn::gdn_gated_norm_kernel<<<(unsigned)M, 256, 0, stream>>>(o, z, ldz, o_norm, out, ldo);
    CLEF_LAUNCH_CHECK();
  }
  return CLEF_OK;
}

}  // namespace clef
