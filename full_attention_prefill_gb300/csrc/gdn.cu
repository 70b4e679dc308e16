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
// Three kernels:
//   gdn_chunk_wy    (parallel over chunks x heads): g, T by forward substitution, W and U'
//   gdn_state_pass  (sequential over chunks, parallel over heads x 8 slices of 16 value rows):
//                   U and the state entering every chunk; the state stays in registers
//   gdn_chunk_out   (parallel over chunks x heads): O, with the z-gated RMSNorm fused in
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
  __half K[C][LDH];
  __half V[C][LDH];
  __half KB[C][LDH];   // beta * exp(g) * K
  __half VB[C][LDH];   // beta * V
  __half T[C][C + 8];  // (I + A)^-1 in fp16 for the products
  float A[C][C + 4];    // 16-byte aligned rows for broadcast float4 reads
  float gc[C];
  float bt[C];
  float eb[C];         // beta_r exp(g_r)
  float ed[C];         // exp(g_C - g_r)
};

__global__ void __launch_bounds__(128) gdn_chunk_wy_kernel(
    const __half* __restrict__ kk, const __half* __restrict__ vv, const float* __restrict__ g,
    const float* __restrict__ beta, float* __restrict__ gcum, __half* __restrict__ Wout,
    float* __restrict__ Uout, __half* __restrict__ Ktout, int L, int nch) {
  extern __shared__ __align__(16) uint8_t smraw[];
  WySmem& s = *reinterpret_cast<WySmem*>(smraw);
  const int cg = blockIdx.x;           // global chunk index = b * nch + c
  const int h = blockIdx.y;            // value head
  const int b = cg / nch, c = cg % nch;
  const int64_t t0 = (int64_t)b * L + (int64_t)c * C;
  const int nvalid = min(C, L - c * C);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // load K (key head h/2) and V (head h) rows, zero past the request's end
  for (int i = tid; i < C * (D / 8); i += 128) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    uint4 ku = make_uint4(0, 0, 0, 0), vu = make_uint4(0, 0, 0, 0);
    if (r < nvalid) {
      ku = *reinterpret_cast<const uint4*>(kk + (t0 + r) * (HK * D) + (h >> 1) * D + c8);
      vu = *reinterpret_cast<const uint4*>(vv + (t0 + r) * (HV * D) + h * D + c8);
    }
    *reinterpret_cast<uint4*>(&s.K[r][c8]) = ku;
    *reinterpret_cast<uint4*>(&s.V[r][c8]) = vu;
  }
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
  __syncthreads();
  if (tid < C && tid < nvalid) gcum[(t0 + tid) * HV + h] = s.gc[tid];

  const uint32_t sK = smem_u32(&s.K[0][0]);
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
    const int gq = lane >> 2, tq = lane & 3;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = warp * 16 + gq + (e >= 2 ? 8 : 0);
        const int col = n * 8 + 2 * tq + (e & 1);
        float val = 0.f;
        if (col < r) val = s.bt[r] * __expf(s.gc[r] - s.gc[col]) * acc[n][e];
        s.A[r][col] = val;
      }
    }
  }
  // scaled operands for W and U', and the decayed keys exp(g_C - g_r) k_r the state pass uses
  const float gC = s.gc[C - 1];  // rows past the end add g = 0, so this is the chunk's last g
  if (tid < C) {
    s.eb[tid] = s.bt[tid] * __expf(s.gc[tid]);
    s.ed[tid] = __expf(gC - s.gc[tid]);
  }
  __syncthreads();
  for (int i = tid; i < C * (D / 2); i += 128) {
    const int r = i / (D / 2), c2 = (i % (D / 2)) * 2;
    const float eb = s.eb[r];
    const float ed = s.ed[r];
    const float2 kf = __half22float2(*reinterpret_cast<const __half2*>(&s.K[r][c2]));
    const float2 vf = __half22float2(*reinterpret_cast<const __half2*>(&s.V[r][c2]));
    *reinterpret_cast<__half2*>(&s.KB[r][c2]) = __floats2half2_rn(eb * kf.x, eb * kf.y);
    *reinterpret_cast<__half2*>(&s.VB[r][c2]) = __floats2half2_rn(s.bt[r] * vf.x, s.bt[r] * vf.y);
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
  const int gq = lane >> 2, tq = lane & 3;
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    const uint32_t sB = smem_u32(which == 0 ? &s.KB[0][0] : &s.VB[0][0]);
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
// Phase 2: the state pass.  One CTA per (request, value head, slice of 16 value rows); the
// 16 x 128 fp32 state slice lives in mma accumulators (warp w: key columns 32w..32w+31).  Per
// chunk: U = U' - W S0^T for the slice, then S <- exp(g_C) S + U^T Kd with the decayed keys
// Kd = diag(exp(g_C - g)) K written by phase 1.  Everything a chunk needs (W, Kd, U', g) is
// prefetched with cp.async while the previous chunk is processed.
// ------------------------------------------------------------------------------------------
constexpr int SL = 16;  // value rows per CTA
struct PassBuf {
  __half W[C][LDH];
  __half K[C][LDH];      // decayed keys
  float U[C][SL + 4];
  float gc[C];
};
struct PassSmem {
  PassBuf buf[2];
  __half S[SL][LDH];       // fp16 copy of the entering state slice (value row, key col)
  __half Vn[C][SL + 8];    // U for the slice (token, value row)
};

__device__ __forceinline__ void pass_prefetch(PassBuf& pb, const __half* __restrict__ Wg,
                                              const __half* __restrict__ Kt,
                                              const float* __restrict__ Ug,
                                              const float* __restrict__ gcum, int64_t t0,
                                              int nvalid, int h, int sl, int tid) {
  for (int i = tid; i < C * (D / 8); i += 128) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    const bool ok = r < nvalid;
    const int64_t rr = ok ? (t0 + r) : t0;
    cp_async16(smem_u32(&pb.W[r][c8]), Wg + (rr * HV + h) * D + c8, ok);
    cp_async16(smem_u32(&pb.K[r][c8]), Kt + (rr * HV + h) * D + c8, ok);
  }
  for (int i = tid; i < C * (SL / 4); i += 128) {
    const int r = i / (SL / 4), c4 = (i % (SL / 4)) * 4;
    const bool ok = r < nvalid;
    const int64_t rr = ok ? (t0 + r) : t0;
    cp_async16(smem_u32(&pb.U[r][c4]), Ug + (rr * HV + h) * D + sl * SL + c4, ok);
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

__global__ void __launch_bounds__(128) gdn_state_pass_kernel(
    const __half* __restrict__ Kt, const __half* __restrict__ Wg, const float* __restrict__ Ug,
    const float* __restrict__ gcum, const float* __restrict__ s0, __half* __restrict__ Vnew,
    __half* __restrict__ S0out, float* __restrict__ s_out, int L, int nch) {
  extern __shared__ __align__(16) uint8_t smraw[];
  PassSmem& s = *reinterpret_cast<PassSmem*>(smraw);
  const int sl = blockIdx.x % (D / SL);
  const int h = (blockIdx.x / (D / SL)) % HV;
  const int b = blockIdx.x / ((D / SL) * HV);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;
  const int ncol = warp * 32;            // key columns of this warp's state tiles

  float S[4][4];
#pragma unroll
  for (int n = 0; n < 4; ++n) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v0 = 0.f;
      if (s0) {
        const int r = sl * SL + gq + (e >= 2 ? 8 : 0);
        const int col = ncol + n * 8 + 2 * tq + (e & 1);
        v0 = s0[(((int64_t)b * HV + h) * D + r) * D + col];
      }
      S[n][e] = v0;
    }
  }
  const int64_t tb = (int64_t)b * L;
  pass_prefetch(s.buf[0], Wg, Kt, Ug, gcum, tb, min(C, L), h, sl, tid);

  for (int c = 0; c < nch; ++c) {
    const int64_t t0 = tb + (int64_t)c * C;
    const int nvalid = min(C, L - c * C);
    PassBuf& pb = s.buf[c & 1];
    // entering state: fp16 copy to shared (for W S0^T) and to global (for the output phase)
#pragma unroll
    for (int n = 0; n < 4; ++n) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = gq + hf * 8;
        const int col = ncol + n * 8 + 2 * tq;
        const uint32_t pk = h2u(S[n][2 * hf], S[n][2 * hf + 1]);
        *reinterpret_cast<uint32_t*>(&s.S[r][col]) = pk;
        *reinterpret_cast<uint32_t*>(
            S0out + ((((int64_t)b * nch + c) * HV + h) * D + sl * SL + r) * D + col) = pk;
      }
    }
    if (c + 1 < nch)
      pass_prefetch(s.buf[(c + 1) & 1], Wg, Kt, Ug, gcum, t0 + C, min(C, L - (c + 1) * C), h, sl,
                    tid);
    else
      cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const float eC = __expf(pb.gc[C - 1]);
    // U = U' - W S0^T  (tokens 16w.., 16 value rows)
    {
      float acc[2][4];
#pragma unroll
      for (int n = 0; n < 2; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.f;
      const uint32_t sW = smem_u32(&pb.W[0][0]);
      const uint32_t sS = smem_u32(&s.S[0][0]);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        uint32_t a[4], bq[4];
        ldsm_x4(a, a_addr(sW, LDH, warp * 16, ks * 16, lane));
        ldsm_x4(bq, bn_addr(sS, LDH, 0, ks * 16, lane));
        mma16816(acc[0], a, bq[0], bq[1]);
        mma16816(acc[1], a, bq[2], bq[3]);
      }
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const int r = warp * 16 + gq + hf * 8;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
          const int col = n * 8 + 2 * tq;
          const float u0 = pb.U[r][col] - acc[n][2 * hf];
          const float u1 = pb.U[r][col + 1] - acc[n][2 * hf + 1];
          const uint32_t pk = (r < nvalid) ? h2u(u0, u1) : 0u;
          *reinterpret_cast<uint32_t*>(&s.Vn[r][col]) = pk;
          if (r < nvalid)
            *reinterpret_cast<uint32_t*>(Vnew + ((t0 + r) * HV + h) * D + sl * SL + col) = pk;
        }
      }
    }
    __syncthreads();
    // S <- exp(g_C) S + U^T Kd
    {
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        S[n][0] *= eC; S[n][1] *= eC; S[n][2] *= eC; S[n][3] *= eC;
      }
      const uint32_t sV = smem_u32(&s.Vn[0][0]);
      const uint32_t sK = smem_u32(&pb.K[0][0]);
#pragma unroll
      for (int ks = 0; ks < C / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4_t(a, at_addr(sV, SL + 8, 0, ks * 16, lane));
#pragma unroll
        for (int n = 0; n < 4; n += 2) {
          uint32_t bq[4];
          ldsm_x4_t(bq, bk_addr(sK, LDH, ncol + n * 8, ks * 16, lane));
          mma16816(S[n], a, bq[0], bq[1]);
          mma16816(S[n + 1], a, bq[2], bq[3]);
        }
      }
    }
    __syncthreads();  // buffers of this chunk are free for the prefetch two chunks ahead
  }
  cp_async_wait<0>();
  if (s_out) {
#pragma unroll
    for (int n = 0; n < 4; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = sl * SL + gq + (e >= 2 ? 8 : 0);
        const int col = ncol + n * 8 + 2 * tq + (e & 1);
        s_out[(((int64_t)b * HV + h) * D + r) * D + col] = S[n][e];
      }
    }
  }
}

// ------------------------------------------------------------------------------------------
// Phase 3: outputs of a (chunk, value head): O = (diag(e^g) Q S0^T + (tril(QK^T) o Gamma) U)
// / sqrt(128); then either a plain fp16 store or the z-gated RMSNorm
//   y = RMSNorm_128(O) * w_o * SiLU(z)  stored at out[token, h*128 + dv].
// ------------------------------------------------------------------------------------------
struct OutSmem {
  __half Q[C][LDH];
  __half K[C][LDH];
  __half U[C][LDH];
  __half S[D][LDH];  // entering state (value row, key col)
  float gc[C];
};

__global__ void __launch_bounds__(128) gdn_chunk_out_kernel(
    const __half* __restrict__ qq, const __half* __restrict__ kk, const __half* __restrict__ Vnew,
    const __half* __restrict__ S0g, const float* __restrict__ gcum, const __half* __restrict__ z,
    int64_t ldz, const __half* __restrict__ o_norm, __half* __restrict__ out, int64_t ldo, int L,
    int nch) {
  extern __shared__ __align__(16) uint8_t smraw[];
  OutSmem& s = *reinterpret_cast<OutSmem*>(smraw);
  const int cg = blockIdx.x, h = blockIdx.y;
  const int b = cg / nch, c = cg % nch;
  const int64_t t0 = (int64_t)b * L + (int64_t)c * C;
  const int nvalid = min(C, L - c * C);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  for (int i = tid; i < C * (D / 8); i += 128) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    const bool ok = r < nvalid;
    const int64_t rr = ok ? t0 + r : t0;
    cp_async16(smem_u32(&s.Q[r][c8]), qq + rr * (HK * D) + (h >> 1) * D + c8, ok);
    cp_async16(smem_u32(&s.K[r][c8]), kk + rr * (HK * D) + (h >> 1) * D + c8, ok);
    cp_async16(smem_u32(&s.U[r][c8]), Vnew + (rr * HV + h) * D + c8, ok);
  }
  const __half* Sg = S0g + (((int64_t)cg) * HV + h) * D * D;
  for (int i = tid; i < D * (D / 8); i += 128) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    cp_async16(smem_u32(&s.S[r][c8]), Sg + r * D + c8, true);
  }
  cp_async_commit();
  if (tid < C) s.gc[tid] = gcum[(t0 + min(tid, nvalid - 1)) * HV + h];
  cp_async_wait<0>();
  __syncthreads();

  const uint32_t sQ = smem_u32(&s.Q[0][0]), sK = smem_u32(&s.K[0][0]);
  const uint32_t sU = smem_u32(&s.U[0][0]), sS = smem_u32(&s.S[0][0]);
  // P = Q K^T for rows 16w..16w+15, masked and decayed
  uint32_t pa[4][4];  // P as A fragments, 4 k-steps of 16 keys
  {
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
#pragma unroll
    for (int n = 0; n < 8; ++n) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int r = warp * 16 + gq + (e >= 2 ? 8 : 0);
        const int col = n * 8 + 2 * tq + (e & 1);
        acc[n][e] = (col <= r) ? acc[n][e] * __expf(s.gc[r] - s.gc[col]) : 0.f;
      }
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      pa[j][0] = h2u(acc[2 * j][0], acc[2 * j][1]);
      pa[j][1] = h2u(acc[2 * j][2], acc[2 * j][3]);
      pa[j][2] = h2u(acc[2 * j + 1][0], acc[2 * j + 1][1]);
      pa[j][3] = h2u(acc[2 * j + 1][2], acc[2 * j + 1][3]);
    }
  }
  // scale this warp's own Q rows by e^{g_r} (only this warp reads them)
  __syncwarp();
  for (int i = lane; i < 16 * (D / 2); i += 32) {
    const int r = warp * 16 + i / (D / 2), c2 = (i % (D / 2)) * 2;
    const float f = __expf(s.gc[r]);
    const float2 qf = __half22float2(*reinterpret_cast<__half2*>(&s.Q[r][c2]));
    *reinterpret_cast<__half2*>(&s.Q[r][c2]) = __floats2half2_rn(qf.x * f, qf.y * f);
  }
  __syncwarp();
  float o[16][4];
#pragma unroll
  for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  // O = P U
#pragma unroll
  for (int ks = 0; ks < C / 16; ++ks) {
#pragma unroll
    for (int n = 0; n < 16; n += 2) {
      uint32_t bq[4];
      ldsm_x4_t(bq, bk_addr(sU, LDH, n * 8, ks * 16, lane));
      mma16816(o[n], pa[ks], bq[0], bq[1]);
      mma16816(o[n + 1], pa[ks], bq[2], bq[3]);
    }
  }
  // O += (e^g Q) S0^T
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    uint32_t a[4];
    ldsm_x4(a, a_addr(sQ, LDH, warp * 16, ks * 16, lane));
#pragma unroll
    for (int n = 0; n < 16; n += 2) {
      uint32_t bq[4];
      ldsm_x4(bq, bn_addr(sS, LDH, n * 8, ks * 16, lane));
      mma16816(o[n], a, bq[0], bq[1]);
      mma16816(o[n + 1], a, bq[2], bq[3]);
    }
  }
  const float scale = 0.08838834764831845f;  // 1 / sqrt(128)
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int r = warp * 16 + gq + hf * 8;
    float inv = 1.f;
    if (z) {
      float ss = 0.f;
#pragma unroll
      for (int n = 0; n < 16; ++n) {
        const float a0 = o[n][2 * hf] * scale, a1 = o[n][2 * hf + 1] * scale;
        ss += a0 * a0 + a1 * a1;
      }
      ss += __shfl_xor_sync(0xffffffffu, ss, 1);
      ss += __shfl_xor_sync(0xffffffffu, ss, 2);
      inv = rsqrtf(ss * (1.f / D) + 1e-6f);
    }
    if (r >= nvalid) continue;
    const int64_t tok = t0 + r;
#pragma unroll
    for (int n = 0; n < 16; ++n) {
      const int col = n * 8 + 2 * tq;
      float a0 = o[n][2 * hf] * scale, a1 = o[n][2 * hf + 1] * scale;
      if (z) {
        const float2 zf = __half22float2(*reinterpret_cast<const __half2*>(z + tok * ldz + h * D + col));
        const float2 wf = __half22float2(*reinterpret_cast<const __half2*>(o_norm + col));
        a0 = a0 * inv * wf.x * silu_f(zf.x);
        a1 = a1 * inv * wf.y * silu_f(zf.y);
      }
      *reinterpret_cast<uint32_t*>(out + tok * ldo + h * D + col) = h2u(a0, a1);
    }
  }
}

}  // namespace gdn

static inline size_t al256g(size_t x) { return (x + 255) & ~size_t(255); }

size_t gdn_scan_workspace_bytes(int64_t B, int64_t L) {
  const int64_t M = B * L;
  const int64_t nch = (L + gdn::C - 1) / gdn::C;
  size_t n = 0;
  n += al256g(M * gdn::HV * 4);                         // g (from alpha)
  n += al256g(M * gdn::HV * 4);                         // gcum
  n += al256g(M * gdn::HV * gdn::D * 2);                // W
  n += al256g(M * gdn::HV * gdn::D * 4);                // U'
  n += al256g(M * gdn::HV * gdn::D * 2);                // U
  n += al256g(M * gdn::HV * gdn::D * 2);                // decayed keys
  n += al256g(B * nch * gdn::HV * gdn::D * gdn::D * 2); // entering states
  return n;
}

struct GdnWs {
  float* g;
  float* gcum;
  __half* W;
  float* U1;
  __half* U;
  __half* Kt;
  __half* S0;
};
static GdnWs carve(void* ws, int64_t B, int64_t L) {
  const int64_t M = B * L;
  uint8_t* p = static_cast<uint8_t*>(ws);
  GdnWs w;
  w.g = reinterpret_cast<float*>(p); p += al256g(M * gdn::HV * 4);
  w.gcum = reinterpret_cast<float*>(p); p += al256g(M * gdn::HV * 4);
  w.W = reinterpret_cast<__half*>(p); p += al256g(M * gdn::HV * gdn::D * 2);
  w.U1 = reinterpret_cast<float*>(p); p += al256g(M * gdn::HV * gdn::D * 4);
  w.U = reinterpret_cast<__half*>(p); p += al256g(M * gdn::HV * gdn::D * 2);
  w.Kt = reinterpret_cast<__half*>(p); p += al256g(M * gdn::HV * gdn::D * 2);
  w.S0 = reinterpret_cast<__half*>(p);
  return w;
}

static bool g_gdn_attr = false;
static clef_status gdn_set_attrs() {
  if (g_gdn_attr) return CLEF_OK;
  CLEF_CUDA_CHECK(cudaFuncSetAttribute(gdn::gdn_chunk_wy_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, sizeof(gdn::WySmem)));
  CLEF_CUDA_CHECK(cudaFuncSetAttribute(gdn::gdn_state_pass_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, sizeof(gdn::PassSmem)));
  CLEF_CUDA_CHECK(cudaFuncSetAttribute(gdn::gdn_chunk_out_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, sizeof(gdn::OutSmem)));
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
    TraceScope ts(stream, "gdn_chunk_wy", nchunks * HVd * 6.0 * C * C * D,
                  (double)M * HVd * D * (2 + 2 + 2 + 4));
    gdn::gdn_chunk_wy_kernel<<<g1, 128, sizeof(gdn::WySmem), stream>>>(k, v, g, beta, w.gcum, w.W,
                                                                        w.U1, w.Kt, (int)L, nch);
    CLEF_LAUNCH_CHECK();
  }
  {
    TraceScope ts(stream, "gdn_state_pass", nchunks * HVd * 4.0 * C * D * D,
                  (double)M * HVd * D * (2 + 4 + 2) + (double)M * 16 * D * 2 + nchunks * HVd * D * D * 2);
    gdn::gdn_state_pass_kernel<<<(unsigned)(B * gdn::HV * (gdn::D / gdn::SL)), 128,
                                 sizeof(gdn::PassSmem), stream>>>(w.Kt, w.W, w.U1, w.gcum, s0, w.U,
                                                                  w.S0, s_out, (int)L, nch);
    CLEF_LAUNCH_CHECK();
  }
  {
    TraceScope ts(stream, "gdn_chunk_out", nchunks * HVd * (4.0 * C * C * D + 2.0 * C * D * D),
                  (double)M * HVd * D * (2 + 2 + 2) + (double)M * 32 * D * 2 * 2 + nchunks * HVd * D * D * 2);
    gdn::gdn_chunk_out_kernel<<<g1, 128, sizeof(gdn::OutSmem), stream>>>(
        q, k, w.U, w.S0, w.gcum, z, ldz, o_norm, out, ldo, (int)L, nch);
    CLEF_LAUNCH_CHECK();
  }
  return CLEF_OK;
}

}  // namespace clef
