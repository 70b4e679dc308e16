// The joint schema head on one request's hidden states (clef_joint_head; clef.h states what the
// pages fix and the reading taken for its layers): span means of the hidden rows -> 1,024-wide
// slots, 4 decoder layers in which the slots attend to the request's tokens, 2 routing layers in
// which they attend to each other, bilinear option logits, a softmax per question.
//
// The head is small beside the prefill (a few hundred GFLOP at 16,384 tokens), so it is a
// sequence of plain kernels: one dense fp16 GEMM on tensor cores (mma.sync m16n8k16, fp32
// accumulation, cp.async double buffering; batched over the attention heads) and CUDA-core
// kernels for the span means, norms, softmax and the readout.  Activations between kernels are
// fp16, the slots' residual stream fp32.
#include <algorithm>

#include "common.cuh"
#include "mma.cuh"

namespace clef {
namespace head {

constexpr int D = 1024, NH = 16, DH = 64, FF = 4096, HID = 4096;

// ---------------------------------------------------------------------------------- dense GEMM
// C[z][M, N] (op)= alpha * A[z][M, K] . B[z]^T, with B stored [N][K] (k contiguous: weights,
// keys) or, with B_KN, [K][N] (n contiguous: values).  Tiles of 64 x 64, k in steps of 32; warp w
// owns rows 16w .. 16w + 15.  Rows of A past M and of B past N read as zero; K % 32 == 0.
enum GemmEpi : int { G_F32 = 0, G_F16 = 1, G_ADD_F32 = 2 };
constexpr int GBM = 64, GBN = 64, GBK = 32, GLD = GBK + 8, GLDN = GBN + 8;

struct GemmArgs {
  const __half* A;
  int64_t lda, sA;
  const __half* B;
  int64_t ldb, sB;
  void* C;
  int64_t ldc, sC;
  int M, N, K;
  float alpha;
};

template <bool B_KN>
struct GemmSmem {
  __half A[2][GBM][GLD];
  __half B[2][B_KN ? GBK : GBN][B_KN ? GLDN : GLD];
};

template <bool B_KN, int EPI>
__global__ void __launch_bounds__(128) gemm_kernel(GemmArgs g) {
  __shared__ __align__(16) GemmSmem<B_KN> s;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m0 = blockIdx.y * GBM, n0 = blockIdx.x * GBN;
  const __half* A = g.A + blockIdx.z * g.sA;
  const __half* B = g.B + blockIdx.z * g.sB;
  auto load = [&](int buf, int k0) {
    for (int i = tid; i < GBM * (GBK / 8); i += 128) {
      const int r = i / (GBK / 8), c8 = (i % (GBK / 8)) * 8;
      const bool ok = m0 + r < g.M;
      cp_async16(smem_u32(&s.A[buf][r][c8]), A + (ok ? (int64_t)(m0 + r) * g.lda : 0) + k0 + c8, ok);
    }
    if (B_KN) {
      for (int i = tid; i < GBK * (GBN / 8); i += 128) {
        const int r = i / (GBN / 8), c8 = (i % (GBN / 8)) * 8;
        const bool ok = n0 + c8 < g.N;
        cp_async16(smem_u32(&s.B[buf][r][c8]), B + (int64_t)(k0 + r) * g.ldb + (ok ? n0 + c8 : 0), ok);
      }
    } else {
      for (int i = tid; i < GBN * (GBK / 8); i += 128) {
        const int r = i / (GBK / 8), c8 = (i % (GBK / 8)) * 8;
        const bool ok = n0 + r < g.N;
        cp_async16(smem_u32(&s.B[buf][r][c8]), B + (ok ? (int64_t)(n0 + r) * g.ldb : 0) + k0 + c8, ok);
      }
    }
    cp_async_commit();
  };
  float acc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
  const int nk = g.K / GBK;
  load(0, 0);
  for (int kt = 0; kt < nk; ++kt) {
    const int buf = kt & 1;
    if (kt + 1 < nk) load(buf ^ 1, (kt + 1) * GBK); else cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const uint32_t sa = smem_u32(&s.A[buf][0][0]), sbb = smem_u32(&s.B[buf][0][0]);
#pragma unroll
    for (int ks = 0; ks < GBK / 16; ++ks) {
      uint32_t a[4];
      ldsm_x4(a, a_addr(sa, GLD, 16 * warp, 16 * ks, lane));
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        uint32_t b[4];
        if (B_KN)
          ldsm_x4_t(b, bk_addr(sbb, GLDN, 16 * j, 16 * ks, lane));
        else
          ldsm_x4(b, bn_addr(sbb, GLD, 16 * j, 16 * ks, lane));
        mma16816(acc[2 * j], a, b[0], b[1]);
        mma16816(acc[2 * j + 1], a, b[2], b[3]);
      }
    }
    __syncthreads();
  }
  const int gr = lane >> 2, gc = 2 * (lane & 3);
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = m0 + 16 * warp + gr + 8 * h;
      const int col = n0 + 8 * j + gc;
      if (row >= g.M) continue;
      const float v0 = g.alpha * acc[j][2 * h], v1 = g.alpha * acc[j][2 * h + 1];
      const int64_t off = blockIdx.z * g.sC + (int64_t)row * g.ldc + col;
      if (EPI == G_F16) {
        __half* c = static_cast<__half*>(g.C) + off;
        if (col < g.N) c[0] = __float2half_rn(v0);
        if (col + 1 < g.N) c[1] = __float2half_rn(v1);
      } else if (EPI == G_F32) {
        float* c = static_cast<float*>(g.C) + off;
        if (col < g.N) c[0] = v0;
        if (col + 1 < g.N) c[1] = v1;
      } else {
        float* c = static_cast<float*>(g.C) + off;
        if (col < g.N) c[0] += v0;
        if (col + 1 < g.N) c[1] += v1;
      }
    }
}

// ------------------------------------------------------------------------------ small kernels
// u[r][:] = sum_t P_r[t] hidden[t][:], P_r the r-th row of [q_avg; o_avg; g_avg] (fp32), fp16 out.
// Every thread reads the same P_r[t], so the zero weights of positions outside a span are
// skipped by the whole block.  Block: 256 threads x 4 columns.
__global__ void pool_kernel(const float* __restrict__ q_avg, const float* __restrict__ o_avg,
                            const float* __restrict__ g_avg, const __half* __restrict__ hidden,
                            int64_t T, int Q, int O, __half* __restrict__ u) {
  const int r = blockIdx.x;
  const float* P = r < Q ? q_avg + (int64_t)r * T : r < Q + O ? o_avg + (int64_t)(r - Q) * T : g_avg;
  const int c = blockIdx.y * 1024 + threadIdx.x * 4;
  float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
  for (int64_t t = 0; t < T; ++t) {
    const float p = P[t];
    if (p == 0.f) continue;
    const uint2 hv = *reinterpret_cast<const uint2*>(hidden + t * HID + c);
    const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&hv.x));
    const float2 y = __half22float2(*reinterpret_cast<const __half2*>(&hv.y));
    a0 += p * x.x;
    a1 += p * x.y;
    a2 += p * y.x;
    a3 += p * y.y;
  }
  uint2 out;
  out.x = h2u(a0, a1);
  out.y = h2u(a2, a3);
  *reinterpret_cast<uint2*>(u + (int64_t)r * HID + c) = out;
}

__global__ void to_half_kernel(const float* __restrict__ x, __half* __restrict__ y, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x)
    y[i] = __float2half_rn(x[i]);
}

// s[r] += the row's embeddings: question-type (questions), lexical projection + option
// embedding (options), global embedding (the last row).
__global__ void slot_init_kernel(float* __restrict__ s, const float* __restrict__ lexp,
                                 const int32_t* __restrict__ type_ids, const __half* __restrict__ e_q,
                                 const __half* __restrict__ e_o, const __half* __restrict__ e_g,
                                 int Q, int O) {
  const int r = blockIdx.x;
  for (int c = threadIdx.x; c < D; c += blockDim.x) {
    float add;
    if (r < Q)
      add = __half2float(e_q[min(max(type_ids[r], 0), 2) * D + c]);   // ids outside 0..2 clamp
    else if (r < Q + O)
      add = lexp[(int64_t)(r - Q) * D + c] + __half2float(e_o[c]);
    else
      add = __half2float(e_g[c]);
    s[(int64_t)r * D + c] += add;
  }
}

// y = x / sqrt(mean(x^2) + 1e-6) * w over rows of 1,024 (fp32 in, fp16 out); one warp per row.
__global__ void rmsnorm1024_kernel(const float* __restrict__ x, const __half* __restrict__ w,
                                   __half* __restrict__ y, int rows) {
  const int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const float* xr = x + (int64_t)row * D;
  float v[32];
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float4 f = *reinterpret_cast<const float4*>(xr + 4 * (lane + 32 * i));
    v[4 * i] = f.x; v[4 * i + 1] = f.y; v[4 * i + 2] = f.z; v[4 * i + 3] = f.w;
    ss += f.x * f.x + f.y * f.y + f.z * f.z + f.w * f.w;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float r = rsqrtf(ss * (1.f / D) + 1e-6f);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int c = 4 * (lane + 32 * i);
    const float2 w01 = __half22float2(*reinterpret_cast<const __half2*>(w + c));
    const float2 w23 = __half22float2(*reinterpret_cast<const __half2*>(w + c + 2));
    uint2 out;
    out.x = h2u(v[4 * i] * r * w01.x, v[4 * i + 1] * r * w01.y);
    out.y = h2u(v[4 * i + 2] * r * w23.x, v[4 * i + 3] * r * w23.y);
    *reinterpret_cast<uint2*>(y + (int64_t)row * D + c) = out;
  }
}

// One attention row (head h, query s): p[t] = softmax over valid keys t < Tk of scale * score,
// written as fp16 with zeros for invalid keys and for Tk <= t < ld.  No valid key: all zero.
__global__ void softmax_kernel(const float* __restrict__ scores, const uint8_t* __restrict__ valid,
                               int Tk, int64_t ld, float scale, __half* __restrict__ p) {
  __shared__ float red[32];
  const int64_t row = blockIdx.x;
  const float* sr = scores + row * ld;
  __half* pr = p + row * ld;
  const int tid = threadIdx.x, nw = blockDim.x >> 5;
  float m = -INFINITY;
  for (int t = tid; t < Tk; t += blockDim.x)
    if (valid[t]) m = fmaxf(m, sr[t] * scale);
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((tid & 31) == 0) red[tid >> 5] = m;
  __syncthreads();
  m = -INFINITY;
  for (int i = 0; i < nw; ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  float sum = 0.f;
  for (int t = tid; t < Tk; t += blockDim.x)
    if (valid[t]) sum += __expf(sr[t] * scale - m);
  for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if ((tid & 31) == 0) red[tid >> 5] = sum;
  __syncthreads();
  sum = 0.f;
  for (int i = 0; i < nw; ++i) sum += red[i];
  const float inv = m == -INFINITY ? 0.f : 1.f / sum;
  for (int64_t t = tid; t < ld; t += blockDim.x)
    pr[t] = __float2half_rn(t < Tk && valid[t] ? __expf(sr[t] * scale - m) * inv : 0.f);
}

// h = SiLU(g) * u (fp32 in, fp16 out)
__global__ void swiglu_kernel(const float* __restrict__ g, const float* __restrict__ u,
                              __half* __restrict__ h, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float x = g[i];
    h[i] = __float2half_rn(x / (1.f + __expf(-x)) * u[i]);
  }
}

// slot validity: questions, options, then the global row (always valid)
__global__ void slot_valid_kernel(const uint8_t* __restrict__ qv, const uint8_t* __restrict__ ov,
                                  int Q, int O, uint8_t* __restrict__ sv) {
  for (int i = threadIdx.x; i < Q + O + 1; i += blockDim.x)
    sv[i] = i < Q ? (qv[i] != 0) : i < Q + O ? (ov[i - Q] != 0) : 1;
}

// c[o][:] = sum_q member[q][o] f[q][:]  (the row of the question option o belongs to), fp16
__global__ void option_question_kernel(const __half* __restrict__ f, const uint8_t* __restrict__ member,
                                       int Q, int O, __half* __restrict__ c) {
  const int o = blockIdx.x;
  for (int col = threadIdx.x; col < D; col += blockDim.x) {
    float acc = 0.f;
    for (int q = 0; q < Q; ++q)
      if (member[q * O + o]) acc += __half2float(f[(int64_t)q * D + col]);
    c[(int64_t)o * D + col] = __float2half_rn(acc);
  }
}

// logit_o = a_o . b_o / 32 for valid options (0 otherwise); one warp per option
__global__ void logits_kernel(const float* __restrict__ a, const float* __restrict__ b,
                              const uint8_t* __restrict__ ov, int O, float* __restrict__ logits) {
  const int o = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (o >= O) return;
  float acc = 0.f;
  for (int c = lane; c < D; c += 32) acc += a[(int64_t)o * D + c] * b[(int64_t)o * D + c];
  for (int s = 16; s; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
  if (lane == 0) logits[o] = ov[o] ? acc * (1.f / 32.f) : 0.f;
}

// Per question (one warp each): a float32 softmax over its valid options; every other option 0.
__global__ void probs_kernel(const float* __restrict__ logits, const uint8_t* __restrict__ member,
                             const uint8_t* __restrict__ qv, const uint8_t* __restrict__ ov, int Q,
                             int O, float* __restrict__ probs) {
  const int lane = threadIdx.x & 31, q = threadIdx.x >> 5;
  for (int o = threadIdx.x; o < O; o += blockDim.x) {
    bool any = false;
    for (int qq = 0; qq < Q; ++qq) any |= member[qq * O + o] && qv[qq] && ov[o];
    if (!any) probs[o] = 0.f;
  }
  if (q >= Q || !qv[q]) return;
  float m = -INFINITY;
  for (int o = lane; o < O; o += 32)
    if (member[q * O + o] && ov[o]) m = fmaxf(m, logits[o]);
  for (int s = 16; s; s >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, s));
  if (m == -INFINITY) return;
  float sum = 0.f;
  for (int o = lane; o < O; o += 32)
    if (member[q * O + o] && ov[o]) sum += expf(logits[o] - m);
  for (int s = 16; s; s >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, s);
  for (int o = lane; o < O; o += 32)
    if (member[q * O + o] && ov[o]) probs[o] = expf(logits[o] - m) / sum;
}

// ---------------------------------------------------------------------------- workspace
struct Ws {
  __half *u16, *lex16, *mem16, *a16, *q16, *k16, *v16, *o16, *h16, *c16, *P16;
  float *s, *lexp, *g, *uu, *scores, *oa, *ob;
  uint8_t* sv;
};

inline int64_t pad64(int64_t x) { return (x + 63) / 64 * 64; }

static size_t carve(int64_t T, int64_t Q, int64_t O, void* base, Ws* w) {
  const int64_t S = Q + O + 1;
  const int64_t Tp = pad64(T), Sp = pad64(S), Kp = std::max(Tp, Sp);
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    void* r = p ? p + off : nullptr;
    off += (bytes + 255) & ~size_t(255);
    return r;
  };
  Ws t;
  t.u16 = static_cast<__half*>(take(S * HID * 2));
  t.lex16 = static_cast<__half*>(take(O * HID * 2));
  t.mem16 = static_cast<__half*>(take(Tp * D * 2));
  t.a16 = static_cast<__half*>(take(Sp * D * 2));
  t.q16 = static_cast<__half*>(take(S * D * 2));
  t.k16 = static_cast<__half*>(take(Kp * D * 2));
  t.v16 = static_cast<__half*>(take(Kp * D * 2));
  t.o16 = static_cast<__half*>(take(S * D * 2));
  t.h16 = static_cast<__half*>(take(S * FF * 2));
  t.c16 = static_cast<__half*>(take(O * D * 2));
  t.P16 = static_cast<__half*>(take(NH * S * Kp * 2));
  t.s = static_cast<float*>(take(S * D * 4));
  t.lexp = static_cast<float*>(take(O * D * 4));
  t.g = static_cast<float*>(take(S * FF * 4));
  t.uu = static_cast<float*>(take(S * FF * 4));
  t.scores = static_cast<float*>(take(NH * S * Kp * 4));
  t.oa = static_cast<float*>(take(O * D * 4));
  t.ob = static_cast<float*>(take(O * D * 4));
  t.sv = static_cast<uint8_t*>(take(Sp));
  if (w) *w = t;
  return off;
}

template <bool B_KN, int EPI>
static clef_status gemm(const __half* A, int64_t lda, int64_t sA, const __half* B, int64_t ldb,
                        int64_t sB, void* C, int64_t ldc, int64_t sC, int M, int N, int K, int batch,
                        float alpha, cudaStream_t st) {
  if (M == 0 || N == 0) return CLEF_OK;
  GemmArgs g{A, lda, sA, B, ldb, sB, C, ldc, sC, M, N, K, alpha};
  dim3 grid((N + GBN - 1) / GBN, (M + GBM - 1) / GBM, batch);
  gemm_kernel<B_KN, EPI><<<grid, 128, 0, st>>>(g);
  CLEF_LAUNCH_CHECK();
  return CLEF_OK;
}

#define HEAD_TRY(expr)              \
  do {                              \
    clef_status _s = (expr);        \
    if (_s != CLEF_OK) return _s;   \
  } while (0)

// One layer on the slots: attention of the S query rows to `Tk` key rows (memory rows mem16 with
// key_valid, or the slots themselves with the slot validity), then the SwiGLU MLP.
static clef_status head_layer(const clef_head_layer& L, const Ws& w, int S, const __half* mem16,
                              int Tk, const uint8_t* valid, cudaStream_t st) {
  const int64_t Kp = pad64(Tk);
  rmsnorm1024_kernel<<<(S + 7) / 8, 256, 0, st>>>(w.s, reinterpret_cast<const __half*>(L.norm1), w.a16, S);
  CLEF_LAUNCH_CHECK();
  const __half* src = mem16 ? mem16 : w.a16;
  HEAD_TRY((gemm<false, G_F16>(w.a16, D, 0, reinterpret_cast<const __half*>(L.wq), D, 0, w.q16, D, 0,
                               S, D, D, 1, 1.f, st)));
  HEAD_TRY((gemm<false, G_F16>(src, D, 0, reinterpret_cast<const __half*>(L.wk), D, 0, w.k16, D, 0,
                               Tk, D, D, 1, 1.f, st)));
  HEAD_TRY((gemm<false, G_F16>(src, D, 0, reinterpret_cast<const __half*>(L.wv), D, 0, w.v16, D, 0,
                               Tk, D, D, 1, 1.f, st)));
  // value rows past Tk meet zero weights in P . V; keep them finite
  if (Kp > Tk)
    CLEF_CUDA_CHECK(cudaMemsetAsync(w.v16 + (int64_t)Tk * D, 0, (size_t)(Kp - Tk) * D * 2, st));
  // scores[h] = q_h . k_h^T  [S, Tk], one batch entry per head
  HEAD_TRY((gemm<false, G_F32>(w.q16, D, DH, w.k16, D, DH, w.scores, Kp, (int64_t)S * Kp, S, Tk, DH,
                               NH, 1.f, st)));
  softmax_kernel<<<NH * S, 256, 0, st>>>(w.scores, valid, Tk, Kp, 0.125f, w.P16);
  CLEF_LAUNCH_CHECK();
  // o_h = P_h . v_h  [S, 64] into columns 64h .. of o16
  HEAD_TRY((gemm<true, G_F16>(w.P16, Kp, (int64_t)S * Kp, w.v16, D, DH, w.o16, D, DH, S, DH, (int)Kp,
                              NH, 1.f, st)));
  HEAD_TRY((gemm<false, G_ADD_F32>(w.o16, D, 0, reinterpret_cast<const __half*>(L.wo), D, 0, w.s, D,
                                   0, S, D, D, 1, 1.f, st)));
  // MLP
  rmsnorm1024_kernel<<<(S + 7) / 8, 256, 0, st>>>(w.s, reinterpret_cast<const __half*>(L.norm2), w.a16, S);
  CLEF_LAUNCH_CHECK();
  HEAD_TRY((gemm<false, G_F32>(w.a16, D, 0, reinterpret_cast<const __half*>(L.wg), D, 0, w.g, FF, 0,
                               S, FF, D, 1, 1.f, st)));
  HEAD_TRY((gemm<false, G_F32>(w.a16, D, 0, reinterpret_cast<const __half*>(L.wu), D, 0, w.uu, FF, 0,
                               S, FF, D, 1, 1.f, st)));
  swiglu_kernel<<<std::min<int64_t>(((int64_t)S * FF + 255) / 256, 2048), 256, 0, st>>>(
      w.g, w.uu, w.h16, (int64_t)S * FF);
  CLEF_LAUNCH_CHECK();
  HEAD_TRY((gemm<false, G_ADD_F32>(w.h16, FF, 0, reinterpret_cast<const __half*>(L.wd), FF, 0, w.s, D,
                                   0, S, D, FF, 1, 1.f, st)));
  return CLEF_OK;
}

}  // namespace head
}  // namespace clef

using namespace clef;
using namespace clef::head;

static bool misaligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

extern "C" {

size_t clef_joint_head_workspace_size(int64_t T, int64_t Q, int64_t O) {
  if (T < 1 || Q < 1 || O < 1 || T > CLEF_MAX_LEN || Q > CLEF_HEAD_MAX_Q || O > CLEF_HEAD_MAX_O)
    return 0;
  return carve(T, Q, O, nullptr, nullptr);
}

clef_status clef_joint_head(const clef_head* hd, const uint16_t* hidden, const uint8_t* key_valid,
                            int64_t T, const float* q_avg, const float* o_avg, const float* g_avg,
                            const float* lexical, const uint8_t* member, const int32_t* type_ids,
                            const uint8_t* q_valid, const uint8_t* o_valid, int64_t Q, int64_t O,
                            float* logits, float* probs, void* workspace, size_t workspace_bytes,
                            clef_stream stream) {
  if (!hd || !hidden || !key_valid || !q_avg || !o_avg || !g_avg || !lexical || !member ||
      !type_ids || !q_valid || !o_valid || !logits || !probs || !workspace) {
    set_error("clef_joint_head: NULL pointer");
    return CLEF_E_INVALID;
  }
  if (T < 1 || Q < 1 || O < 1) {
    set_error("clef_joint_head: need T, Q, O >= 1");
    return CLEF_E_INVALID;
  }
  if (T > CLEF_MAX_LEN || Q > CLEF_HEAD_MAX_Q || O > CLEF_HEAD_MAX_O) {
    set_error("clef_joint_head: T = %lld, Q = %lld, O = %lld beyond %d, %d, %d", (long long)T,
              (long long)Q, (long long)O, CLEF_MAX_LEN, CLEF_HEAD_MAX_Q, CLEF_HEAD_MAX_O);
    return T > CLEF_MAX_LEN ? CLEF_E_TOO_LONG : CLEF_E_SHAPE;
  }
  const void* weights[] = {hd->w_mem, hd->w_in, hd->w_lex, hd->e_qtype, hd->e_opt, hd->e_glob,
                           hd->norm_f, hd->w_opt, hd->w_qst};
  for (const void* p : weights)
    if (!p || misaligned16(p)) {
      set_error("clef_joint_head: a head weight is NULL or not 16-byte aligned");
      return p ? CLEF_E_ALIGN : CLEF_E_INVALID;
    }
  for (int l = 0; l < 6; ++l) {
    const clef_head_layer& L = l < 4 ? hd->dec[l] : hd->route[l - 4];
    const void* lw[] = {L.norm1, L.wq, L.wk, L.wv, L.wo, L.norm2, L.wg, L.wu, L.wd};
    for (const void* p : lw)
      if (!p || misaligned16(p)) {
        set_error("clef_joint_head: a layer weight is NULL or not 16-byte aligned");
        return p ? CLEF_E_ALIGN : CLEF_E_INVALID;
      }
  }
  if (misaligned16(hidden) || misaligned16(lexical) || misaligned16(workspace)) {
    set_error("clef_joint_head: hidden, lexical and the workspace must be 16-byte aligned");
    return CLEF_E_ALIGN;
  }
  const size_t need = carve(T, Q, O, nullptr, nullptr);
  if (workspace_bytes < need) {
    set_error("clef_joint_head: workspace of %zu bytes, need %zu", workspace_bytes, need);
    return CLEF_E_WORKSPACE;
  }
  if (debug_should_fail()) return CLEF_E_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  Ws w;
  carve(T, Q, O, workspace, &w);
  const int S = (int)(Q + O + 1), Ti = (int)T, Qi = (int)Q, Oi = (int)O;
  const __half* hid = reinterpret_cast<const __half*>(hidden);
  TraceScope ts(st, "joint_head",
                2.0 * T * HID * D + 4 * 2.0 * 2 * T * D * D + 6 * 2.0 * S * (4.0 * D * D + 3.0 * D * FF),
                T * HID * 2.0);
  // slots: span means and the global row, projected; plus the embeddings and the lexical rows
  pool_kernel<<<dim3(S, HID / 1024), 256, 0, st>>>(q_avg, o_avg, g_avg, hid, T, Qi, Oi, w.u16);
  CLEF_LAUNCH_CHECK();
  to_half_kernel<<<(unsigned)std::min<int64_t>((O * HID + 255) / 256, 2048), 256, 0, st>>>(
      lexical, w.lex16, O * HID);
  CLEF_LAUNCH_CHECK();
  HEAD_TRY((gemm<false, G_F32>(w.u16, HID, 0, reinterpret_cast<const __half*>(hd->w_in), HID, 0, w.s,
                               D, 0, S, D, HID, 1, 1.f, st)));
  HEAD_TRY((gemm<false, G_F32>(w.lex16, HID, 0, reinterpret_cast<const __half*>(hd->w_lex), HID, 0,
                               w.lexp, D, 0, Oi, D, HID, 1, 1.f, st)));
  slot_init_kernel<<<S, 256, 0, st>>>(w.s, w.lexp, type_ids,
                                      reinterpret_cast<const __half*>(hd->e_qtype),
                                      reinterpret_cast<const __half*>(hd->e_opt),
                                      reinterpret_cast<const __half*>(hd->e_glob), Qi, Oi);
  CLEF_LAUNCH_CHECK();
  slot_valid_kernel<<<1, 256, 0, st>>>(q_valid, o_valid, Qi, Oi, w.sv);
  CLEF_LAUNCH_CHECK();
  // the memory: the request's tokens at the head's width
  HEAD_TRY((gemm<false, G_F16>(hid, HID, 0, reinterpret_cast<const __half*>(hd->w_mem), HID, 0,
                               w.mem16, D, 0, Ti, D, HID, 1, 1.f, st)));
  for (int l = 0; l < 4; ++l) HEAD_TRY(head_layer(hd->dec[l], w, S, w.mem16, Ti, key_valid, st));
  for (int l = 0; l < 2; ++l) HEAD_TRY(head_layer(hd->route[l], w, S, nullptr, S, w.sv, st));
  // readout
  rmsnorm1024_kernel<<<(S + 7) / 8, 256, 0, st>>>(w.s, reinterpret_cast<const __half*>(hd->norm_f), w.a16, S);
  CLEF_LAUNCH_CHECK();
  option_question_kernel<<<Oi, 256, 0, st>>>(w.a16, member, Qi, Oi, w.c16);
  CLEF_LAUNCH_CHECK();
  HEAD_TRY((gemm<false, G_F32>(w.a16 + (int64_t)Qi * D, D, 0, reinterpret_cast<const __half*>(hd->w_opt),
                               D, 0, w.oa, D, 0, Oi, D, D, 1, 1.f, st)));
  HEAD_TRY((gemm<false, G_F32>(w.c16, D, 0, reinterpret_cast<const __half*>(hd->w_qst), D, 0, w.ob, D,
                               0, Oi, D, D, 1, 1.f, st)));
  logits_kernel<<<(Oi + 7) / 8, 256, 0, st>>>(w.oa, w.ob, o_valid, Oi, logits);
  CLEF_LAUNCH_CHECK();
  probs_kernel<<<1, 32 * CLEF_HEAD_MAX_Q, 0, st>>>(logits, member, q_valid, o_valid, Qi, Oi, probs);
  CLEF_LAUNCH_CHECK();
  return CLEF_OK;
}

}  // extern "C"
