// Causal GQA attention of the gated full-attention layers.
//
// "Clef-Flash-ANE-LUT6" model card, "Model architecture": 16 query and 4 key-value heads of 256.
// "clef-flash-LiteRT" README, "Host contract" step 5: rotary with theta = 1e7 and, for text, the
// position (i, i, i) on all three planes, i.e. a 1-D rotary; "clef-flash-coreml" README: cos/sin
// tables [L, 64], i.e. 64 rotated dims per head.  "Provenance": grouped keys/values shared by the
// query heads of a group, causal additive mask.
//
//   rope_kernel   rotates dims 0..63 of every q and k head (rotate-half pairs (j, j+32), angle
//                 pos * 1e7^(-j/32), computed in fp64), in place or into a copy.
//   flash_kernel  one CTA = 32 positions x the 4 query heads of one kv head (128 rows), so each
//                 K/V tile is read once for the group; online softmax over 64-key tiles
//                 (tensor-core mma.sync, fp32 accumulation); epilogue o * sigmoid(gate).
#include "attn.cuh"
#include "common.cuh"
#include "mma.cuh"

namespace clef {
namespace attn {

constexpr int D = 256;
constexpr int HQ = 16, HKV = 4;
constexpr int BM = 128;            // rows per CTA = 32 positions x 4 heads
constexpr int POS = BM / 4;        // positions per CTA
constexpr int BN = 64;             // keys per tile
constexpr int LDS = D + 8;         // padded smem row (528 bytes)
constexpr int THREADS = 256;

__global__ void __launch_bounds__(128) rope_kernel(const __half* __restrict__ qin, int64_t ldqi,
                                                   __half* __restrict__ qout, int64_t ldqo,
                                                   const __half* __restrict__ kin, int64_t ldki,
                                                   __half* __restrict__ kout, int64_t ldko, int L) {
  __shared__ float cs[32], sn[32];
  const int64_t tok = blockIdx.x;
  const int pos = (int)(tok % L);
  const int tid = threadIdx.x;
  if (tid < 32) {
    // angle = pos * theta^(-j/32), reduced and evaluated in fp64 (ln 1e7 = 16.118...)
    const double inv_freq = exp(-(double)tid * (16.11809565095832 / 32.0));
    double s, c;
    sincos((double)pos * inv_freq, &s, &c);
    cs[tid] = (float)c;
    sn[tid] = (float)s;
  }
  __syncthreads();
  const bool copy_q = qout != qin, copy_k = kout != kin;
  // rotated dims: (head, j) pairs
  for (int i = tid; i < (HQ + HKV) * 32; i += blockDim.x) {
    const int head = i / 32, j = i % 32;
    const __half* src;
    __half* dst;
    if (head < HQ) {
      src = qin + tok * ldqi + head * D;
      dst = qout + tok * ldqo + head * D;
    } else {
      src = kin + tok * ldki + (head - HQ) * D;
      dst = kout + tok * ldko + (head - HQ) * D;
    }
    const float x1 = __half2float(src[j]), x2 = __half2float(src[j + 32]);
    dst[j] = __float2half_rn(x1 * cs[j] - x2 * sn[j]);
    dst[j + 32] = __float2half_rn(x2 * cs[j] + x1 * sn[j]);
  }
  // pass-through dims 64..255 when writing a copy
  if (copy_q) {
    for (int i = tid; i < HQ * (D - 64) / 8; i += blockDim.x) {
      const int head = i / ((D - 64) / 8), c8 = 64 + (i % ((D - 64) / 8)) * 8;
      *reinterpret_cast<uint4*>(qout + tok * ldqo + head * D + c8) =
          *reinterpret_cast<const uint4*>(qin + tok * ldqi + head * D + c8);
    }
  }
  if (copy_k) {
    for (int i = tid; i < HKV * (D - 64) / 8; i += blockDim.x) {
      const int head = i / ((D - 64) / 8), c8 = 64 + (i % ((D - 64) / 8)) * 8;
      *reinterpret_cast<uint4*>(kout + tok * ldko + head * D + c8) =
          *reinterpret_cast<const uint4*>(kin + tok * ldki + head * D + c8);
    }
  }
}

struct FlashSmem {
  __half Q[BM][LDS];
  __half K[2][BN][LDS];
  __half V[2][BN][LDS];
};

__device__ __forceinline__ void load_kv(FlashSmem& s, int buf, const __half* __restrict__ k,
                                        int64_t ldk, const __half* __restrict__ v, int64_t ldv,
                                        int64_t tb, int key0, int L, int g, int tid) {
  for (int i = tid; i < BN * (D / 8); i += THREADS) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    const int key = key0 + r;
    const bool ok = key < L;
    const int64_t row = tb + (ok ? key : 0);
    cp_async16(smem_u32(&s.K[buf][r][c8]), k + row * ldk + g * D + c8, ok);
    cp_async16(smem_u32(&s.V[buf][r][c8]), v + row * ldv + g * D + c8, ok);
  }
  cp_async_commit();
}

__global__ void __launch_bounds__(THREADS, 1) flash_kernel(
    const __half* __restrict__ q, int64_t ldq, const __half* __restrict__ k, int64_t ldk,
    const __half* __restrict__ v, int64_t ldv, const __half* __restrict__ gate, int64_t ldg,
    __half* __restrict__ out, int64_t ldo, int L) {
  extern __shared__ __align__(16) uint8_t smraw[];
  FlashSmem& s = *reinterpret_cast<FlashSmem*>(smraw);
  // heavy (late) position blocks first
  const int pblk = gridDim.x - 1 - blockIdx.x;
  const int p0 = pblk * POS;
  const int g = blockIdx.y % HKV;
  const int b = blockIdx.y / HKV;
  const int64_t tb = (int64_t)b * L;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int gq = lane >> 2, tq = lane & 3;

  // Q rows: row r = 4 * (position - p0) + (query head - 4g)
  for (int i = tid; i < BM * (D / 8); i += THREADS) {
    const int r = i / (D / 8), c8 = (i % (D / 8)) * 8;
    const int p = p0 + (r >> 2);
    const bool ok = p < L;
    const int64_t row = tb + (ok ? p : 0);
    cp_async16(smem_u32(&s.Q[r][c8]), q + row * ldq + (4 * g + (r & 3)) * D + c8, ok);
  }
  cp_async_commit();
  const int last_pos = min(p0 + POS, L) - 1;
  const int ntiles = last_pos / BN + 1;
  load_kv(s, 0, k, ldk, v, ldv, tb, 0, L, g, tid);

  // this thread's two rows
  const int r_lo = warp * 16 + gq, r_hi = r_lo + 8;
  const int pos_lo = p0 + (r_lo >> 2), pos_hi = p0 + (r_hi >> 2);
  const float sl2 = 0.0625f * 1.4426950408889634f;  // softmax scale 1/sqrt(256), base 2
  float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
  float o[32][4];
#pragma unroll
  for (int n = 0; n < 32; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  const uint32_t sQ = smem_u32(&s.Q[0][0]);

  for (int t = 0; t < ntiles; ++t) {
    const int buf = t & 1;
    if (t + 1 < ntiles)
      load_kv(s, buf ^ 1, k, ldk, v, ldv, tb, (t + 1) * BN, L, g, tid);
    else
      cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();
    const int key0 = t * BN;
    const uint32_t sK = smem_u32(&s.K[buf][0][0]);
    const uint32_t sV = smem_u32(&s.V[buf][0][0]);
    // S = Q K^T for this warp's 16 rows x 64 keys
    float sc[8][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) {
      uint32_t a[4];
      ldsm_x4(a, a_addr(sQ, LDS, warp * 16, ks * 16, lane));
#pragma unroll
      for (int n = 0; n < 8; n += 2) {
        uint32_t bq[4];
        ldsm_x4(bq, bn_addr(sK, LDS, n * 8, ks * 16, lane));
        mma16816(sc[n], a, bq[0], bq[1]);
        mma16816(sc[n + 1], a, bq[2], bq[3]);
      }
    }
    // causal mask + online softmax (base-2 exponent, scale folded in)
    float mx_lo = -INFINITY, mx_hi = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const int key = key0 + n * 8 + 2 * tq;
      sc[n][0] = (key <= pos_lo) ? sc[n][0] * sl2 : -INFINITY;
      sc[n][1] = (key + 1 <= pos_lo) ? sc[n][1] * sl2 : -INFINITY;
      sc[n][2] = (key <= pos_hi) ? sc[n][2] * sl2 : -INFINITY;
      sc[n][3] = (key + 1 <= pos_hi) ? sc[n][3] * sl2 : -INFINITY;
      mx_lo = fmaxf(mx_lo, fmaxf(sc[n][0], sc[n][1]));
      mx_hi = fmaxf(mx_hi, fmaxf(sc[n][2], sc[n][3]));
    }
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 1));
    mx_lo = fmaxf(mx_lo, __shfl_xor_sync(0xffffffffu, mx_lo, 2));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 1));
    mx_hi = fmaxf(mx_hi, __shfl_xor_sync(0xffffffffu, mx_hi, 2));
    const float mn_lo = fmaxf(m_lo, mx_lo), mn_hi = fmaxf(m_hi, mx_hi);
    // rows whose keys are all masked so far keep m = -inf; use 0 as the reference then
    const float ref_lo = mn_lo == -INFINITY ? 0.f : mn_lo;
    const float ref_hi = mn_hi == -INFINITY ? 0.f : mn_hi;
    const float al_lo = exp2f(m_lo - ref_lo), al_hi = exp2f(m_hi - ref_hi);
    m_lo = mn_lo;
    m_hi = mn_hi;
    float rs_lo = 0.f, rs_hi = 0.f;
    uint32_t pa[4][4];
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const float e0 = exp2f(sc[n][0] - ref_lo), e1 = exp2f(sc[n][1] - ref_lo);
      const float e2 = exp2f(sc[n][2] - ref_hi), e3 = exp2f(sc[n][3] - ref_hi);
      rs_lo += e0 + e1;
      rs_hi += e2 + e3;
      const int j = n >> 1;
      if ((n & 1) == 0) {
        pa[j][0] = h2u(e0, e1);
        pa[j][1] = h2u(e2, e3);
      } else {
        pa[j][2] = h2u(e0, e1);
        pa[j][3] = h2u(e2, e3);
      }
    }
    l_lo = l_lo * al_lo + rs_lo;
    l_hi = l_hi * al_hi + rs_hi;
#pragma unroll
    for (int n = 0; n < 32; ++n) {
      o[n][0] *= al_lo; o[n][1] *= al_lo;
      o[n][2] *= al_hi; o[n][3] *= al_hi;
    }
    // O += P V
#pragma unroll
    for (int ks = 0; ks < BN / 16; ++ks) {
#pragma unroll
      for (int n = 0; n < 32; n += 2) {
        uint32_t bq[4];
        ldsm_x4_t(bq, bk_addr(sV, LDS, n * 8, ks * 16, lane));
        mma16816(o[n], pa[ks], bq[0], bq[1]);
        mma16816(o[n + 1], pa[ks], bq[2], bq[3]);
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();
  // epilogue: normalise, gate, store
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
  l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
  l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
  const float inv_lo = l_lo > 0.f ? 1.f / l_lo : 0.f;
  const float inv_hi = l_hi > 0.f ? 1.f / l_hi : 0.f;
#pragma unroll
  for (int hf = 0; hf < 2; ++hf) {
    const int r = hf ? r_hi : r_lo;
    const int p = hf ? pos_hi : pos_lo;
    if (p >= L) continue;
    const float inv = hf ? inv_hi : inv_lo;
    const int hq = 4 * g + (r & 3);
    const int64_t row = tb + p;
#pragma unroll
    for (int n = 0; n < 32; ++n) {
      const int col = n * 8 + 2 * tq;
      float a0 = o[n][2 * hf] * inv, a1 = o[n][2 * hf + 1] * inv;
      if (gate) {
        const float2 gf =
            __half22float2(*reinterpret_cast<const __half2*>(gate + row * ldg + hq * D + col));
        a0 *= sigmoid_f(gf.x);
        a1 *= sigmoid_f(gf.y);
      }
      *reinterpret_cast<uint32_t*>(out + row * ldo + hq * D + col) = h2u(a0, a1);
    }
  }
}

}  // namespace attn

clef_status rope_launch(const __half* qin, int64_t ldqi, __half* qout, int64_t ldqo,
                        const __half* kin, int64_t ldki, __half* kout, int64_t ldko, int64_t M,
                        int64_t L, cudaStream_t stream) {
  if (M == 0) return CLEF_OK;
  TraceScope ts(stream, "rope", 0.0, M * (20.0 * 64 * 2 * 2));
  attn::rope_kernel<<<(unsigned)M, 128, 0, stream>>>(qin, ldqi, qout, ldqo, kin, ldki, kout, ldko,
                                                     (int)L);
  CLEF_LAUNCH_CHECK();
  return CLEF_OK;
}

clef_status flash_launch(const __half* q, int64_t ldq, const __half* k, int64_t ldk,
                         const __half* v, int64_t ldv, const __half* gate, int64_t ldg, __half* out,
                         int64_t ldo, int64_t B, int64_t L, cudaStream_t stream) {
  if (B == 0 || L == 0) return CLEF_OK;
  static bool attr = false;
  if (!attr) {
    CLEF_CUDA_CHECK(cudaFuncSetAttribute(attn::flash_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         sizeof(attn::FlashSmem)));
    attr = true;
  }
  dim3 grid((unsigned)((L + attn::POS - 1) / attn::POS), (unsigned)(B * attn::HKV));
  TraceScope ts(stream, "flash_attn", 4.0 * attn::D * attn::HQ * (double)B * L * (L + 1) / 2.0,
                (double)B * L * (16 + 4 + 4 + 16 + 16) * attn::D * 2.0);
  attn::flash_kernel<<<grid, attn::THREADS, sizeof(attn::FlashSmem), stream>>>(
      q, ldq, k, ldk, v, ldv, gate, ldg, out, ldo, (int)L);
  CLEF_LAUNCH_CHECK();
  return CLEF_OK;
}

}  // namespace clef
