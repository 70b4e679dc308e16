// LUT-6 weights: host pack/unpack, a dense dequant kernel (parity aid) and the LUT-6 GEMM.
//
// Format ("Clef-Flash-ANE-LUT6" model card, sections "Weight precision" and "LUT-6 text
// weights"): 6-bit indices, one 64-entry fp16 table per 16 output channels, four indices packed
// into three bytes as one little-endian (LSB-first) bit stream, rows of W in order, k fastest.
//
// GEMM design (sm_103a): Y[m, n] = sum_k X[m, k] * T[n/16][idx[n, k]], computed as the
// transposed product D[n, m] = W X^T so that the weights are the MMA's A operand, held in tensor
// memory, and never pass through shared memory:
//   * one CTA per 128 (output channels) x 256 (tokens) tile, K walked in blocks of 64;
//   * warp 0 issues TMA loads of the X tile (256 tokens x 64, 128-byte swizzle) and of the packed
//     index tile (128 rows x 48 bytes) into a 4-stage ring;
//   * warps 4..11 dequantise: each warp owns one 16-row table group and writes its 16 x 64
//     weights straight into a tensor-memory A stage with one tcgen05.st.16x256b.x4; every
//     lookup of a warp hits the same 64-entry table (128 bytes, one entry pair per bank), so the
//     lookups never conflict; each lane takes the packed quadruples its fragment needs out of
//     two aligned words with one funnel shift, and cuts index*2 into the table address with one
//     logic op per index;
//   * warp 1 issues tcgen05.mma (M=128 channels from tensor memory, N=256 tokens from shared
//     memory, K=16) into a 128 x 256 fp32 accumulator in tensor memory;
//   * the epilogue (warps 4..11) drains the accumulator with tcgen05.ld into shared memory in
//     token-major order and writes Y coalesced (fp16 or fp32 store, fp32 residual add, or SwiGLU
//     of an interleaved gate/up tile).
// The dense weight never reaches global memory.
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"
#include "lut6.cuh"

namespace clef {
namespace lut {

constexpr int BN = 128;                       // output channels per tile: MMA M (A operand)
constexpr int BT = 256;                       // tokens per tile: MMA N (B operand)
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int X_BYTES = BT * BK * 2;          // 32 KB
constexpr int P_ROW = BK * 3 / 4;             // 48 packed bytes per row per k-block
constexpr int P_BYTES = BN * P_ROW;           // 6 KB
constexpr int TBL_BYTES = (BN / 16) * 64 * 2; // 1 KB: the 8 tables of the tile's rows
constexpr int NUM_DQ_WARPS = 8;               // one per 16-row group
constexpr int NUM_THREADS = 32 * (4 + NUM_DQ_WARPS);
constexpr int TMEM_COLS = 512;
constexpr uint32_t A_COL = BT;                // A stages: 32 columns each from column 256

constexpr int OFF_X = 0;                      // also the epilogue's staging area (128 KB)
constexpr int OFF_P = OFF_X + STAGES * X_BYTES;
constexpr int OFF_T = OFF_P + STAGES * P_BYTES;
constexpr int OFF_BAR = OFF_T + TBL_BYTES;
constexpr int OFF_SLOT = OFF_BAR + 16 * 8;
constexpr int SMEM_USED = OFF_SLOT + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(STAGES * X_BYTES >= BT * BN * 4, "epilogue staging fits in the X ring");
static_assert(BN == 2 * CLEF_SWIGLU_BLOCK, "a SwiGLU tile holds one gate block and its up block");
static_assert(A_COL + STAGES * 32 <= TMEM_COLS, "tensor memory budget");

__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}
__device__ __forceinline__ void sts_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Two fp16 table entries packed into one 32-bit word (first in the low half).
__device__ __forceinline__ uint32_t lds_pair(uint32_t a0, uint32_t a1) {
  uint32_t v;
  asm volatile(
      "{\n\t.reg .b16 lo, hi;\n\t"
      "ld.shared.b16 lo, [%1];\n\t"
      "ld.shared.b16 hi, [%2];\n\t"
      "mov.b32 %0, {lo, hi};\n\t}"
      : "=r"(v)
      : "r"(a0), "r"(a1));
  return v;
}

// 16 TMEM lanes x 32 columns from registers: thread t holds, for column block j (8 columns),
// r[4j], r[4j+1] = row t/4, columns 8j + 2(t%4) + {0, 1} and r[4j+2], r[4j+3] = row t/4 + 8.
__device__ __forceinline__ void tmem_st_16x256b_x4(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

// The packed quadruple q (indices 4q..4q+3 of a row, 24 bits at byte 3q) of a row starting at
// shared address `row`, as four table addresses (index * 2 OR'd into the 128-byte aligned tb).
__device__ __forceinline__ void quad_addrs(uint32_t row, int q, uint32_t tb, uint32_t (&a)[4]) {
  const int off = 3 * q;
  const uint32_t wa = row + (off & ~3);
  const uint32_t lo = lds_u32(wa), hi = lds_u32(wa + 4);
  const uint32_t w = __funnelshift_r(lo, hi, (off & 3) * 8);
  a[0] = ((w << 1) & 0x7Eu) | tb;
  a[1] = ((w >> 5) & 0x7Eu) | tb;
  a[2] = ((w >> 11) & 0x7Eu) | tb;
  a[3] = ((w >> 17) & 0x7Eu) | tb;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    lut6_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                     const __grid_constant__ CUtensorMap tmap_p, const __half* __restrict__ lut,
                     void* __restrict__ y, int64_t ldy, int M, int N, int K, int mode,
                     unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN;
  const int m0 = blockIdx.y * BT;
  const int num_kb = K / BK;

  const uint32_t bar_full = sb + OFF_BAR;                   // [STAGES] X + packed landed
  const uint32_t bar_aready = sb + OFF_BAR + 8 * STAGES;    // [STAGES] A stage written
  const uint32_t bar_empty = sb + OFF_BAR + 16 * STAGES;    // [STAGES] MMAs of a stage done
  const uint32_t bar_acc = sb + OFF_BAR + 24 * STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_SLOT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_aready + 8 * s, NUM_DQ_WARPS);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_acc, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_p);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      for (int kb = 0; kb < num_kb; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (kb / STAGES) & 1;
        if (kb >= STAGES && !mbar_wait(bar_empty + 8 * s, ph ^ 1, status, DEV_TIMEOUT_TMA)) break;
        mbar_arrive_expect_tx(bar_full + 8 * s, X_BYTES + P_BYTES);
        tma_load_2d(sb + OFF_X + s * X_BYTES, &tmap_x, bar_full + 8 * s, kb * BK, m0);
        tma_load_2d(sb + OFF_P + s * P_BYTES, &tmap_p, bar_full + 8 * s, kb * P_ROW, n0);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BN, BT);
      bool ok = true;
      for (int kb = 0; kb < num_kb && ok; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (kb / STAGES) & 1;
        ok = mbar_wait(bar_full + 8 * s, ph, status, DEV_TIMEOUT_MMA) &&
             mbar_wait(bar_aready + 8 * s, ph, status, DEV_TIMEOUT_MMA);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t bd = sdesc_k_sw128(sb + OFF_X + s * X_BYTES + kk * 32);
          tc_mma_f16_ts(tmem, tmem + A_COL + s * 32 + kk * 8, bd, idesc, (kb | kk) != 0);
        }
        tc_commit(bar_empty + 8 * s);
      }
      tc_commit(bar_acc);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- dequant, then epilogue
    const int dq = warp - 4;              // 0..7
    const int t = threadIdx.x - 128;      // 0..255
    {
      // the tile's 8 tables (rows n0 .. n0+127); groups past N read as zero
      const int e = t * 2;
      const int g = n0 / 16 + e / 64;
      uint32_t v = 0u;
      if (g < N / 16) v = *reinterpret_cast<const uint32_t*>(lut + (size_t)g * 64 + (e & 63));
      *reinterpret_cast<uint32_t*>(smem + OFF_T + e * 2) = v;
    }
    named_bar_sync(1, 32 * NUM_DQ_WARPS);
    const int quarter = warp & 3;         // TMEM lanes 32*quarter .. (this warp's access window)
    const int grp = 2 * quarter + (dq >> 2);          // 16-row group of this warp
    const int r0 = grp * 16 + (lane >> 2);            // rows r0 and r0 + 8 of the group
    const int u = lane & 3;
    const uint32_t tb = sb + OFF_T + grp * 128;
    const uint32_t tl = tmem + ((uint32_t)(grp * 16) << 16) + A_COL;
    bool ok = true;
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      // full[s] completing implies the producer saw empty[s] of the previous round, so the
      // MMAs that read A stage s before have finished as well.
      if (!mbar_wait(bar_full + 8 * s, ph, status, DEV_TIMEOUT_DEQUANT)) {
        ok = false;
        break;
      }
      const uint32_t prow0 = sb + OFF_P + s * P_BYTES + r0 * P_ROW;
      const uint32_t prow1 = prow0 + 8 * P_ROW;
      uint32_t rg[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // fragment block j holds k = 16j + 4u .. 16j + 4u + 3: packed quadruple 4j + u
        uint32_t a0[4], a1[4];
        quad_addrs(prow0, 4 * j + u, tb, a0);
        quad_addrs(prow1, 4 * j + u, tb, a1);
        rg[4 * j + 0] = lds_pair(a0[0], a0[1]);
        rg[4 * j + 1] = lds_pair(a0[2], a0[3]);
        rg[4 * j + 2] = lds_pair(a1[0], a1[1]);
        rg[4 * j + 3] = lds_pair(a1[2], a1[3]);
      }
      tmem_st_16x256b_x4(tl + s * 32, rg);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_aready + 8 * s);
    }
    // ---- epilogue: accumulator (lane = channel, column = token) -> shared, token-major fp32
    const bool got = ok && mbar_wait(bar_acc, 0, status, DEV_TIMEOUT_EPILOGUE);
    if (got) {
      tc_fence_after();
      float* stg = reinterpret_cast<float*>(smem + OFF_X);
      const int ch = quarter * 32 + lane;
      const int tok0 = (dq >> 2) * 128;
#pragma unroll 1
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + ((uint32_t)(quarter * 32) << 16) + tok0 + c * 32, r);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i) stg[(tok0 + c * 32 + i) * BN + ch] = __uint_as_float(r[i]);
      }
    }
    named_bar_sync(2, 32 * NUM_DQ_WARPS);
    if (got) {
      const float* stg = reinterpret_cast<const float*>(smem + OFF_X);
      if (mode == EPI_SWIGLU_F16) {
        const int c8 = (t & 7) * 8;
#pragma unroll 1
        for (int tok = t >> 3; tok < BT; tok += 32) {
          const int row = m0 + tok;
          if (row >= M) break;
          const float4* gp = reinterpret_cast<const float4*>(stg + tok * BN + c8);
          const float4* up = reinterpret_cast<const float4*>(stg + tok * BN + BN / 2 + c8);
          const float4 g0 = gp[0], g1 = gp[1], u0 = up[0], u1 = up[1];
          uint4 o;
          o.x = pack_half2(silu_f(g0.x) * u0.x, silu_f(g0.y) * u0.y);
          o.y = pack_half2(silu_f(g0.z) * u0.z, silu_f(g0.w) * u0.w);
          o.z = pack_half2(silu_f(g1.x) * u1.x, silu_f(g1.y) * u1.y);
          o.w = pack_half2(silu_f(g1.z) * u1.z, silu_f(g1.w) * u1.w);
          *reinterpret_cast<uint4*>(reinterpret_cast<__half*>(y) + (int64_t)row * ldy + n0 / 2 + c8) = o;
        }
      } else {
        const int c8 = (t & 15) * 8;
        const bool col_ok = n0 + c8 < N;
#pragma unroll 1
        for (int tok = t >> 4; tok < BT; tok += 16) {
          const int row = m0 + tok;
          if (row >= M) break;
          if (!col_ok) continue;
          const float4 a = reinterpret_cast<const float4*>(stg + tok * BN + c8)[0];
          const float4 b = reinterpret_cast<const float4*>(stg + tok * BN + c8)[1];
          if (mode == EPI_F16) {
            __half* out = reinterpret_cast<__half*>(y) + (int64_t)row * ldy + n0 + c8;
            *reinterpret_cast<uint4*>(out) = make_uint4(pack_half2(a.x, a.y), pack_half2(a.z, a.w),
                                                        pack_half2(b.x, b.y), pack_half2(b.z, b.w));
          } else {
            float4* out = reinterpret_cast<float4*>(reinterpret_cast<float*>(y) + (int64_t)row * ldy + n0 + c8);
            float4 a2 = a, b2 = b;
            if (mode == EPI_ADD_F32) {
              const float4 a0 = out[0], b0 = out[1];
              a2.x += a0.x; a2.y += a0.y; a2.z += a0.z; a2.w += a0.w;
              b2.x += b0.x; b2.y += b0.y; b2.z += b0.z; b2.w += b0.w;
            }
            out[0] = a2;
            out[1] = b2;
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// One thread per packed quadruple (3 bytes -> 4 fp16 weights).
__global__ void lut6_dequant_kernel(const uint8_t* __restrict__ packed, const __half* __restrict__ lut,
                                    int64_t n, int64_t k, __half* __restrict__ w) {
  const int64_t quads = n * (k / 4);
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < quads;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = q / (k / 4);
    const uint8_t* p = packed + q * 3;
    const uint32_t word = (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16);
    const __half* tbl = lut + (row / 16) * 64;
    __half* out = w + q * 4;
#pragma unroll
    for (int j = 0; j < 4; ++j) out[j] = tbl[(word >> (6 * j)) & 63u];
  }
}

}  // namespace lut

clef_status lut6_gemm_launch(const __half* x, const uint8_t* packed, const __half* lut, void* y,
                             int64_t ldy, int64_t M, int64_t N, int64_t K, int mode,
                             cudaStream_t stream) {
  using namespace lut;
  if (M == 0) return CLEF_OK;
  CUtensorMap tx, tp;
  if (tma_encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, (uint64_t)K, (uint64_t)M,
                    (uint64_t)K * 2, BK, BT, CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess)
    return CLEF_E_CUDA;
  if (tma_encode_2d(&tp, CU_TENSOR_MAP_DATA_TYPE_UINT8, packed, (uint64_t)K * 3 / 4, (uint64_t)N,
                    (uint64_t)K * 3 / 4, P_ROW, BN, CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess)
    return CLEF_E_CUDA;
  static bool attr_set = false;
  if (!attr_set) {
    CLEF_CUDA_CHECK(cudaFuncSetAttribute(lut6_gemm_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES));
    attr_set = true;
  }
  dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BT - 1) / BT));
  const double out_bytes = mode == EPI_F16 ? 2.0 * M * N
                           : mode == EPI_F32 ? 4.0 * M * N
                           : mode == EPI_ADD_F32 ? 8.0 * M * N
                                                 : 1.0 * M * N;  // SwiGLU: fp16 [M, N/2]
  TraceScope ts(stream, "lut6_gemm", 2.0 * M * N * K,
                0.75 * N * K + 8.0 * N + 2.0 * M * K + out_bytes);
  lut6_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, stream>>>(
      tx, tp, lut, y, ldy, (int)M, (int)N, (int)K, mode, status_word_ptr());
  CLEF_LAUNCH_CHECK();
  return CLEF_OK;
}

clef_status lut6_dequant_launch(const uint8_t* packed, const __half* lut, int64_t n, int64_t k,
                                __half* w, cudaStream_t stream) {
  const int64_t quads = n * (k / 4);
  if (quads == 0) return CLEF_OK;
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((quads + threads - 1) / threads, 65535LL * 8);
  TraceScope ts(stream, "lut6_dequant", 0.0, 0.75 * n * k + 2.0 * n * k);
  lut::lut6_dequant_kernel<<<(unsigned)blocks, threads, 0, stream>>>(packed, lut, n, k, w);
  CLEF_LAUNCH_CHECK();
  return CLEF_OK;
}

}  // namespace clef
