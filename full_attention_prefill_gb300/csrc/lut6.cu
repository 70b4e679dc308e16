// LUT-6 weights: host pack/unpack, a dense dequant kernel (parity aid) and the LUT-6 GEMM.
//
// Format ("Clef-Flash-ANE-LUT6" model card, sections "Weight precision" and "LUT-6 text
// weights"): 6-bit indices, one 64-entry fp16 table per 16 output channels, four indices packed
// into three bytes as one little-endian (LSB-first) bit stream, rows of W in order, k fastest.
//
// GEMM design (sm_103a): Y[m, n] = sum_k X[m, k] * T[n/16][idx[n, k]].
//   * one CTA per 256 (tokens) x 128 (output channels) tile, K walked in blocks of 64;
//   * warp 0 issues TMA loads of the X tile (256 rows, 128-byte swizzle) and of the packed
//     index tile (128 rows x 48 bytes) into a 4-stage ring;
//   * warps 4..19 turn the packed tile into the fp16 weight tile in shared memory: each lane
//     unpacks 16 indices from 12 bytes (index*2 is cut out and OR'd into its table's address in
//     one logic op) and looks them up in its group's 64-entry table, which sits in 128 bytes =
//     one entry pair per bank, so a warp (8 rows of one 16-row group) never conflicts; the tile
//     is written directly in the 128-byte-swizzled K-major layout;
//   * warp 1 issues two tcgen05.mma per K=16 step (M=128 each, N=128, fp16 x fp16 -> fp32), one
//     per 128-token half, both reading the same weight tile, into two 128 x 128 fp32
//     accumulators in tensor memory: each dequantised weight serves 256 tokens;
//   * warps 4..19 then read the accumulators with tcgen05.ld and run the fused epilogue (fp16
//     or fp32 store, fp32 residual add, or SwiGLU of an interleaved gate/up tile).
// The dense weight never reaches global memory.
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"
#include "lut6.cuh"

namespace clef {
namespace lut {

constexpr int BM = 256;                       // tokens per tile: two M = 128 MMAs
constexpr int BN = 128;                       // output channels per tile
constexpr int BK = 64;
constexpr int STAGES = 4;
constexpr int X_BYTES = BM * BK * 2;          // 32 KB
constexpr int W_BYTES = BN * BK * 2;          // 16 KB
constexpr int P_ROW = BK * 3 / 4;             // 48 packed bytes per row per k-block
constexpr int P_BYTES = BN * P_ROW;           // 6 KB
constexpr int TBL_BYTES = (BN / 16) * 64 * 2; // 1 KB: the 8 tables of the tile's rows
constexpr int NUM_DQ_WARPS = 16;
constexpr int NUM_THREADS = 32 * (4 + NUM_DQ_WARPS);
constexpr int TMEM_COLS = 256;                // two 128-column fp32 accumulators

constexpr int OFF_X = 0;
constexpr int OFF_W = OFF_X + STAGES * X_BYTES;
constexpr int OFF_P = OFF_W + STAGES * W_BYTES;
constexpr int OFF_T = OFF_P + STAGES * P_BYTES;
constexpr int OFF_BAR = OFF_T + TBL_BYTES;
constexpr int OFF_SLOT = OFF_BAR + 16 * 8;
constexpr int SMEM_USED = OFF_SLOT + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(BN == 2 * CLEF_SWIGLU_BLOCK, "a SwiGLU tile holds one gate block and its up block");

static_assert(OFF_W % 1024 == 0 && OFF_P % 1024 == 0, "tile alignment");

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

// Table addresses of 16 indices of 6 bits taken from 96 bits (w0 | w1 << 32 | w2 << 64), LSB
// first: index i sits at bits 6i..6i+5; (index * 2) is cut out and OR'd into the table base tb
// (128-byte aligned), one shift and one logic op per index.
__device__ __forceinline__ void table_addrs16(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t tb,
                                              uint32_t (&a)[16]) {
  a[0] = ((w0 << 1) & 0x7Eu) | tb;
  a[1] = ((w0 >> 5) & 0x7Eu) | tb;
  a[2] = ((w0 >> 11) & 0x7Eu) | tb;
  a[3] = ((w0 >> 17) & 0x7Eu) | tb;
  a[4] = ((w0 >> 23) & 0x7Eu) | tb;
  a[5] = (__funnelshift_r(w0, w1, 29) & 0x7Eu) | tb;
  a[6] = ((w1 >> 3) & 0x7Eu) | tb;
  a[7] = ((w1 >> 9) & 0x7Eu) | tb;
  a[8] = ((w1 >> 15) & 0x7Eu) | tb;
  a[9] = ((w1 >> 21) & 0x7Eu) | tb;
  a[10] = (__funnelshift_r(w1, w2, 27) & 0x7Eu) | tb;
  a[11] = ((w2 >> 1) & 0x7Eu) | tb;
  a[12] = ((w2 >> 7) & 0x7Eu) | tb;
  a[13] = ((w2 >> 13) & 0x7Eu) | tb;
  a[14] = ((w2 >> 19) & 0x7Eu) | tb;
  a[15] = ((w2 >> 25) & 0x7Eu) | tb;
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
  const int m0 = blockIdx.y * BM;
  const int num_kb = K / BK;

  const uint32_t bar_full = sb + OFF_BAR;                   // [STAGES]
  const uint32_t bar_wready = sb + OFF_BAR + 8 * STAGES;    // [STAGES]
  const uint32_t bar_empty = sb + OFF_BAR + 16 * STAGES;    // [STAGES]
  const uint32_t bar_acc = sb + OFF_BAR + 24 * STAGES;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_SLOT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(bar_full + 8 * s, 1);
      mbar_init(bar_wready + 8 * s, NUM_DQ_WARPS);
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
      constexpr uint32_t idesc = idesc_f16_f32(128, BN);
      bool ok = true;
      for (int kb = 0; kb < num_kb && ok; ++kb) {
        const int s = kb % STAGES;
        const uint32_t ph = (kb / STAGES) & 1;
        ok = mbar_wait(bar_full + 8 * s, ph, status, DEV_TIMEOUT_MMA) &&
             mbar_wait(bar_wready + 8 * s, ph, status, DEV_TIMEOUT_MMA);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t bd = sdesc_k_sw128(sb + OFF_W + s * W_BYTES + kk * 32);
          const uint64_t a0 = sdesc_k_sw128(sb + OFF_X + s * X_BYTES + kk * 32);
          const uint64_t a1 = sdesc_k_sw128(sb + OFF_X + s * X_BYTES + 16384 + kk * 32);
          tc_mma_f16_ss(tmem, a0, bd, idesc, (kb | kk) != 0);
          tc_mma_f16_ss(tmem + BN, a1, bd, idesc, (kb | kk) != 0);
        }
        tc_commit(bar_empty + 8 * s);
      }
      tc_commit(bar_acc);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- dequant, then epilogue
    const int dq = warp - 4;              // 0..15
    const int t = threadIdx.x - 128;      // 0..511
    if (t < 256) {
      // the tile's 8 tables (rows n0 .. n0+127); groups past N read as zero
      const int e = t * 2;
      const int g = n0 / 16 + e / 64;
      uint32_t v = 0u;
      if (g < N / 16) v = *reinterpret_cast<const uint32_t*>(lut + (size_t)g * 64 + (e & 63));
      *reinterpret_cast<uint32_t*>(smem + OFF_T + e * 2) = v;
    }
    named_bar_sync(1, 32 * NUM_DQ_WARPS);
    const int rsub = lane >> 2;  // row inside the 8-row task
    const int q4 = lane & 3;     // which 16 of the 64 k-values
    bool ok = true;
    for (int kb = 0; kb < num_kb; ++kb) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      // full[s] completing implies the producer saw empty[s] of the previous round, so the
      // weight buffer of stage s is free as well.
      if (!mbar_wait(bar_full + 8 * s, ph, status, DEV_TIMEOUT_DEQUANT)) {
        ok = false;
        break;
      }
      const uint32_t pbase = sb + OFF_P + s * P_BYTES;
      const uint32_t wbase = sb + OFF_W + s * W_BYTES;
#pragma unroll
      for (int it = 0; it < BN / 8 / NUM_DQ_WARPS; ++it) {
        const int row = (dq + NUM_DQ_WARPS * it) * 8 + rsub;  // 0..127
        const uint32_t pa = pbase + row * P_ROW + q4 * 12;
        const uint32_t w0 = lds_u32(pa), w1 = lds_u32(pa + 4), w2 = lds_u32(pa + 8);
        uint32_t a[16];
        table_addrs16(w0, w1, w2, sb + OFF_T + (row >> 4) * 128, a);
        uint32_t o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = lds_pair(a[2 * i], a[2 * i + 1]);
        const uint32_t wrow = wbase + (row >> 3) * 1024 + (row & 7) * 128;
        sts_v4(wrow + (((2 * q4) ^ (row & 7)) << 4), o[0], o[1], o[2], o[3]);
        sts_v4(wrow + (((2 * q4 + 1) ^ (row & 7)) << 4), o[4], o[5], o[6], o[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_wready + 8 * s);
    }
    // ---- epilogue: warp dq drains accumulator (dq >> 2) & 1 (tokens 0..127 or 128..255),
    //      TMEM lanes 32 (dq & 3).., columns 64 (dq >> 3) .. +63
    if (ok && mbar_wait(bar_acc, 0, status, DEV_TIMEOUT_EPILOGUE)) {
      tc_fence_after();
      const int quarter = warp & 3;
      const int half = (dq >> 2) & 1;
      const int chalf = dq >> 3;
      const int row = m0 + half * 128 + quarter * 32 + lane;
      const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16) + half * BN;
      if (mode == EPI_SWIGLU_F16) {
        {
          const int j0 = chalf * 32;
          uint32_t g[32], u[32];
          tmem_ld_32x32b_x32(tl + j0, g);
          tmem_ld_32x32b_x32(tl + BN / 2 + j0, u);
          tc_wait_ld();
          if (row < M) {
            __half* out = reinterpret_cast<__half*>(y) + (int64_t)row * ldy + n0 / 2 + j0;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t pk[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float g0 = __uint_as_float(g[8 * q + 2 * i]);
                const float g1 = __uint_as_float(g[8 * q + 2 * i + 1]);
                const float u0 = __uint_as_float(u[8 * q + 2 * i]);
                const float u1 = __uint_as_float(u[8 * q + 2 * i + 1]);
                pk[i] = pack_half2(silu_f(g0) * u0, silu_f(g1) * u1);
              }
              *reinterpret_cast<uint4*>(out + 8 * q) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
          }
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
          const int col0 = chalf * 64 + c * 32;
          uint32_t r[32];
          tmem_ld_32x32b_x32(tl + col0, r);
          tc_wait_ld();
          if (row < M) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int n = n0 + col0 + 8 * q;
              if (n >= N) continue;
              if (mode == EPI_F16) {
                __half* out = reinterpret_cast<__half*>(y) + (int64_t)row * ldy + n;
                *reinterpret_cast<uint4*>(out) = make_uint4(
                    pack_half2(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1])),
                    pack_half2(__uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3])),
                    pack_half2(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5])),
                    pack_half2(__uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7])));
              } else {
                float* out = reinterpret_cast<float*>(y) + (int64_t)row * ldy + n;
                float4 a = make_float4(__uint_as_float(r[8 * q + 0]), __uint_as_float(r[8 * q + 1]),
                                       __uint_as_float(r[8 * q + 2]), __uint_as_float(r[8 * q + 3]));
                float4 b = make_float4(__uint_as_float(r[8 * q + 4]), __uint_as_float(r[8 * q + 5]),
                                       __uint_as_float(r[8 * q + 6]), __uint_as_float(r[8 * q + 7]));
                if (mode == EPI_ADD_F32) {
                  const float4 a0 = reinterpret_cast<float4*>(out)[0];
                  const float4 b0 = reinterpret_cast<float4*>(out)[1];
                  a.x += a0.x; a.y += a0.y; a.z += a0.z; a.w += a0.w;
                  b.x += b0.x; b.y += b0.y; b.z += b0.z; b.w += b0.w;
                }
                reinterpret_cast<float4*>(out)[0] = a;
                reinterpret_cast<float4*>(out)[1] = b;
              }
            }
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
                    (uint64_t)K * 2, BK, BM, CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess)
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
  dim3 grid((unsigned)((N + BN - 1) / BN), (unsigned)((M + BM - 1) / BM));
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
