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
//   * warp 0 issues TMA loads of the X tile (256 tokens x 64, 128-byte swizzle) and of the 8
//     packed 768-byte blocks of the tile's rows (tiled layout, see clef_lut6_tile) into a 4-stage
//     ring;
//   * warps 4..19 dequantise: each warp owns one 16-row table group on every other k-block and
//     writes its 16 x 64 weights straight into a tensor-memory A stage with one
//     tcgen05.st.16x256b.x4 (two warps per group take turns, so each has two MMA periods to
//     cover its chain of dependent loads); every
//     lookup of a warp hits the same 64-entry table (128 bytes, one entry pair per bank), so the
//     lookups never conflict; in the tiled layout the 32 indices a lane's fragment needs are 24
//     contiguous bytes (three 8-byte loads), and index*2 is cut into the table address with one
//     shift and one logic op per index;
//   * warp 1 issues tcgen05.mma (M=128 channels from tensor memory, N=256 tokens from shared
//     memory, K=16) into a 128 x 256 fp32 accumulator in tensor memory;
//   * the epilogue (warps 4..19) drains the accumulator with tcgen05.ld into shared memory in
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
constexpr int P_BLOCK = 768;                  // packed bytes of one 16-row group per k-block
constexpr int P_BYTES = (BN / 16) * P_BLOCK;  // 6 KB
constexpr int TBL_BYTES = (BN / 16) * 64 * 2; // 1 KB: the 8 tables of the tile's rows
constexpr int NUM_DQ_WARPS = 16;              // two per 16-row group (even / odd k-blocks)
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
__device__ __forceinline__ void lds_v2(uint32_t addr, uint32_t& a, uint32_t& b) {
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(a), "=r"(b) : "r"(addr));
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
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
      mbar_init(bar_aready + 8 * s, NUM_DQ_WARPS / 2);
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
        // the 8 groups' 768-byte blocks of k-block kb: box {256 B, 3, 8 groups}
        tma_load_3d(sb + OFF_P + s * P_BYTES, &tmap_p, bar_full + 8 * s, 0, 3 * kb, n0 / 16);
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
    const int quarter = warp & 3;         // TMEM lanes 32*quarter .. (this warp's access window)
    const int grp = 2 * quarter + ((dq >> 2) & 1);    // 16-row group of this warp
    const int par = dq >> 3;                          // k-blocks kb with kb % 2 == par
    const uint32_t tb = sb + OFF_T + grp * 128;
    const uint32_t tl = tmem + ((uint32_t)(grp * 16) << 16) + A_COL;
    bool ok = true;
    for (int kb = par; kb < num_kb; kb += 2) {
      const int s = kb % STAGES;
      const uint32_t ph = (kb / STAGES) & 1;
      // full[s] completing implies the producer saw empty[s] of the previous round, so the
      // MMAs that read A stage s before have finished as well.
      if (!mbar_wait(bar_full + 8 * s, ph, status, DEV_TIMEOUT_DEQUANT)) {
        ok = false;
        break;
      }
      // this lane's 24 bytes: quadruples j = 0..3 of row r0, then of row r0 + 8
      const uint32_t pa = sb + OFF_P + s * P_BYTES + (grp & 7) * P_BLOCK + lane * 24;
      uint32_t w[6];
      lds_v2(pa, w[0], w[1]);
      lds_v2(pa + 8, w[2], w[3]);
      lds_v2(pa + 16, w[4], w[5]);
      uint32_t a0[16], a1[16];
      table_addrs16(w[0], w[1], w[2], tb, a0);
      table_addrs16(w[3], w[4], w[5], tb, a1);
      uint32_t rg[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        // fragment block j holds k = 16j + 4u .. 16j + 4u + 3 of rows r0 and r0 + 8
        rg[4 * j + 0] = lds_pair(a0[4 * j], a0[4 * j + 1]);
        rg[4 * j + 1] = lds_pair(a0[4 * j + 2], a0[4 * j + 3]);
        rg[4 * j + 2] = lds_pair(a1[4 * j], a1[4 * j + 1]);
        rg[4 * j + 3] = lds_pair(a1[4 * j + 2], a1[4 * j + 3]);
      }
      tmem_st_16x256b_x4(tl + s * 32, rg);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_aready + 8 * s);
    }
    // ---- epilogue: accumulator (lane = channel, column = token) -> shared, token-major fp32;
    //      warp dq takes TMEM lanes 32 (dq & 3).. and token columns 64 (dq >> 2) .. +63
    const bool got = ok && mbar_wait(bar_acc, 0, status, DEV_TIMEOUT_EPILOGUE);
    if (got) {
      tc_fence_after();
      float* stg = reinterpret_cast<float*>(smem + OFF_X);
      const int ch = quarter * 32 + lane;
      const int tok0 = (dq >> 2) * 64;
#pragma unroll 1
      for (int c = 0; c < 2; ++c) {
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
        for (int tok = t >> 3; tok < BT; tok += 64) {
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
        for (int tok = t >> 4; tok < BT; tok += 32) {
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

// Canonical packed [n, k*3/4] -> tiled: one thread per 3-byte quadruple of the output.
//   tiled[((G * (k/64) + kb) * 32 + t) * 24 + 3 * (4h + j) + b]
//     = packed[16G + t/4 + 8h][3 * (16kb + 4j + t%4) + b]
__global__ void lut6_tile_kernel(const uint8_t* __restrict__ packed, int64_t n, int64_t k,
                                 uint8_t* __restrict__ tiled) {
  const int64_t quads = n * (k / 4);
  const int64_t kbs = k / 64;
  for (int64_t q = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; q < quads;
       q += (int64_t)gridDim.x * blockDim.x) {
    const int hj = (int)(q % 8);
    const int t = (int)((q / 8) % 32);
    const int64_t blk = q / 256;  // G * kbs + kb
    const int64_t kb = blk % kbs, G = blk / kbs;
    const int h = hj >> 2, j = hj & 3;
    const int64_t row = 16 * G + t / 4 + 8 * h;
    const int64_t src = row * (k / 4 * 3) + 3 * (16 * kb + 4 * j + t % 4);
    uint8_t* d = tiled + q * 3;
    d[0] = packed[src];
    d[1] = packed[src + 1];
    d[2] = packed[src + 2];
  }
}

}  // namespace lut

clef_status lut6_gemm_launch(const __half* x, const uint8_t* tiled, const __half* lut, void* y,
                             int64_t ldy, int64_t M, int64_t N, int64_t K, int mode,
                             cudaStream_t stream) {
  using namespace lut;
  if (M == 0) return CLEF_OK;
  CUtensorMap tx, tp;
  if (tma_encode_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, (uint64_t)K, (uint64_t)M,
                    (uint64_t)K * 2, BK, BT, CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess)
    return CLEF_E_CUDA;
  {
    // tiled weights as [N/16 groups][3 * K/64][256 bytes]; groups past N read as zero
    const uint64_t dims[3] = {256, (uint64_t)(3 * (K / BK)), (uint64_t)(N / 16)};
    const uint64_t st[2] = {256, (uint64_t)(K / BK) * P_BLOCK};
    const uint32_t box[3] = {256, 3, BN / 16};
    if (tma_encode(&tp, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, tiled, dims, st, box,
                   CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess)
      return CLEF_E_CUDA;
  }
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

clef_status lut6_tile_launch(const uint8_t* packed, int64_t n, int64_t k, uint8_t* tiled,
                             cudaStream_t stream) {
  const int64_t quads = n * (k / 4);
  if (quads == 0) return CLEF_OK;
  const int threads = 256;
  const int64_t blocks = std::min<int64_t>((quads + threads - 1) / threads, 65535LL * 8);
  lut::lut6_tile_kernel<<<(unsigned)blocks, threads, 0, stream>>>(packed, n, k, tiled);
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
