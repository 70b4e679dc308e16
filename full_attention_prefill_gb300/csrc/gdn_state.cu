// Gated DeltaNet: the sequential state pass on tcgen05, one CTA per (request, value head).
//
// The chunked form of the gated delta rule ("Clef-Flash-ANE-LUT6" model card, "Model
// architecture"; "clef-flash-LiteRT" README, "Provenance": chunks of 64 positions), for the chunk
// of rows t0 .. t0+63 entering with state S (value rows x key columns, fp32):
//     U   = U' - W S^T                          (per token: the new value minus the predicted one)
//     O   = diag(exp(g)) Q S^T / sqrt(128) + Aqk U
//     S  <- exp(g_C) S + U^T Kd                 (Kd = exp(g_C - g) K, the decayed keys)
// W, U', Kd, Aqk and exp(g) come from the parallel chunk phase.  Only U and S depend on the
// previous chunk, so the pass is a chain of two products per chunk; the O products hang off it.
// One launch walks a range of chunks (all of them, or one piece of a pieced scan), entering from
// s0 and leaving the state in s_out.
//
// Everything transposed so that the 128 value rows are the MMA's M dimension (TMEM lanes), and
// the products that share an A operand merged into one MMA chain:
//     [U^T | O1^T] [v, 128]  = S0h . [W ; Q]^T      M=128, N=128, K=128   A = S0h (TMEM)
//     [S | O2^T]   [v, 192] += U^T . [Kd | Aqk^T]   M=128, N=192, K=64    A = U^T (TMEM)
// with S0h the fp16 copy of S, U^T the fp16 U, O = exp(g)/sqrt(128) O1 + O2.  [W ; Q] is a
// K-major shared operand (W's 64 token rows, then Q's), [Kd | Aqk^T] an MN-major one (per token
// s: 128 key columns of Kd, then the 64 entries Aqk[., s]).  The second chain accumulates into S
// (scaled by exp(g_C) in place beforehand) and into O2 (zeroed after each drain).  The fp32
// state never leaves tensor memory.
//
// Warp roles (512 threads):
//   warp 0      TMA: per chunk part A = W, Q (two 64-column boxes each, 128-byte swizzle) and U'
//               (fp32 [64 tok][128 v], one bulk copy); part B = Kd (two boxes) and Aqk^T; two
//               stages of each.  W, U', Kd, Aqk^T are the chunk phase's per-(chunk, head) blocks.
//   warp 1      MMA issue (one thread) and tensor-memory allocation
//   warps 4-11  row threads, two per value row v = TMEM lane (warps 4-7 key columns / tokens
//               0..63 / 0..31, warps 8-11 the rest): per chunk copy S to S0h (fp16) and scale S
//               by exp(g_C) in place; then U = U' - acc, fp16, into TMEM
//   warps 12-15 output: O -> fp16, staged in shared memory and written by a TMA store (rows past
//               the request's end are clipped)
// Tensor memory (512 columns): S [0,128) | O2 [128,192), U acc [192,256) | O1 [256,320),
// S0h fp16 [320,384), U fp16 [384,416).
#include "common.cuh"
#include "gdn.cuh"

namespace clef {
namespace gdn {

constexpr int ST_THREADS = 512;
constexpr int BLK = C * 128;                   // one [64 rows][64 fp16] swizzled block: 8 KB
// part A (per stage): [W kb0 | Q kb0 | W kb1 | Q kb1], U'
constexpr int A_WQ = 0;                        // key block kb at kb * 2 BLK (W rows, then Q rows)
constexpr int A_U = 4 * BLK;                   // fp32 [64 tok][128 v]
constexpr int A_BYTES = A_U + C * D * 4;       // 64 KB
// part B (per stage): [Kd kb0 | Kd kb1 | Aqk^T]
constexpr int B_BYTES = 3 * BLK;               // 24 KB
constexpr int NSTAGE = 2;
constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + NSTAGE * A_BYTES;
constexpr int OFF_EPI = OFF_B + NSTAGE * B_BYTES;   // 4 x [64 tok][32 v] fp16
constexpr int EPI_BYTES = C * 32 * 2;
constexpr int OFF_BAR = OFF_EPI + 4 * EPI_BYTES;
constexpr int NUM_BARS = 4 * NSTAGE + 6;
constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int ST_SMEM = OFF_SLOT + 16 + 1024;  // slack to align the base to 1024
static_assert(ST_SMEM <= 232448, "shared memory per CTA");
static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzled blocks stay 1024-aligned");

constexpr uint32_t COL_S = 0;
constexpr uint32_t COL_O2 = 128;
constexpr uint32_t COL_UACC = 192;
constexpr uint32_t COL_O1 = 256;
constexpr uint32_t COL_S0H = 320;
constexpr uint32_t COL_UH = 384;

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

__global__ void __launch_bounds__(ST_THREADS, 1) gdn_state_tc_kernel(
    const __grid_constant__ CUtensorMap tW, const __grid_constant__ CUtensorMap tQ,
    const __grid_constant__ CUtensorMap tKd, const __grid_constant__ CUtensorMap tA,
    const __grid_constant__ CUtensorMap tO, const float* __restrict__ U1, const float* __restrict__ ef, const float* __restrict__ s0, float* __restrict__ s_out, int L,
    int nch, int c0, int ncl, unsigned* status) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x % HV;
  const int b = blockIdx.x / HV;
  // this launch walks chunks c0 .. c0 + ncl - 1 of each request (i counts them: stages and
  // barrier phases follow i, data addresses follow c)
  const float* efh = ef + ((int64_t)b * nch * HV + h) * C;   // chunk c at efh + c * HV * C

  const uint32_t bar_fa = sb + OFF_BAR;            // [2] part A landed
  const uint32_t bar_ea = bar_fa + 16;             // [2] part A consumed
  const uint32_t bar_fb = bar_ea + 16;             // [2] part B landed
  const uint32_t bar_eb = bar_fb + 16;             // [2] part B consumed
  const uint32_t bar_s0 = bar_eb + 16;             // S0h written and S scaled (row threads)
  const uint32_t bar_uh = bar_s0 + 8;              // U (fp16) written (row threads)
  const uint32_t bar_u = bar_uh + 8;               // [U acc | O1] complete
  const uint32_t bar_s = bar_u + 8;                // [S | O2] complete
  const uint32_t bar_oe = bar_s + 8;               // O1, O2 drained and O2 zeroed
  const uint32_t bar_fin = bar_oe + 8;             // every MMA issued has completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_SLOT);

  if (threadIdx.x == 0) {
    for (int i = 0; i < NSTAGE; ++i) {
      mbar_init(bar_fa + 8 * i, 1);
      mbar_init(bar_ea + 8 * i, 1 + 8);            // first chain's commit + the 8 row warps
      mbar_init(bar_fb + 8 * i, 1);
      mbar_init(bar_eb + 8 * i, 1);                // second chain's commit
    }
    mbar_init(bar_s0, 8);
    mbar_init(bar_uh, 8);
    mbar_init(bar_u, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_oe, 4);
    mbar_init(bar_fin, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tW);
    tma_prefetch_desc(&tQ);
    tma_prefetch_desc(&tKd);
    tma_prefetch_desc(&tA);
    tma_prefetch_desc(&tO);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();   // the barriers and tensor memory are set up; now the inputs

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued_a = 0, issued_b = 0;
      for (int i = 0; i < ncl; ++i) {
        const int c = c0 + i;
        const int st = i & 1;
        const int t0 = c * C;
        if (i >= NSTAGE &&
            !mbar_wait(bar_ea + 8 * st, ((i - NSTAGE) >> 1) & 1, status, DEV_TIMEOUT_TMA))
          break;
        {
          const uint32_t base = sb + OFF_A + st * A_BYTES;
          const uint32_t fb = bar_fa + 8 * st;
          const int64_t blk = ((int64_t)b * nch + c) * HV + h;   // the chunk phase's block
          mbar_arrive_expect_tx(fb, A_BYTES);
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
            tma_load_2d(base + A_WQ + kb * 2 * BLK, &tW, fb, kb * 64, (int)(blk * C));
            tma_load_4d(base + A_WQ + kb * 2 * BLK + BLK, &tQ, fb, kb * 64, h >> 1, t0, b);
          }
          bulk_copy_g2s(base + A_U, U1 + blk * C * D, C * D * 4, fb);
          issued_a = i + 1;
        }
        if (i >= NSTAGE &&
            !mbar_wait(bar_eb + 8 * st, ((i - NSTAGE) >> 1) & 1, status, DEV_TIMEOUT_TMA))
          break;
        {
          const uint32_t base = sb + OFF_B + st * B_BYTES;
          const uint32_t fb = bar_fb + 8 * st;
          const int64_t blk = ((int64_t)b * nch + c) * HV + h;
          mbar_arrive_expect_tx(fb, B_BYTES);
          tma_load_2d(base, &tKd, fb, 0, (int)(blk * C));
          tma_load_2d(base + BLK, &tKd, fb, 64, (int)(blk * C));
          tma_load_2d(base + 2 * BLK, &tA, fb, 0, (int)(blk * C));
          issued_b = i + 1;
        }
      }
      // copies still in flight land before the CTA may exit (no later phase of these barriers
      // can complete, so the parity tests are unambiguous)
      for (int c = issued_a > NSTAGE ? issued_a - NSTAGE : 0; c < issued_a; ++c)
        mbar_wait(bar_fa + 8 * (c & 1), (c >> 1) & 1, status, DEV_TIMEOUT_TMA);
      for (int c = issued_b > NSTAGE ? issued_b - NSTAGE : 0; c < issued_b; ++c)
        mbar_wait(bar_fb + 8 * (c & 1), (c >> 1) & 1, status, DEV_TIMEOUT_TMA);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t id_1 = idesc_f16_f32(128, 128);          // [W ; Q] K-major
      constexpr uint32_t id_2 = idesc_f16_f32(128, 192, 0, 1);    // [Kd | Aqk^T] MN-major
      bool any = false;
      for (int i = 0; i < ncl; ++i) {
        const int st = i & 1;
        const uint32_t ph = (uint32_t)i & 1;
        // one descriptor per operand and chunk; the K slices are constant offsets of its
        // address field, formed before the waits so that the MMAs issue as soon as they pass
        const uint64_t ad = sdesc_k_sw128(sb + OFF_A + st * A_BYTES + A_WQ);
        const uint64_t bd = sdesc_mn_sw128(sb + OFF_B + st * B_BYTES, BLK, 1024);
        // [U^T | O1^T] = S0h . [W ; Q]^T, once the previous chunk's O has been drained
        if (!mbar_wait(bar_fa + 8 * st, (i >> 1) & 1, status, DEV_TIMEOUT_MMA) ||
            !mbar_wait(bar_s0, ph, status, DEV_TIMEOUT_MMA) ||
            (i >= 1 && !mbar_wait(bar_oe, (i - 1) & 1, status, DEV_TIMEOUT_MMA)))
          break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_f16_ts(tmem + COL_UACC, tmem + COL_S0H + kk * 8,
                        ad + (uint64_t)(((kk >> 2) * 2 * BLK + (kk & 3) * 32) >> 4), id_1, kk != 0);
        tc_commit(bar_u);
        tc_commit(bar_ea + 8 * st);   // W, Q no longer read (the row threads add theirs for U')
        any = true;
        // [S | O2^T] += U^T . [Kd | Aqk^T]
        if (!mbar_wait(bar_fb + 8 * st, (i >> 1) & 1, status, DEV_TIMEOUT_MMA) ||
            !mbar_wait(bar_uh, ph, status, DEV_TIMEOUT_MMA))
          break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < C / 16; ++kk)
          tc_mma_f16_ts(tmem + COL_S, tmem + COL_UH + kk * 8, bd + (uint64_t)((kk * 16 * 128) >> 4),
                        id_2, 1);
        tc_commit(bar_s);
        tc_commit(bar_eb + 8 * st);
      }
      // tensor memory is freed only after every MMA issued here has completed
      if (any) {
        tc_commit(bar_fin);
        mbar_wait(bar_fin, 0, status, DEV_TIMEOUT_MMA);
      }
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------------ row threads
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;                        // which half of the columns
    const int v = quarter * 32 + lane;                       // value row = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    // entering state: s0 row v (this thread's 64 key columns), or zero; O2 starts at zero
#pragma unroll 1
    for (int cb = 2 * half; cb < 2 * half + 2; ++cb) {
      uint32_t r[32];
      if (s0) {
        const float4* src =
            reinterpret_cast<const float4*>(s0 + (((int64_t)b * HV + h) * D + v) * D + cb * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 x = __ldg(src + i);
          r[4 * i] = __float_as_uint(x.x);
          r[4 * i + 1] = __float_as_uint(x.y);
          r[4 * i + 2] = __float_as_uint(x.z);
          r[4 * i + 3] = __float_as_uint(x.w);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) r[i] = 0u;
      }
      tmem_st_32x32b_x32(tl + COL_S + cb * 32, r);
    }
    {
      uint32_t z[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) z[i] = 0u;
      tmem_st_32x32b_x32(tl + COL_O2 + half * 32, z);
    }
    tc_wait_st();
    float eC_next = __ldg(efh + (int64_t)c0 * HV * C + (C - 1));
    bool ok = true;
    for (int i = 0; i < ncl; ++i) {
      const int c = c0 + i;
      const int st = i & 1;
      // exp(g_C) of this chunk; the next chunk's is fetched now, its latency hidden by the chunk
      const float eC = eC_next;
      if (i + 1 < ncl) eC_next = __ldg(efh + (int64_t)(c + 1) * HV * C + (C - 1));
      ok = ok && mbar_wait(bar_fa + 8 * st, (i >> 1) & 1, status, DEV_TIMEOUT_EPILOGUE);
      ok = ok && (i == 0 || mbar_wait(bar_s, (i - 1) & 1, status, DEV_TIMEOUT_EPILOGUE));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // S0h = fp16(S); S <- exp(g_C) S   (this thread: key columns 64 half .. 64 half + 63)
      {
        uint32_t r0[32], r1[32], hh[32];
        tmem_ld_32x32b_x32(tl + COL_S + half * 64, r0);
        tmem_ld_32x32b_x32(tl + COL_S + half * 64 + 32, r1);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          hh[i] = pack_half2(u2f(r0[2 * i]), u2f(r0[2 * i + 1]));
          hh[16 + i] = pack_half2(u2f(r1[2 * i]), u2f(r1[2 * i + 1]));
        }
        tmem_st_32x32b_x32(tl + COL_S0H + half * 32, hh);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          r0[i] = __float_as_uint(u2f(r0[i]) * eC);
          r1[i] = __float_as_uint(u2f(r1[i]) * eC);
        }
        tmem_st_32x32b_x32(tl + COL_S + half * 64, r0);
        tmem_st_32x32b_x32(tl + COL_S + half * 64 + 32, r1);
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_s0);
      // U' of this row for tokens 32 half .. 32 half + 31, read while the MMAs run
      const float* us = reinterpret_cast<const float*>(smem + OFF_A + st * A_BYTES + A_U) +
                        (half * 32) * D + v;
      float up[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) up[j] = us[j * D];
      ok = __all_sync(0xffffffffu, mbar_wait(bar_u, (uint32_t)i & 1, status, DEV_TIMEOUT_EPILOGUE));
      if (!ok) break;
      tc_fence_after();
      // U = U' - W S0^T (rows past the request's end have W = U' = 0 from the zero-filled
      // loads, hence U = 0)
      {
        uint32_t a[32], uh[16];
        tmem_ld_32x32b_x32(tl + COL_UACC + half * 32, a);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          uh[i] = pack_half2(up[2 * i] - u2f(a[2 * i]), up[2 * i + 1] - u2f(a[2 * i + 1]));
        tmem_st_32x32b_x16(tl + COL_UH + half * 16, uh);
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_uh);
        mbar_arrive(bar_ea + 8 * st);   // done with this stage's U'
      }
    }
    if (ok && s_out) {
      // the state after the last chunk
      if (mbar_wait(bar_s, (ncl - 1) & 1, status, DEV_TIMEOUT_EPILOGUE)) {
        tc_fence_after();
        float* dst = s_out + (((int64_t)b * HV + h) * D + v) * D;
#pragma unroll 1
        for (int cb = 2 * half; cb < 2 * half + 2; ++cb) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(tl + COL_S + cb * 32, r);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 8; ++i)
            reinterpret_cast<float4*>(dst + cb * 32)[i] =
                make_float4(u2f(r[4 * i]), u2f(r[4 * i + 1]), u2f(r[4 * i + 2]), u2f(r[4 * i + 3]));
        }
      }
    }
  } else if (warp >= 12) {
    // ------------------------------------------------------------------ output
    const int quarter = warp & 3;
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    const float inv_sqrt_d = 0.08838834764831845f;
    // staging [64 tok][32 v] fp16 for this warp's 32 value rows
    const uint32_t stg = sb + OFF_EPI + quarter * EPI_BYTES;
    // exp(g) of the chunk's rows: lane j holds rows j and 32 + j (fetched one chunk ahead)
    const float* efc = efh + (int64_t)c0 * HV * C;
    float fa_next = __ldg(efc + lane), fb_next = __ldg(efc + 32 + lane);
    bool ok = true;
    for (int i = 0; i < ncl; ++i) {
      const int c = c0 + i;
      const float fa = fa_next * inv_sqrt_d, fb = fb_next * inv_sqrt_d;
      if (i + 1 < ncl) {
        fa_next = __ldg(efh + (int64_t)(c + 1) * HV * C + lane);
        fb_next = __ldg(efh + (int64_t)(c + 1) * HV * C + 32 + lane);
      }
      // O1 is complete with [U | O1]: read and scale it while U is converted and S updated
      ok = __all_sync(0xffffffffu, mbar_wait(bar_u, (uint32_t)i & 1, status, DEV_TIMEOUT_EPILOGUE));
      if (!ok) break;
      tc_fence_after();
      float fo[64];
      {
        uint32_t o1[32];
        tmem_ld_32x32b_x32(tl + COL_O1, o1);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) fo[j] = __shfl_sync(0xffffffffu, fa, j) * u2f(o1[j]);
        tmem_ld_32x32b_x32(tl + COL_O1 + 32, o1);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) fo[32 + j] = __shfl_sync(0xffffffffu, fb, j) * u2f(o1[j]);
      }
      // O2 with [S | O2]; O = exp(g)/sqrt(128) O1 + O2, kept as fp16 pairs
      ok = __all_sync(0xffffffffu, mbar_wait(bar_s, (uint32_t)i & 1, status, DEV_TIMEOUT_EPILOGUE));
      if (!ok) break;
      tc_fence_after();
      uint32_t y[32];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t o2[32];
        tmem_ld_32x32b_x32(tl + COL_O2 + hf * 32, o2);
        tc_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j)
          y[hf * 16 + j] = pack_half2(fo[hf * 32 + 2 * j] + u2f(o2[2 * j]),
                                      fo[hf * 32 + 2 * j + 1] + u2f(o2[2 * j + 1]));
      }
      {
        // O2 accumulates from zero in the next chunk
        uint32_t z[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) z[i] = 0u;
        tmem_st_32x32b_x32(tl + COL_O2, z);
        tmem_st_32x32b_x32(tl + COL_O2 + 32, z);
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar_oe);
        bulk_wait_read0();   // the previous chunk's store has finished reading the staging
      }
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(stg + ((2 * j) * 32 + lane) * 2),
                     "h"((unsigned short)(y[j] & 0xffffu)) : "memory");
        asm volatile("st.shared.b16 [%0], %1;" ::"r"(stg + ((2 * j + 1) * 32 + lane) * 2),
                     "h"((unsigned short)(y[j] >> 16)) : "memory");
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_store_4d(&tO, stg, quarter * 32, h, c * C, b);
        bulk_commit_group();
      }
    }
    if (lane == 0) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace gdn

clef_status gdn_state_launch(const __half* q, const __half* Kd, const __half* W, const float* U1,
                             const __half* Aqk, const float* ef, const float* s0, float* s_out,
                             __half* out, int64_t ldo, int64_t B, int64_t L, cudaStream_t stream,
                             int64_t c0, int64_t ncl) {
  using namespace gdn;
  if (B == 0 || L == 0) return CLEF_OK;
  if ((ldo % 8) != 0 || (reinterpret_cast<uintptr_t>(out) & 15) != 0) {
    set_error("GDN scan output: row stride must be a multiple of 8 and the base 16-byte aligned");
    return CLEF_E_ALIGN;
  }
  const int64_t nch = (L + C - 1) / C;
  if (ncl < 0) ncl = nch - c0;
  if (c0 < 0 || ncl < 1 || c0 + ncl > nch) return CLEF_E_INVALID;
  static std::atomic<uint64_t> attr{0};
  CLEF_CUDA_CHECK(smem_opt_in((const void*)gdn_state_tc_kernel, ST_SMEM, &attr));
  CUtensorMap tW, tQ, tKd, tA, tO;
  {
    // the chunk phase's outputs: one block of 64 rows per (chunk, head)
    const uint64_t rows = (uint64_t)(B * nch * HV * C);
    if (tma_encode_2d(&tW, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, W, (uint64_t)D, rows, (uint64_t)D * 2,
                      64, (uint32_t)C, CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess ||
        tma_encode_2d(&tKd, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Kd, (uint64_t)D, rows,
                      (uint64_t)D * 2, 64, (uint32_t)C, CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess ||
        tma_encode_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, Aqk, (uint64_t)C, rows,
                      (uint64_t)C * 2, (uint32_t)C, (uint32_t)C,
                      CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess)
      return CLEF_E_CUDA;
    const uint64_t dims[4] = {(uint64_t)D, (uint64_t)HV, (uint64_t)L, (uint64_t)B};
    const uint32_t box[4] = {64, 1, (uint32_t)C, 1};
    const uint64_t dq[4] = {(uint64_t)D, (uint64_t)HK, (uint64_t)L, (uint64_t)B};
    const uint64_t sq[3] = {(uint64_t)D * 2, (uint64_t)HK * D * 2, (uint64_t)L * HK * D * 2};
    if (tma_encode(&tQ, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, q, dq, sq, box,
                   CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess)
      return CLEF_E_CUDA;
    const uint64_t so[3] = {(uint64_t)D * 2, (uint64_t)ldo * 2, (uint64_t)L * ldo * 2};
    const uint32_t bo[4] = {32, 1, (uint32_t)C, 1};
    if (tma_encode(&tO, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, out, dims, so, bo,
                   CU_TENSOR_MAP_SWIZZLE_NONE) != cudaSuccess)
      return CLEF_E_CUDA;
  }
  const double Cd = C, Dd = D, chunks = (double)B * ncl * HV;
  TraceScope ts(stream, "gdn_state_pass", chunks * (6.0 * Cd * Dd * Dd + 2.0 * Cd * Cd * Dd),
                // per (chunk, value head): W, Kd, U', out rows (2 + 2 + 4 + 2 bytes x D), its
                // share of the q rows (a key head serves two value heads), Aqk^T
                chunks * Cd * (Dd * (2 + 2 + 4 + 2) + Dd * 2.0 * HK / HV + Cd * 2));
  CLEF_CUDA_CHECK(launch_pdl(gdn_state_tc_kernel, dim3((unsigned)(B * HV)), dim3(ST_THREADS), ST_SMEM, stream,
       tW, tQ, tKd, tA, tO, U1, ef, s0, s_out, (int)L, (int)nch, (int)c0, (int)ncl,
       status_word_ptr()));
  return CLEF_OK;
}

}  // namespace clef
