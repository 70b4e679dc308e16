// LUT-6 weights: host pack/unpack, a dense dequant kernel (parity aid) and the LUT-6 GEMM.
//
// Format ("Clef-Flash-ANE-LUT6" model card, sections "Weight precision" and "LUT-6 text
// weights"): a 6-bit index per weight, an fp16 table of 64 values for each block of 16 output
// channels, 4 indices to 3 bytes as one little-endian (LSB-first) bit stream, rows of W in
// order, k fastest.
//
// GEMM design (sm_103a): Y[m, n] = sum_k X[m, k] * T[n/16][idx[n, k]], computed as the
// transposed product D[n, m] = W X^T so that the weights are the MMA's A operand, held in tensor
// memory, and never pass through shared memory.  A persistent kernel (one CTA per SM) walks
// 128 (output channels) x 256 (tokens) tiles, K in blocks of 64 ("steps"); the step count runs
// on across tiles, so every ring below keeps flowing at tile boundaries:
//   * warp 0 loads X (256 tokens x 64, 128-byte swizzle) into a 5-slot ring;
//   * warp 2 loads the tile's packed indices (8 blocks of 768 bytes per step, tiled layout, see
//     clef_lut6_tile) into an 8-slot ring, and its 8 tables (1 KB) into one of two slots;
//   * warps 4..19 dequantise into an 8-slot ring of tensor-memory A stages (32 columns each):
//     each warp owns one 16-row table group on every other step and writes its 16 x 64 weights
//     with one tcgen05.st.16x256b.x4; all lookups of a warp hit one 64-entry table (128 bytes,
//     one entry pair per bank) and never conflict; a lane's 32 indices are 24 contiguous bytes
//     and index*2 is cut into the table address with one shift and one logic op;
//   * warp 1 issues tcgen05.mma (M=128 channels from tensor memory, N=256 tokens from shared
//     memory, K=16) into a 128 x 256 fp32 accumulator (tensor-memory columns 0..255);
//   * the same 16 warps drain the accumulator of tile i once they have dequantised the first
//     steps of tile i+1: each loads its 32 lanes x 64 columns into registers and releases the
//     accumulator, so the MMAs of tile i+1 start on stages already prepared, then writes Y from
//     registers (fp16 or fp32 store, fp32 residual add, or SwiGLU of a gate/up tile interleaved
//     in 16-row blocks: a gate row and its up row sit 16 lanes apart in one warp and meet
//     through one shuffle).
// Long prefills take lut6_gemm_wide_kernel (below): 128 x 384 tiles, two 192-column
// accumulators and four A stages filling tensor memory, so each weight is dequantised once per
// 384 tokens.
// The tensor pipe queues only about two MMAs ahead of the issuing thread, so time that thread
// spends between MMAs shows up as idle tensor cycles: measured on this part, a loop of 4 MMAs
// per step runs at the full 8192 flop/clk with no wait, ~91% with one mbarrier wait before the
// MMAs of each step, and ~70% with two waits or with the wait placed between the MMAs.  The
// protocol therefore gives the MMA thread exactly one wait per step, ahead of its 4 MMAs (a
// "ready" barrier that counts the X bytes and the dequant warps' arrivals), and one commit per
// step (an "empty" barrier that frees the step's X slot, A stage and index slot together).  Every wait is bounded: on a timeout the kernel records a code in the device
// status word, lets its own copies in flight land and frees its tensor memory.  The dense
// weight never reaches global memory.
#include <stdarg.h>
#include <stdio.h>

#include "common.cuh"
#include "lut6.cuh"

namespace clef {
namespace lut {

constexpr int BN = 128;                       // output channels per tile: MMA M (A operand)
constexpr int BT = 256;                       // tokens per tile: MMA N (B operand)
constexpr int BK = 64;                        // one step
constexpr int XS = 5;                         // X ring stages
constexpr int AS = 8;                         // packed-index ring = tensor-memory A ring stages
constexpr int X_BYTES = BT * BK * 2;          // 32 KB
constexpr int P_BLOCK = 768;                  // packed bytes of one 16-row group per step
constexpr int P_BYTES = (BN / 16) * P_BLOCK;  // 6 KB
constexpr int TBL_BYTES = (BN / 16) * 64 * 2; // 1 KB: the 8 tables of a tile's rows
constexpr int NUM_DQ_WARPS = 16;              // two per 16-row group (even / odd steps)
constexpr int NUM_THREADS = 32 * (4 + NUM_DQ_WARPS);
constexpr int TMEM_COLS = 512;
constexpr uint32_t A_COL = BT;                // A stages: 32 columns each from column 256

constexpr int OFF_X = 0;
constexpr int OFF_P = OFF_X + XS * X_BYTES;
constexpr int OFF_T = OFF_P + AS * P_BYTES;
constexpr int OFF_BAR = OFF_T + 2 * TBL_BYTES;
constexpr int NUM_BARS = 3 * AS + 4 + 3;
constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_USED = OFF_SLOT + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(A_COL + AS * 32 <= TMEM_COLS, "tensor memory budget");
static_assert(CLEF_SWIGLU_BLOCK == 16 && BN % (2 * CLEF_SWIGLU_BLOCK) == 0,
              "a gate row and its up row are 16 lanes apart in one warp's 32 lanes");

// The wide tile (long prefills): 128 channels x 384 tokens, two N = 192 accumulators (tensor
// memory columns 0..383, token t of the tile in column t) and four A stages (columns 384..511).
constexpr int WH = 192;                           // tokens per half (one MMA's N)
constexpr int WT = 2 * WH;                        // tokens per wide tile
constexpr int W_AS = 4;                           // ring: X slot = A stage = index slot per step
constexpr int W_H_BYTES = WH * BK * 2;            // 24 KB: one half of a step's X
constexpr int W_X_BYTES = 2 * W_H_BYTES;          // 48 KB
constexpr uint32_t W_A_COL = WT;                  // A stages: 32 columns each from column 384
constexpr int W_OFF_X = 0;
constexpr int W_OFF_P = W_OFF_X + W_AS * W_X_BYTES;
constexpr int W_OFF_T = W_OFF_P + W_AS * P_BYTES;
constexpr int W_OFF_BAR = W_OFF_T + 2 * TBL_BYTES;
constexpr int W_NUM_BARS = 3 * W_AS + 4 + 3;
constexpr int W_OFF_SLOT = W_OFF_BAR + W_NUM_BARS * 8;
constexpr int W_SMEM_BYTES = W_OFF_SLOT + 16 + 1024;  // slack to align the base to 1024
static_assert(W_SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(W_H_BYTES % 1024 == 0, "swizzle atoms stay 1024-aligned");
static_assert(W_A_COL + W_AS * 32 <= TMEM_COLS, "tensor memory budget");

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
__device__ __forceinline__ void red_add_f32(float* p, float v) {
  asm volatile("red.global.add.f32 [%0], %1;" ::"l"(p), "f"(v) : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
      : "memory");
}

// Tile t of the persistent walk -> (first output channel n0, first token m0).  Tiles go in
// groups of group_m token tiles: inside a group the token tile varies fastest, so the CTAs
// running at one time share a few weight tiles and a few X tiles, which stay in L2.  The X rows
// of a group stay in L2 while all channel tiles pass over them; the packed weights are read
// again from DRAM for every group.
__device__ __forceinline__ void tile_coord(int t, int n_tiles, int m_tiles, int group_m, int bt,
                                           int& n0, int& m0) {
  const int per_group = group_m * n_tiles;
  const int grp = t / per_group;
  const int first_m = grp * group_m;
  const int gm = min(group_m, m_tiles - first_m);
  const int local = t - grp * per_group;
  m0 = (first_m + local % gm) * bt;
  n0 = (local / gm) * BN;
}

// Y for nt = 64 (or 32) tokens (tok0 ..) of the 32 channels n0e + 32 quarter + lane held by one
// warp (this lane's channel col): r0 holds tokens tok0 + 0..31, r1 tok0 + 32..63 (fp32; unused
// for nt = 32), written in `mode`.
__device__ __forceinline__ void store_y_block(int mode, void* __restrict__ y, int64_t ldy, int M,
                                              int N, int n0e, int col, int tok0, int quarter,
                                              int lane, int kpart, const uint32_t (&r0)[32],
                                              const uint32_t (&r1)[32], int nt = 64) {
  if (mode == EPI_SWIGLU_F16) {
    // lanes 0..15: gate rows, lanes 16..31: the up rows of the same channels; of the block's
    // tokens the gate lane writes the first half, the up lane the second (64 tokens: r0 and r1;
    // 32 tokens: r0 alone, 16 each)
    const bool up = lane >= 16;
    const int oc = n0e / 2 + quarter * 16 + (lane & 15);
    __half* out = reinterpret_cast<__half*>(y);
    const bool oc_ok = oc < N / 2;
    if (nt == 64) {
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const uint32_t send = up ? r0[i] : r1[i];
        const float other = __uint_as_float(__shfl_xor_sync(0xffffffffu, send, 16));
        const float gate = up ? other : __uint_as_float(r0[i]);
        const float upv = up ? __uint_as_float(r1[i]) : other;
        const int tok = tok0 + (up ? 32 : 0) + i;
        if (oc_ok && tok < M) out[(int64_t)tok * ldy + oc] = __float2half_rn(silu_f(gate) * upv);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t send = up ? r0[i] : r0[16 + i];
        const float other = __uint_as_float(__shfl_xor_sync(0xffffffffu, send, 16));
        const float gate = up ? other : __uint_as_float(r0[i]);
        const float upv = up ? __uint_as_float(r0[16 + i]) : other;
        const int tok = tok0 + (up ? 16 : 0) + i;
        if (oc_ok && tok < M) out[(int64_t)tok * ldy + oc] = __float2half_rn(silu_f(gate) * upv);
      }
    }
  } else if (col < N) {
    if (mode == EPI_F16) {
      __half* out = reinterpret_cast<__half*>(y) + col;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (tok0 + i < M) out[(int64_t)(tok0 + i) * ldy] = __float2half_rn(__uint_as_float(r0[i]));
        if (nt == 64 && tok0 + 32 + i < M)
          out[(int64_t)(tok0 + 32 + i) * ldy] = __float2half_rn(__uint_as_float(r1[i]));
      }
    } else if (mode == EPI_F32 || mode == EPI_PART_F32) {
      // a k-part of a split residual add goes to its own slice [kpart][M][ldy]
      float* out = reinterpret_cast<float*>(y) + col +
                   (mode == EPI_PART_F32 ? (int64_t)kpart * M * ldy : 0);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (tok0 + i < M) out[(int64_t)(tok0 + i) * ldy] = __uint_as_float(r0[i]);
        if (nt == 64 && tok0 + 32 + i < M) out[(int64_t)(tok0 + 32 + i) * ldy] = __uint_as_float(r1[i]);
      }
    } else {
      // residual add, done by L2; no load latency on this path.  Without a K split each
      // element receives exactly one add per launch (the same as load + add + store); with
      // one, the parts' adds land in any order, so such launches repeat only to fp32
      // rounding
      float* out = reinterpret_cast<float*>(y) + col;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (tok0 + i < M) red_add_f32(out + (int64_t)(tok0 + i) * ldy, __uint_as_float(r0[i]));
        if (nt == 64 && tok0 + 32 + i < M)
          red_add_f32(out + (int64_t)(tok0 + 32 + i) * ldy, __uint_as_float(r1[i]));
      }
    }
  }
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    lut6_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                     const __grid_constant__ CUtensorMap tmap_p, const __half* __restrict__ lut,
                     void* __restrict__ y, int64_t ldy, int M, int N, int K, int mode,
                     int ksplit, int group_m, unsigned* status) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int num_kb = K / BK;
  const int n_tiles = (N + BN - 1) / BN;
  const int m_tiles = (M + BT - 1) / BT;
  const int num_tiles = n_tiles * m_tiles;
  // work units: (tile, k part); with ksplit > 1 (residual-add mode only) each unit covers
  // num_kb / ksplit steps and adds its partial sum into Y
  const int nkb = num_kb / ksplit;
  const int num_units = num_tiles * ksplit;
  // the accumulator of tile i is drained after the first `lead` steps of tile i+1 have been
  // dequantised, so the MMAs of tile i+1 start as soon as it is free
  const int lead = min(AS - 1, nkb - 1);

  // One "ready" and one "empty" barrier per step (ring of AS): step g may run its MMAs once its
  // X tile has landed and its A stage is written (ready[g % AS]: the X bytes plus one arrival
  // per dequantising warp); the MMA thread's single commit per step (empty[g % AS]) frees the X
  // slot, the A stage and the packed-index slot of that step at once.  The MMA thread thus waits
  // on one barrier per step, and does so while the previous step's last MMAs still run.
  const uint32_t bar_ready = sb + OFF_BAR;             // [AS]
  const uint32_t bar_empty = bar_ready + 8 * AS;       // [AS]
  const uint32_t bar_pfull = bar_empty + 8 * AS;       // [AS] packed indices landed
  const uint32_t bar_tfull = bar_pfull + 8 * AS;       // [2] tables landed
  const uint32_t bar_tempty = bar_tfull + 16;          // [2] tables no longer read
  const uint32_t bar_accf = bar_tempty + 16;           // accumulator complete
  const uint32_t bar_acce = bar_accf + 8;              // accumulator drained
  const uint32_t bar_fin = bar_acce + 8;               // the MMA thread's last MMAs completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_SLOT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < AS; ++s) {
      mbar_init(bar_ready + 8 * s, 1 + NUM_DQ_WARPS / 2);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_pfull + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_tfull + 8 * s, 1);
      mbar_init(bar_tempty + 8 * s, NUM_DQ_WARPS);
    }
    mbar_init(bar_accf, 1);
    mbar_init(bar_acce, NUM_DQ_WARPS);
    mbar_init(bar_fin, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_p);
  }
  // table slots start at zero: rows past N (a partial last tile) then see finite entries
  for (int i = threadIdx.x; i < 2 * TBL_BYTES / 4; i += NUM_THREADS)
    reinterpret_cast<uint32_t*>(smem + OFF_T)[i] = 0u;
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();   // the barriers and tensor memory are set up; now the inputs
  const int first = blockIdx.x;
  const int stride = gridDim.x;

  if (warp == 0) {
    // ---------------------------------------------------------------- X loads
    if (lane == 0) {
      int64_t g = 0;
      bool ok = true;
      for (int u = first; u < num_units && ok; u += stride) {
        int n0, m0;
        tile_coord(u % num_tiles, n_tiles, m_tiles, group_m, BT, n0, m0);
        const int kb0 = (u / num_tiles) * nkb;
        for (int kb = kb0; kb < kb0 + nkb; ++kb, ++g) {
          // X slot g % XS was last read by step g - XS
          const int64_t f = g - XS;
          if (f >= 0 && !mbar_wait(bar_empty + 8 * (int)(f % AS), (uint32_t)(f / AS) & 1, status,
                                   DEV_TIMEOUT_TMA)) {
            ok = false;
            break;
          }
          const uint32_t rb = bar_ready + 8 * (int)(g % AS);
          mbar_arrive_expect_tx(rb, X_BYTES);
          tma_load_2d(sb + OFF_X + (int)(g % XS) * X_BYTES, &tmap_x, rb, kb * BK, m0);
        }
      }
      // copies still in flight land before the CTA may exit (a phase that already completed
      // passes at once)
      for (int64_t h = g > XS ? g - XS : 0; h < g; ++h)
        mbar_wait(bar_ready + 8 * (int)(h % AS), (uint32_t)(h / AS) & 1, status, DEV_TIMEOUT_TMA);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- tables + packed indices
    if (lane == 0) {
      int64_t g = 0;
      int it = 0;
      bool ok = true;
      for (int u = first; u < num_units && ok; u += stride, ++it) {
        int n0, m0;
        tile_coord(u % num_tiles, n_tiles, m_tiles, group_m, BT, n0, m0);
        const int kb0 = (u / num_tiles) * nkb;
        const int ts = it & 1;
        if (it >= 2 && !mbar_wait(bar_tempty + 8 * ts, ((uint32_t)(it >> 1) & 1) ^ 1, status,
                                  DEV_TIMEOUT_TMA)) {
          ok = false;
          break;
        }
        const int groups = min(BN / 16, N / 16 - n0 / 16);
        mbar_arrive_expect_tx(bar_tfull + 8 * ts, groups * 128);
        bulk_load(sb + OFF_T + ts * TBL_BYTES, lut + (size_t)(n0 / 16) * 64, groups * 128,
                  bar_tfull + 8 * ts);
        for (int kb = kb0; kb < kb0 + nkb; ++kb, ++g) {
          // slot s (indices and A stage) was last used by step g - AS
          const int s = (int)(g % AS);
          const uint32_t ph = (uint32_t)(g / AS) & 1;
          if (g >= AS && !mbar_wait(bar_empty + 8 * s, ph ^ 1, status, DEV_TIMEOUT_TMA)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_pfull + 8 * s, P_BYTES);
          // the 8 groups' 768-byte blocks of k-block kb: box {256 B, 3, 8 groups}
          tma_load_3d(sb + OFF_P + s * P_BYTES, &tmap_p, bar_pfull + 8 * s, 0, 3 * kb, n0 / 16);
        }
      }
      for (int64_t h = g > AS ? g - AS : 0; h < g; ++h)
        mbar_wait(bar_pfull + 8 * (int)(h % AS), (uint32_t)(h / AS) & 1, status, DEV_TIMEOUT_TMA);
      for (int u = it > 2 ? it - 2 : 0; u < it; ++u)
        mbar_wait(bar_tfull + 8 * (u & 1), (uint32_t)(u >> 1) & 1, status, DEV_TIMEOUT_TMA);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BN, BT);
      int sx = 0, sa = 0;      // X slot and ready/empty slot of the current step
      uint32_t ph = 0;         // phase parity of ready[sa]
      int it = 0;
      bool ok = true;
      for (int u = first; u < num_units && ok; u += stride, ++it) {
        if (it >= 1 && !mbar_wait(bar_acce, (uint32_t)(it - 1) & 1, status, DEV_TIMEOUT_MMA)) {
          ok = false;
          break;
        }
        for (int kb = 0; kb < nkb; ++kb) {
          // operands of this step, formed before the wait so that the MMAs issue as soon as it
          // passes (the four K slices are constant offsets of the descriptor's address field)
          const uint32_t a = tmem + A_COL + sa * 32;
          const uint64_t bd = sdesc_k_sw128(sb + OFF_X + sx * X_BYTES);
          if (!mbar_wait(bar_ready + 8 * sa, ph, status, DEV_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          tc_mma_f16_ts(tmem, a, bd, idesc, kb != 0);
          tc_mma_f16_ts(tmem, a + 8, bd + 2, idesc, 1);
          tc_mma_f16_ts(tmem, a + 16, bd + 4, idesc, 1);
          tc_mma_f16_ts(tmem, a + 24, bd + 6, idesc, 1);
          tc_commit(bar_empty + 8 * sa);
          sx = sx + 1 == XS ? 0 : sx + 1;
          if (++sa == AS) {
            sa = 0;
            ph ^= 1;
          }
        }
        if (ok) tc_commit(bar_accf);
      }
      // tensor memory is freed below only after every MMA issued here has completed
      tc_commit(bar_fin);
      mbar_wait(bar_fin, 0, status, DEV_TIMEOUT_MMA);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- dequant + epilogue
    const int dq = warp - 4;                           // 0..15
    const int quarter = warp & 3;                      // TMEM lanes 32*quarter .. +31
    const int grp = 2 * quarter + ((dq >> 2) & 1);     // 16-row group dequantised by this warp
    const int par = dq >> 3;                           // steps g with g % 2 == par
    const int ecol = (dq >> 2) * 64;                   // epilogue: token columns ecol .. +63
    const uint32_t tl = tmem + ((uint32_t)(grp * 16) << 16) + A_COL;
    const uint32_t tacc = tmem + ((uint32_t)(quarter * 32) << 16) + ecol;

    // Drain this warp's 32 lanes x 64 columns of the accumulator of the tile at (n0e, m0e),
    // release it, then write Y from registers.
    auto epilogue = [&](int n0e, int m0e, int ite, int kpart) -> bool {
      const int tok0 = m0e + ecol;
      const int col = n0e + quarter * 32 + lane;
      if (!mbar_wait(bar_accf, (uint32_t)ite & 1, status, DEV_TIMEOUT_EPILOGUE)) return false;
      tc_fence_after();
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(tacc, r0);
      tmem_ld_32x32b_x32(tacc + 32, r1);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acce);
      store_y_block(mode, y, ldy, M, N, n0e, col, tok0, quarter, lane, kpart, r0, r1);
      return true;
    };

    int64_t g = 0;
    int it = 0;
    bool ok = true;
    int pn0 = -1, pm0 = 0, pkp = 0;  // tile (and k-part) whose epilogue is pending
    for (int u = first; u < num_units && ok; u += stride, ++it) {
      int n0, m0;
      tile_coord(u % num_tiles, n_tiles, m_tiles, group_m, BT, n0, m0);
      const int ts = it & 1;
      if (!mbar_wait(bar_tfull + 8 * ts, (uint32_t)(it >> 1) & 1, status, DEV_TIMEOUT_DEQUANT)) {
        ok = false;
        break;
      }
      const uint32_t tb = sb + OFF_T + ts * TBL_BYTES + grp * 128;
      for (int kb = 0; kb < nkb; ++kb, ++g) {
        if (kb == lead && pn0 >= 0) {
          ok = epilogue(pn0, pm0, it - 1, pkp);
          pn0 = -1;
          if (!ok) break;
        }
        if ((int)(g & 1) != par) continue;
        const int s = (int)(g % AS);
        const uint32_t ph = (uint32_t)(g / AS) & 1;
        // the indices of step g landed only after step g - AS had finished with slot s, so A
        // stage s is free as well
        ok = mbar_wait(bar_pfull + 8 * s, ph, status, DEV_TIMEOUT_DEQUANT);
        if (!ok) break;
        // this lane's 24 bytes: quadruples j = 0..3 of row r0, then of row r0 + 8
        const uint32_t pa = sb + OFF_P + s * P_BYTES + grp * P_BLOCK + lane * 24;
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
        if (lane == 0) mbar_arrive(bar_ready + 8 * s);
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * ts);  // done with this tile's tables
      pn0 = n0;
      pm0 = m0;
      pkp = u / num_tiles;
    }
    if (ok && pn0 >= 0) epilogue(pn0, pm0, it - 1, pkp);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// The wide-tile GEMM (no K split): lut6_gemm_kernel's walk, producers, protocol and
// dequantisation with 128 x 384 tiles, so each weight is dequantised once per 384 tokens instead
// of 256 (the dequantising warps' integer and shared-memory work is what limits the 256-token
// tile).  Tensor memory holds two N = 192 accumulators (columns 0..383: token t of the tile in
// column t) and four A stages (columns 384..511); X, A stage and index slot share one 4-deep
// ring, each step 48 KB of X as two 192-token boxes (a copy from L2 takes ~1,600 cycles to land;
// the ring keeps three steps, ~2,300 cycles, ahead).  The MMA thread waits once per step (X bytes
// and the 8 dequantising warps), issues 8 MMAs (4 K slices x the two accumulators, M = 128,
// N = 192, A from tensor memory) and commits once; waits between MMAs cost the tensor pipe a
// third of its rate.  The 16 epilogue warps drain the tile in 32-column blocks (warp e of a lane
// quarter: blocks e, e + 4, e + 8), releasing the accumulators after the last block's load.
__global__ void __launch_bounds__(NUM_THREADS, 1)
    lut6_gemm_wide_kernel(const __grid_constant__ CUtensorMap tmap_x,
                          const __grid_constant__ CUtensorMap tmap_p, const __half* __restrict__ lut,
                          void* __restrict__ y, int64_t ldy, int M, int N, int K, int mode,
                          int group_m, unsigned* status) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkb = K / BK;
  const int n_tiles = (N + BN - 1) / BN;
  const int m_tiles = (M + WT - 1) / WT;
  const int num_tiles = n_tiles * m_tiles;
  // the accumulators of tile i are drained after the first `lead` steps of tile i+1 have been
  // dequantised, so the MMAs of tile i+1 start as soon as they are free
  const int lead = min(W_AS - 1, nkb - 1);

  const uint32_t bar_ready = sb + W_OFF_BAR;            // [W_AS] X landed and A stage written
  const uint32_t bar_empty = bar_ready + 8 * W_AS;      // [W_AS] step done: X slot, A stage, indices free
  const uint32_t bar_pfull = bar_empty + 8 * W_AS;      // [W_AS] packed indices landed
  const uint32_t bar_tfull = bar_pfull + 8 * W_AS;      // [2] tables landed
  const uint32_t bar_tempty = bar_tfull + 16;           // [2] tables no longer read
  const uint32_t bar_accf = bar_tempty + 16;            // accumulators complete
  const uint32_t bar_acce = bar_accf + 8;               // accumulators drained
  const uint32_t bar_fin = bar_acce + 8;                // the MMA thread's last MMAs completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + W_OFF_SLOT);

  if (threadIdx.x == 0) {
    for (int s = 0; s < W_AS; ++s) {
      mbar_init(bar_ready + 8 * s, 1 + NUM_DQ_WARPS / 2);
      mbar_init(bar_empty + 8 * s, 1);
      mbar_init(bar_pfull + 8 * s, 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_tfull + 8 * s, 1);
      mbar_init(bar_tempty + 8 * s, NUM_DQ_WARPS);
    }
    mbar_init(bar_accf, 1);
    mbar_init(bar_acce, NUM_DQ_WARPS);
    mbar_init(bar_fin, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmap_x);
    tma_prefetch_desc(&tmap_p);
  }
  // table slots start at zero: rows past N (a partial last tile) then see finite entries
  for (int i = threadIdx.x; i < 2 * TBL_BYTES / 4; i += NUM_THREADS)
    reinterpret_cast<uint32_t*>(smem + W_OFF_T)[i] = 0u;
  fence_proxy_async_smem();
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();   // the barriers and tensor memory are set up; now the inputs
  const int first = blockIdx.x;
  const int stride = gridDim.x;

  if (warp == 0) {
    // ---------------------------------------------------------------- X loads
    if (lane == 0) {
      int64_t g = 0;
      bool ok = true;
      for (int u = first; u < num_tiles && ok; u += stride) {
        int n0, m0;
        tile_coord(u, n_tiles, m_tiles, group_m, WT, n0, m0);
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          // X slot g % W_AS was last read by step g - W_AS
          const int s = (int)(g % W_AS);
          if (g >= W_AS && !mbar_wait(bar_empty + 8 * s, ((uint32_t)(g / W_AS) & 1) ^ 1, status,
                                      DEV_TIMEOUT_TMA)) {
            ok = false;
            break;
          }
          const uint32_t rb = bar_ready + 8 * s;
          mbar_arrive_expect_tx(rb, W_X_BYTES);
          tma_load_2d(sb + W_OFF_X + s * W_X_BYTES, &tmap_x, rb, kb * BK, m0);
          tma_load_2d(sb + W_OFF_X + s * W_X_BYTES + W_H_BYTES, &tmap_x, rb, kb * BK, m0 + WH);
        }
      }
      // copies still in flight land before the CTA may exit (a phase that already completed
      // passes at once)
      for (int64_t h = g > W_AS ? g - W_AS : 0; h < g; ++h)
        mbar_wait(bar_ready + 8 * (int)(h % W_AS), (uint32_t)(h / W_AS) & 1, status, DEV_TIMEOUT_TMA);
    }
  } else if (warp == 2) {
    // ---------------------------------------------------------------- tables + packed indices
    if (lane == 0) {
      int64_t g = 0;
      int it = 0;
      bool ok = true;
      for (int u = first; u < num_tiles && ok; u += stride, ++it) {
        int n0, m0;
        tile_coord(u, n_tiles, m_tiles, group_m, WT, n0, m0);
        const int ts = it & 1;
        if (it >= 2 && !mbar_wait(bar_tempty + 8 * ts, ((uint32_t)(it >> 1) & 1) ^ 1, status,
                                  DEV_TIMEOUT_TMA)) {
          ok = false;
          break;
        }
        const int groups = min(BN / 16, N / 16 - n0 / 16);
        mbar_arrive_expect_tx(bar_tfull + 8 * ts, groups * 128);
        bulk_load(sb + W_OFF_T + ts * TBL_BYTES, lut + (size_t)(n0 / 16) * 64, groups * 128,
                  bar_tfull + 8 * ts);
        for (int kb = 0; kb < nkb; ++kb, ++g) {
          // slot s (indices and A stage) was last used by step g - W_AS
          const int s = (int)(g % W_AS);
          const uint32_t ph = (uint32_t)(g / W_AS) & 1;
          if (g >= W_AS && !mbar_wait(bar_empty + 8 * s, ph ^ 1, status, DEV_TIMEOUT_TMA)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(bar_pfull + 8 * s, P_BYTES);
          tma_load_3d(sb + W_OFF_P + s * P_BYTES, &tmap_p, bar_pfull + 8 * s, 0, 3 * kb, n0 / 16);
        }
      }
      for (int64_t h = g > W_AS ? g - W_AS : 0; h < g; ++h)
        mbar_wait(bar_pfull + 8 * (int)(h % W_AS), (uint32_t)(h / W_AS) & 1, status, DEV_TIMEOUT_TMA);
      for (int u = it > 2 ? it - 2 : 0; u < it; ++u)
        mbar_wait(bar_tfull + 8 * (u & 1), (uint32_t)(u >> 1) & 1, status, DEV_TIMEOUT_TMA);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_f16_f32(BN, WH);
      int s = 0;          // ring slot of the current step
      uint32_t ph = 0;    // phase parity of ready[s]
      int it = 0;
      bool ok = true;
      for (int u = first; u < num_tiles && ok; u += stride, ++it) {
        if (it >= 1 && !mbar_wait(bar_acce, (uint32_t)(it - 1) & 1, status, DEV_TIMEOUT_MMA)) {
          ok = false;
          break;
        }
        for (int kb = 0; kb < nkb; ++kb) {
          // operands of this step, formed before the wait so that the MMAs issue as soon as it
          // passes
          const uint32_t a = tmem + W_A_COL + s * 32;
          const uint64_t xd = sdesc_k_sw128(sb + W_OFF_X + s * W_X_BYTES);
          if (!mbar_wait_spin(bar_ready + 8 * s, ph, status, DEV_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            tc_mma_f16_ts(tmem, a + 8 * ks, xd + 2 * ks, idesc, (kb | ks) != 0);
            tc_mma_f16_ts(tmem + WH, a + 8 * ks, xd + (W_H_BYTES >> 4) + 2 * ks, idesc, (kb | ks) != 0);
          }
          tc_commit(bar_empty + 8 * s);
          if (++s == W_AS) {
            s = 0;
            ph ^= 1;
          }
        }
        if (ok) tc_commit(bar_accf);
      }
      // tensor memory is freed below only after every MMA issued here has completed
      tc_commit(bar_fin);
      mbar_wait(bar_fin, 0, status, DEV_TIMEOUT_MMA);
    }
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- dequant + epilogue
    const int dq = warp - 4;                           // 0..15
    const int quarter = warp & 3;                      // TMEM lanes 32*quarter .. +31
    const int grp = 2 * quarter + ((dq >> 2) & 1);     // 16-row group dequantised by this warp
    const int par = dq >> 3;                           // steps g with g % 2 == par
    const int eb = dq >> 2;                            // epilogue: 32-column blocks eb, eb+4, eb+8
    const uint32_t tl = tmem + ((uint32_t)(grp * 16) << 16) + W_A_COL;
    const uint32_t tacc = tmem + ((uint32_t)(quarter * 32) << 16);

    // Drain this warp's three 32-column blocks (tokens 32 b .. 32 b + 31 of the tile) of the
    // tile at (n0e, m0e); the accumulators are released after the last block's load.
    auto epilogue = [&](int n0e, int m0e, int ite) -> bool {
      const int col = n0e + quarter * 32 + lane;
      if (!mbar_wait(bar_accf, (uint32_t)ite & 1, status, DEV_TIMEOUT_EPILOGUE)) return false;
      tc_fence_after();
      uint32_t ra[32], rb[32];
      tmem_ld_32x32b_x32(tacc + 32 * eb, ra);
      tmem_ld_32x32b_x32(tacc + 32 * (eb + 4), rb);
      tc_wait_ld();
      store_y_block(mode, y, ldy, M, N, n0e, col, m0e + 32 * eb, quarter, lane, 0, ra, ra, 32);
      tmem_ld_32x32b_x32(tacc + 32 * (eb + 8), ra);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acce);
      store_y_block(mode, y, ldy, M, N, n0e, col, m0e + 32 * (eb + 4), quarter, lane, 0, rb, rb, 32);
      store_y_block(mode, y, ldy, M, N, n0e, col, m0e + 32 * (eb + 8), quarter, lane, 0, ra, ra, 32);
      return true;
    };

    int64_t g = 0;
    int it = 0;
    bool ok = true;
    int pn0 = -1, pm0 = 0;  // tile whose epilogue is pending
    for (int u = first; u < num_tiles && ok; u += stride, ++it) {
      int n0, m0;
      tile_coord(u, n_tiles, m_tiles, group_m, WT, n0, m0);
      const int ts = it & 1;
      if (!mbar_wait(bar_tfull + 8 * ts, (uint32_t)(it >> 1) & 1, status, DEV_TIMEOUT_DEQUANT)) {
        ok = false;
        break;
      }
      const uint32_t tb = sb + W_OFF_T + ts * TBL_BYTES + grp * 128;
      for (int kb = 0; kb < nkb; ++kb, ++g) {
        if (kb == lead && pn0 >= 0) {
          ok = epilogue(pn0, pm0, it - 1);
          pn0 = -1;
          if (!ok) break;
        }
        if ((int)(g & 1) != par) continue;
        const int s = (int)(g % W_AS);
        const uint32_t ph = (uint32_t)(g / W_AS) & 1;
        // the indices of step g landed only after step g - W_AS had finished with slot s, so A
        // stage s is free as well
        ok = mbar_wait(bar_pfull + 8 * s, ph, status, DEV_TIMEOUT_DEQUANT);
        if (!ok) break;
        // this lane's 24 bytes: quadruples j = 0..3 of row r0, then of row r0 + 8
        const uint32_t pa = sb + W_OFF_P + s * P_BYTES + grp * P_BLOCK + lane * 24;
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
        if (lane == 0) mbar_arrive(bar_ready + 8 * s);
      }
      if (!ok) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_tempty + 8 * ts);  // done with this tile's tables
      pn0 = n0;
      pm0 = m0;
    }
    if (ok && pn0 >= 0) epilogue(pn0, pm0, it - 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// y[t][c] += part[0][t][c] + part[1][t][c] + ... added one part at a time in part order (the
// same sequence of fp32 additions on every run); part is [parts][M][N].  Four columns per thread.
__global__ void split_reduce_kernel(float* __restrict__ y, int64_t ldy, const float* __restrict__ part,
                                    int parts, int64_t M, int64_t N) {
  pdl_trigger();
  pdl_wait();
  const int64_t quads = M * (N / 4);
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < quads;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t t = i / (N / 4), c = 4 * (i % (N / 4));
    float4 acc = *reinterpret_cast<const float4*>(y + t * ldy + c);
    for (int p = 0; p < parts; ++p) {
      const float4 v = *reinterpret_cast<const float4*>(part + ((int64_t)p * M + t) * N + c);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    *reinterpret_cast<float4*>(y + t * ldy + c) = acc;
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

bool lut6_use_wide(int64_t M, int64_t N) {
  // 384-token tiles once there are enough of them to fill the GPU's SMs
  using namespace lut;
  const int64_t wtiles = ((N + BN - 1) / BN) * ((M + WT - 1) / WT);
  return M >= 2048 && wtiles >= num_sms();
}

int lut6_group_m(int64_t K, int mode, int tile_tokens) {
  // As many token tiles per group as keep the group's X rows (tile_tokens x K fp16 each) within
  // 32 MB of L2, which leaves room for the weight tiles and the output in flight: fewer groups
  // mean fewer passes of the packed weights through DRAM.  Measured at 16,384 tokens with
  // 256-token tiles: 16 tiles (32 MB of X) at K = 4096 cut a SwiGLU launch's DRAM reads from 736
  // to 474 MB, 32 tiles made X itself miss (2.3 GB); residual adds, whose fp32
  // read-modify-write of Y also passes through L2, keep 2,048 tokens per group (16 tiles read
  // 17% more and ran 2% slower).
  using namespace lut;
  if (mode == EPI_ADD_F32 || mode == EPI_PART_F32) return 8 * BT / tile_tokens;
  constexpr int64_t kXBudget = 32ll << 20;
  int g = 2;
  while (g < 64 && 2 * g * (int64_t)tile_tokens * K * 2 <= kXBudget) g *= 2;
  return g;
}

int lut6_add_split(int64_t M, int64_t N, int64_t K) {
  // When there are too few tiles to fill the GPU, pick the split that minimises the longest
  // CTA's work, counted in k-steps plus about four steps per unit for its epilogue.
  using namespace lut;
  const int64_t tiles = ((N + BN - 1) / BN) * ((M + BT - 1) / BT);
  const int64_t sms = num_sms();
  const int64_t nkb = K / BK;
  int ksplit = 1;
  int64_t best = -1;
  for (int s = 1; s <= 8; ++s) {
    if (nkb % s != 0 || nkb / s < 4) continue;
    const int64_t rounds = (tiles * s + sms - 1) / sms;
    const int64_t cost = rounds * (nkb / s + 4);
    if (best < 0 || cost < best) {
      best = cost;
      ksplit = s;
    }
  }
  return ksplit;
}

clef_status lut6_gemm_launch(const __half* x, const uint8_t* tiled, const __half* lut, void* y,
                             int64_t ldy, int64_t M, int64_t N, int64_t K, int mode,
                             cudaStream_t stream, float* part_ws) {
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
  // the tables are fetched with 16-byte bulk copies
  if ((reinterpret_cast<uintptr_t>(lut) & 15) != 0) return CLEF_E_ALIGN;
  const int64_t tiles = ((N + BN - 1) / BN) * ((M + BT - 1) / BT);
  const int sms = num_sms();
  // Residual-add mode may split K across CTAs (each part adds its partial sum, or with part_ws
  // writes it to its own slice for the ordered reduction below)
  const int ksplit = mode == EPI_ADD_F32 ? lut6_add_split(M, N, K) : 1;
  const double out_bytes = mode == EPI_F16 ? 2.0 * M * N
                           : mode == EPI_F32 ? 4.0 * M * N
                           : mode == EPI_ADD_F32 ? 8.0 * M * N
                                                 : 1.0 * M * N;  // SwiGLU: fp16 [M, N/2]
  if (ksplit == 1 && lut6_use_wide(M, N)) {
    CUtensorMap txw;
    if (tma_encode_2d(&txw, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x, (uint64_t)K, (uint64_t)M,
                      (uint64_t)K * 2, BK, WH, CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess)
      return CLEF_E_CUDA;
    static std::atomic<uint64_t> wattr{0};
    CLEF_CUDA_CHECK(smem_opt_in((const void*)lut6_gemm_wide_kernel, W_SMEM_BYTES, &wattr));
    const int64_t wtiles = ((N + BN - 1) / BN) * ((M + WT - 1) / WT);
    const unsigned grid = (unsigned)(wtiles < sms ? wtiles : sms);
    TraceScope ts(stream, "lut6_gemm", 2.0 * M * N * K,
                  0.75 * N * K + 8.0 * N + 2.0 * M * K + out_bytes);
    CLEF_CUDA_CHECK(launch_pdl(lut6_gemm_wide_kernel, dim3(grid), dim3(NUM_THREADS), W_SMEM_BYTES,
                               stream, txw, tp, lut, y, ldy, (int)M, (int)N, (int)K, mode,
                               lut6_group_m(K, mode, WT), status_word_ptr()));
    return CLEF_OK;
  }
  static std::atomic<uint64_t> attr{0};
  CLEF_CUDA_CHECK(smem_opt_in((const void*)lut6_gemm_kernel, SMEM_BYTES, &attr));
  const bool ordered = ksplit > 1 && part_ws != nullptr;
  if (ordered && (N % 4 != 0 || ldy % 4 != 0 || (reinterpret_cast<uintptr_t>(part_ws) & 15) != 0))
    return CLEF_E_ALIGN;
  const int64_t units = tiles * ksplit;
  const unsigned grid = (unsigned)(units < sms ? units : sms);
  {
    TraceScope ts(stream, "lut6_gemm", 2.0 * M * N * K,
                  0.75 * N * K + 8.0 * N + 2.0 * M * K + out_bytes);
    CLEF_CUDA_CHECK(launch_pdl(lut6_gemm_kernel, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, stream,
         tx, tp, lut, ordered ? static_cast<void*>(part_ws) : y, ordered ? N : ldy, (int)M, (int)N,
         (int)K, ordered ? (int)EPI_PART_F32 : mode, ksplit, lut6_group_m(K, mode, BT), status_word_ptr()));
  }
  if (ordered) {
    TraceScope ts(stream, "split_reduce", 0.0, 4.0 * M * N * (2 + ksplit));
    const int64_t quads = M * (N / 4);
    const int64_t blocks = std::min<int64_t>((quads + 255) / 256, (int64_t)sms * 8);
    CLEF_CUDA_CHECK(launch_pdl(split_reduce_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
         static_cast<float*>(y), ldy, part_ws,
         ksplit, M, N));
  }
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
