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
constexpr int GROUP_M = 8;                    // token tiles walked together (L2 reuse)
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
constexpr int NUM_BARS = 3 * AS + 4 + 3 + 2;
constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_FLAG = OFF_SLOT + 16;       // stream-K: "this CTA finishes the tile"
constexpr int SMEM_USED = OFF_FLAG + 16;
constexpr int SMEM_BYTES = SMEM_USED + 1024;  // slack to align the base to 1024
static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
static_assert(A_COL + AS * 32 <= TMEM_COLS, "tensor memory budget");
static_assert(CLEF_SWIGLU_BLOCK == 16 && BN % (2 * CLEF_SWIGLU_BLOCK) == 0,
              "a gate row and its up row are 16 lanes apart in one warp's 32 lanes");

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
// groups of GROUP_M token tiles: inside a group the token tile varies fastest, so the CTAs
// running at one time share a few weight tiles and a few X tiles, which stay in L2.
__device__ __forceinline__ void tile_coord(int t, int n_tiles, int m_tiles, int& n0, int& m0) {
  const int per_group = GROUP_M * n_tiles;
  const int grp = t / per_group;
  const int first_m = grp * GROUP_M;
  const int gm = min(GROUP_M, m_tiles - first_m);
  const int local = t - grp * per_group;
  m0 = (first_m + local % gm) * BT;
  n0 = (local / gm) * BN;
}

// ---- schedule ------------------------------------------------------------------------------
// Tiles [0, dp) go whole to the CTAs in turn (CTA c: tiles c, c + G, ...).  The k-steps of the
// remaining tiles are shared evenly by the first `sk` CTAs (stream-K): CTA c takes steps
// [c S / sk, (c + 1) S / sk) of the S = (tiles - dp) * num_kb steps (tile-major), cut into one
// segment per tile it touches (at most 3: the tiles left over are fewer than 2 G, so a share is
// under 2 num_kb steps).  A stream-K segment writes its partial sums to partial slot 3 c + i;
// the last CTA to finish a tile adds the tile's pieces in CTA order and writes the output.
struct Seg {
  int tile, kb0, kb1;
  int slot;        // -1: a whole tile of the data-parallel part
  int sk_tile;     // stream-K tile index (tile - dp)
};

// 32-bit arithmetic throughout: the shared steps S are fewer than 2 SMs x num_kb (num_kb <=
// 2^14), so c * S stays far below 2^31.
struct Sched {
  int G, num_tiles, num_kb, dp, sk;
  __host__ __device__ int sk_steps() const { return (num_tiles - dp) * num_kb; }
  __host__ __device__ int share_begin(int c) const {
    return (int)((unsigned)c * (unsigned)sk_steps() / (unsigned)sk);
  }
  // segment j of CTA c; false when there is none
  __host__ __device__ bool seg(int c, int j, Seg& g) const {
    const int n_dp = c < dp ? (dp - 1 - c) / G + 1 : 0;
    if (j < n_dp) {
      g.tile = c + j * G;
      g.kb0 = 0;
      g.kb1 = num_kb;
      g.slot = -1;
      g.sk_tile = -1;
      return true;
    }
    if (c >= sk || sk_steps() == 0) return false;
    const int i = j - n_dp;
    const int a = share_begin(c), b = share_begin(c + 1);
    const int t = a / num_kb + i;
    const int s0 = t * num_kb > a ? t * num_kb : a;
    const int s1 = (t + 1) * num_kb < b ? (t + 1) * num_kb : b;
    if (s0 >= s1) return false;
    g.tile = dp + t;
    g.kb0 = s0 - t * num_kb;
    g.kb1 = s1 - t * num_kb;
    g.slot = 3 * c + i;
    g.sk_tile = t;
    return true;
  }
  // the CTA whose share holds shared step s
  __host__ __device__ int owner(int s) const {
    int c = (int)((unsigned)s * (unsigned)sk / (unsigned)sk_steps());
    while (c > 0 && share_begin(c) > s) --c;
    while (share_begin(c + 1) <= s) ++c;
    return c;
  }
  // the CTAs whose shares hold steps of stream-K tile t: c_lo .. c_hi
  __host__ __device__ void pieces(int t, int& c_lo, int& c_hi) const {
    c_lo = owner(t * num_kb);
    c_hi = owner(t * num_kb + num_kb - 1);
  }
};

// What one epilogue warp needs to write its 32 channels x 64 tokens of a tile.
struct EpiCtx {
  void* y;
  int64_t ldy;
  int M, N, mode;
  int ecol, ch, quarter, lane;
};

// Write Y for the warp's 32 channels x 64 tokens of the tile at (n0e, m0e) from r0 (tokens
// ecol .. ecol + 31) and r1 (tokens ecol + 32 .. ecol + 63).
__device__ __forceinline__ void store_tile(const EpiCtx& x, int n0e, int m0e,
                                           const uint32_t (&r0)[32], const uint32_t (&r1)[32]) {
  const int tok0 = m0e + x.ecol;
  const int col = n0e + x.ch;
  if (x.mode == EPI_SWIGLU_F16) {
    // lanes 0..15: gate rows, lanes 16..31: the up rows of the same channels; the gate lane
    // writes tokens 0..31 of the warp's 64, the up lane tokens 32..63
    const bool up = x.lane >= 16;
    const int oc = n0e / 2 + x.quarter * 16 + (x.lane & 15);
    __half* out = reinterpret_cast<__half*>(x.y);
    const bool oc_ok = oc < x.N / 2;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const uint32_t send = up ? r0[i] : r1[i];
      const float other = __uint_as_float(__shfl_xor_sync(0xffffffffu, send, 16));
      const float gate = up ? other : __uint_as_float(r0[i]);
      const float upv = up ? __uint_as_float(r1[i]) : other;
      const int tok = tok0 + (up ? 32 : 0) + i;
      if (oc_ok && tok < x.M) out[(int64_t)tok * x.ldy + oc] = __float2half_rn(silu_f(gate) * upv);
    }
  } else if (col < x.N) {
    if (x.mode == EPI_F16) {
      __half* out = reinterpret_cast<__half*>(x.y) + col;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (tok0 + i < x.M) out[(int64_t)(tok0 + i) * x.ldy] = __float2half_rn(__uint_as_float(r0[i]));
        if (tok0 + 32 + i < x.M)
          out[(int64_t)(tok0 + 32 + i) * x.ldy] = __float2half_rn(__uint_as_float(r1[i]));
      }
    } else if (x.mode == EPI_F32) {
      float* out = reinterpret_cast<float*>(x.y) + col;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (tok0 + i < x.M) out[(int64_t)(tok0 + i) * x.ldy] = __uint_as_float(r0[i]);
        if (tok0 + 32 + i < x.M) out[(int64_t)(tok0 + 32 + i) * x.ldy] = __uint_as_float(r1[i]);
      }
    } else {
      // residual add, done by L2: each element receives exactly one add per launch (the same
      // as load + add + store), so launches repeat bit for bit
      float* out = reinterpret_cast<float*>(x.y) + col;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        if (tok0 + i < x.M) red_add_f32(out + (int64_t)(tok0 + i) * x.ldy, __uint_as_float(r0[i]));
        if (tok0 + 32 + i < x.M)
          red_add_f32(out + (int64_t)(tok0 + 32 + i) * x.ldy, __uint_as_float(r1[i]));
      }
    }
  }
}

// The end of a stream-K piece, once every epilogue warp has stored its partial sums (and fenced
// them) and arrived on bar_pc: one thread counts the piece for the tile; the CTA that brings the
// count to the tile's number of pieces adds all pieces (its own included, read back from L2) in
// CTA order and writes the tile.
__device__ __forceinline__ bool sk_finish(const EpiCtx& x, const Sched& sc, int tile, int sk_tile,
                                       int n0e, int m0e, const float* part,
                                       unsigned* tile_count, uint32_t bar_pc, uint32_t bar_pd,
                                       volatile int* sk_last, int parity, bool leader,
                                       unsigned* status) {
  int c_lo, c_hi;
  sc.pieces(sk_tile, c_lo, c_hi);
  if (leader) {
    int last = 0;
    if (mbar_wait(bar_pc, (uint32_t)parity, status, DEV_TIMEOUT_EPILOGUE)) {
      const unsigned before = atomicAdd(tile_count + sk_tile, 1u);
      last = before == (unsigned)(c_hi - c_lo) ? 1 : 0;
      if (last) tile_count[sk_tile] = 0u;   // ready for the next launch
      __threadfence();
    }
    *sk_last = last;
    mbar_arrive(bar_pd);
  }
  if (!mbar_wait(bar_pd, (uint32_t)parity, status, DEV_TIMEOUT_EPILOGUE)) return false;
  if (*sk_last) {
    uint32_t r0[32], r1[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r0[i] = r1[i] = __float_as_uint(0.f);
    for (int c = c_lo; c <= c_hi; ++c) {
      const int slot = 3 * c + (sk_tile - sc.share_begin(c) / sc.num_kb);
      const float* piece = part + (int64_t)slot * (BT * BN);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        r0[i] = __float_as_uint(__uint_as_float(r0[i]) + __ldcg(piece + (x.ecol + i) * BN + x.ch));
        r1[i] = __float_as_uint(__uint_as_float(r1[i]) +
                                __ldcg(piece + (x.ecol + 32 + i) * BN + x.ch));
      }
    }
    store_tile(x, n0e, m0e, r0, r1);
  }
  (void)tile;
  return true;
}

__global__ void __launch_bounds__(NUM_THREADS, 1)
    lut6_gemm_kernel(const __grid_constant__ CUtensorMap tmap_x,
                     const __grid_constant__ CUtensorMap tmap_p, const __half* __restrict__ lut,
                     void* __restrict__ y, int64_t ldy, int M, int N, int K, int mode, Sched sc,
                     float* __restrict__ part, unsigned* __restrict__ tile_count,
                     unsigned* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int n_tiles = (N + BN - 1) / BN;
  const int m_tiles = (M + BT - 1) / BT;
  const int cta = blockIdx.x;

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
  const uint32_t bar_pc = bar_fin + 8;                 // stream-K: every warp's partial stored
  const uint32_t bar_pd = bar_pc + 8;                  // stream-K: the tile counter was read
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_SLOT);
  volatile int* sk_last = reinterpret_cast<volatile int*>(smem + OFF_FLAG);

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
    mbar_init(bar_pc, NUM_DQ_WARPS);
    mbar_init(bar_pd, 1);
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

  if (warp == 0) {
    // ---------------------------------------------------------------- X loads
    if (lane == 0) {
      int64_t g = 0;
      bool ok = true;
      Seg sg;
      for (int j = 0; ok && sc.seg(cta, j, sg); ++j) {
        int n0, m0;
        tile_coord(sg.tile, n_tiles, m_tiles, n0, m0);
        for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++g) {
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
      Seg sg;
      for (; ok && sc.seg(cta, it, sg); ++it) {
        int n0, m0;
        tile_coord(sg.tile, n_tiles, m_tiles, n0, m0);
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
        for (int kb = sg.kb0; kb < sg.kb1; ++kb, ++g) {
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
      // `it` segments had their tables requested (the loop stops on the first missing one)
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
      bool ok = true;
      Seg sg;
      for (int it = 0; ok && sc.seg(cta, it, sg); ++it) {
        if (it >= 1 && !mbar_wait(bar_acce, (uint32_t)(it - 1) & 1, status, DEV_TIMEOUT_MMA)) {
          ok = false;
          break;
        }
        for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
          if (!mbar_wait(bar_ready + 8 * sa, ph, status, DEV_TIMEOUT_MMA)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a = tmem + A_COL + sa * 32;
          const uint32_t b = sb + OFF_X + sx * X_BYTES;
          tc_mma_f16_ts(tmem, a, sdesc_k_sw128(b), idesc, kb != sg.kb0);
          tc_mma_f16_ts(tmem, a + 8, sdesc_k_sw128(b + 32), idesc, 1);
          tc_mma_f16_ts(tmem, a + 16, sdesc_k_sw128(b + 64), idesc, 1);
          tc_mma_f16_ts(tmem, a + 24, sdesc_k_sw128(b + 96), idesc, 1);
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
    const int ch = quarter * 32 + lane;                // this lane's channel in the tile
    int sk_done = 0;                                   // stream-K epilogues so far (parities)

    const EpiCtx ex{y, ldy, M, N, mode, ecol, ch, quarter, lane};

    // Drain this warp's 32 lanes x 64 columns of the accumulator of this CTA's segment `ite`,
    // release it, then write Y, or (a stream-K piece) store the partial sums and finish the
    // piece (sk_finish).  The segment is looked up again here, so that the dequantisation loop
    // keeps only its index.
    auto epilogue = [&](int ite) -> bool {
      Seg e;
      sc.seg(cta, ite, e);
      int n0e, m0e;
      tile_coord(e.tile, n_tiles, m_tiles, n0e, m0e);
      if (!mbar_wait(bar_accf, (uint32_t)ite & 1, status, DEV_TIMEOUT_EPILOGUE)) return false;
      tc_fence_after();
      uint32_t r0[32], r1[32];
      tmem_ld_32x32b_x32(tacc, r0);
      tmem_ld_32x32b_x32(tacc + 32, r1);
      tc_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_acce);
      if (e.slot < 0) {
        store_tile(ex, n0e, m0e, r0, r1);
        return true;
      }
      // a stream-K piece: partial sums [token][channel] in its slot, fenced before the count
      float* mine = part + (int64_t)e.slot * (BT * BN);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        mine[(ecol + i) * BN + ch] = __uint_as_float(r0[i]);
        mine[(ecol + 32 + i) * BN + ch] = __uint_as_float(r1[i]);
      }
      __threadfence();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_pc);
      const bool done = sk_finish(ex, sc, e.tile, e.sk_tile, n0e, m0e, part, tile_count, bar_pc,
                                  bar_pd, sk_last, sk_done & 1, dq == 0 && lane == 0, status);
      ++sk_done;
      return done;
    };

    int64_t g = 0;
    bool ok = true;
    int pending = -1;       // the segment whose epilogue is due
    Seg sg;
    int it = 0;
    for (; ok && sc.seg(cta, it, sg); ++it) {
      const int ts = it & 1;
      if (!mbar_wait(bar_tfull + 8 * ts, (uint32_t)(it >> 1) & 1, status, DEV_TIMEOUT_DEQUANT)) {
        ok = false;
        break;
      }
      const uint32_t tb = sb + OFF_T + ts * TBL_BYTES + grp * 128;
      // the accumulator of the previous segment is drained after the first `lead` steps of this
      // one have been dequantised, so its MMAs start as soon as the accumulator is free
      const int nsteps = sg.kb1 - sg.kb0;
      const int lead = min(AS - 1, nsteps - 1);
      for (int step = 0; step < nsteps; ++step, ++g) {
        if (step == lead && pending >= 0) {
          ok = epilogue(pending);
          pending = -1;
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
      if (lane == 0) mbar_arrive(bar_tempty + 8 * ts);  // done with this segment's tables
      pending = it;
    }
    if (ok && pending >= 0) epilogue(pending);
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

int64_t lut6_split_part_bytes() { return (int64_t)num_sms() * 3 * lut::BT * lut::BN * 4; }
int64_t lut6_split_count_bytes() { return (int64_t)num_sms() * 2 * 4; }

// The schedule of one launch: every tile data-parallel, or (given the partial-sum workspace)
// the full waves data-parallel and the rest stream-K, whichever leaves the busiest CTA fewer
// k-steps (an epilogue counted as about 4 steps; a stream-K share adds two partial epilogues
// and the final sum, about 14), by a margin of 8 steps.
static lut::Sched plan_schedule(int64_t M, int64_t N, int64_t K, int sms, bool can_split) {
  using namespace lut;
  const int tiles = (int)(((N + BN - 1) / BN) * ((M + BT - 1) / BT));
  const int nkb = (int)(K / BK);
  Sched dp_only{tiles < sms ? tiles : sms, tiles, nkb, tiles, 0};
  if (!can_split || tiles % sms == 0) return dp_only;
  const int64_t cost_dp = (int64_t)((tiles + sms - 1) / sms) * (nkb + 4);
  const int waves = tiles / sms;
  const int dp = waves >= 1 ? (waves - 1) * sms : 0;
  const int64_t S = (int64_t)(tiles - dp) * nkb;   // < 2 sms num_kb: fits the 32-bit schedule
  const int sk = (int)std::max<int64_t>(1, std::min<int64_t>(sms, S / 8));
  const int64_t cost_sk = (int64_t)(dp / sms) * (nkb + 4) + (S + sk - 1) / sk + 14;
  if (cost_sk + 8 >= cost_dp) return dp_only;
  return Sched{sms, tiles, nkb, dp, sk};
}

clef_status lut6_gemm_launch(const __half* x, const uint8_t* tiled, const __half* lut, void* y,
                             int64_t ldy, int64_t M, int64_t N, int64_t K, int mode,
                             cudaStream_t stream, float* part, unsigned* counts) {
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
  static std::atomic<uint64_t> attr{0};
  CLEF_CUDA_CHECK(smem_opt_in((const void*)lut6_gemm_kernel, SMEM_BYTES, &attr));
  // the tables are fetched with 16-byte bulk copies
  if ((reinterpret_cast<uintptr_t>(lut) & 15) != 0) return CLEF_E_ALIGN;
  const int sms = num_sms();
  const bool can_split = part != nullptr && counts != nullptr &&
                         (reinterpret_cast<uintptr_t>(part) & 15) == 0;
  const Sched sc = plan_schedule(M, N, K, sms, can_split);
  const double out_bytes = mode == EPI_F16 ? 2.0 * M * N
                           : mode == EPI_F32 ? 4.0 * M * N
                           : mode == EPI_ADD_F32 ? 8.0 * M * N
                                                 : 1.0 * M * N;  // SwiGLU: fp16 [M, N/2]
  TraceScope ts(stream, "lut6_gemm", 2.0 * M * N * K,
                0.75 * N * K + 8.0 * N + 2.0 * M * K + out_bytes);
  lut6_gemm_kernel<<<(unsigned)sc.G, NUM_THREADS, SMEM_BYTES, stream>>>(
      tx, tp, lut, y, ldy, (int)M, (int)N, (int)K, mode, sc, part, counts, status_word_ptr());
  CLEF_LAUNCH_CHECK();
  return CLEF_OK;
}

}  // namespace clef

// Host only: the schedule a LUT-6 GEMM launch of this shape would use on `sms` SMs with the
// stream-K workspace (for tests of its index arithmetic without a GPU).  plan[4] = grid,
// data-parallel tiles, stream-K CTAs, tiles; segs[5 * i ..] = (cta, tile, kb0, kb1, slot) of
// every CTA's segments in order; pieces[2 * t ..] = (first, last) CTA of stream-K tile t.
extern "C" clef_status clef_debug_lut6_schedule(int64_t M, int64_t N, int64_t K, int32_t sms,
                                                int32_t* plan, int32_t* segs, int32_t max_segs,
                                                int32_t* n_segs, int32_t* pieces,
                                                int32_t max_pieces) {
  using namespace clef;
  using namespace clef::lut;
  if (!plan || !segs || !n_segs || !pieces || M < 1 || N < 16 || K < 64 || sms < 1)
    return CLEF_E_INVALID;
  const Sched sc = plan_schedule(M, N, K, sms, true);
  plan[0] = sc.G;
  plan[1] = sc.dp;
  plan[2] = sc.sk;
  plan[3] = sc.num_tiles;
  int n = 0;
  for (int c = 0; c < sc.G; ++c) {
    Seg g;
    for (int j = 0; sc.seg(c, j, g); ++j) {
      if (n == max_segs) return CLEF_E_SHAPE;
      int32_t* r = segs + 5 * n++;
      r[0] = c;
      r[1] = g.tile;
      r[2] = g.kb0;
      r[3] = g.kb1;
      r[4] = g.slot;
    }
  }
  *n_segs = n;
  const int sk_tiles = sc.num_tiles - sc.dp;
  if (sk_tiles > max_pieces) return CLEF_E_SHAPE;
  for (int t = 0; t < sk_tiles && sc.sk > 0; ++t) sc.pieces(t, pieces[2 * t], pieces[2 * t + 1]);
  return CLEF_OK;
}

namespace clef {

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
