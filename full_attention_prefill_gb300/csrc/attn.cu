// Causal GQA attention of the gated full-attention layers.
//
// "Clef-Flash-ANE-LUT6" model card, "Model architecture": heads of size 256, 16 for queries and
// 4 shared key/value heads.
// "clef-flash-LiteRT" README, "Host contract" step 5: rotary with theta = 1e7 and, for text, the
// position (i, i, i) on all three planes, i.e. a 1-D rotary; "clef-flash-coreml" README: cos/sin
// tables [L, 64], i.e. 64 rotated dims per head.  "Provenance": grouped keys/values shared by the
// query heads of a group, causal additive mask.
//
//   rope_kernel   rotates dims 0..63 of every q and k head (rotate-half pairs (j, j+32), angle
//                 pos * 1e7^(-j/32), formed and reduced to [-pi, pi] in fp64), in place or into a copy.  With a picture
//                 block (M-RoPE, "Host contract" step 5: three planes, sections 11 / 11 / 10
//                 interleaved, so pair j reads plane j mod 3), a picture token k at index s + k
//                 has planes (s, s + k / W, s + k % W) and tokens after the block move back by
//                 N - max(H, W) ("clef-flash - Core AI" README, "Core AI shape").
//   flash_tc_kernel  one CTA = 32 positions x the 4 query heads of one kv head (128 rows), so
//                 each K/V tile is read once for the group; tcgen05 MMAs with S and O in tensor
//                 memory; online softmax over 64-key tiles; epilogue o * sigmoid(gate).
#include <algorithm>
#include <cmath>

#include "attn.cuh"
#include "common.cuh"

namespace clef {
namespace attn {

constexpr int D = 256;
constexpr int HQ = 16, HKV = 4;
constexpr int BM = 128;            // rows per CTA = 32 positions x 4 heads
constexpr int POS = BM / 4;        // positions per CTA

// The 32 rotary frequencies 1e7^(-j/32), computed once in fp64 on the host.
struct RopeFreq {
  double f[32];
};

// One CTA (96 threads) per token.  Thread i < 80 owns head i / 4 (q heads 0..15, then the 4 k
// heads) and the rotated pairs j = 8 (i mod 4) .. + 7: it loads dims j .. j + 7 and j + 32 ..
// j + 39 of its head (two 16-byte loads) before the angles are formed, so the loads are in
// flight meanwhile; the first warp forms the token's 32 angles.
__global__ void __launch_bounds__(96) rope_kernel(const __half* __restrict__ qin, int64_t ldqi,
                                                  __half* __restrict__ qout, int64_t ldqo,
                                                  const __half* __restrict__ kin, int64_t ldki,
                                                  __half* __restrict__ kout, int64_t ldko, int L,
                                                  int pos0, int64_t kctx, int mstart, int mh,
                                                  int mw, const __grid_constant__ RopeFreq fr) {
  pdl_trigger();
  pdl_wait();
  __shared__ float cs[32], sn[32];
  const int64_t tok = blockIdx.x;
  const int64_t t = tok % L;
  const int idx = pos0 + (int)t;   // token index in the request
  // k goes to row (request * kctx + idx) of kout (kctx = L, pos0 = 0: the token's own row)
  const int64_t krow = (tok / L) * kctx + idx;
  const int tid = threadIdx.x;
  const int head = tid / 4, j0 = (tid % 4) * 8;
  uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
  __half* dst = nullptr;
  if (tid < 4 * (HQ + HKV)) {
    const __half* src;
    if (head < HQ) {
      src = qin + tok * ldqi + head * D;
      dst = qout + tok * ldqo + head * D;
    } else {
      src = kin + tok * ldki + (head - HQ) * D;
      dst = kout + krow * ldko + (head - HQ) * D;
    }
    lo = *reinterpret_cast<const uint4*>(src + j0);
    hi = *reinterpret_cast<const uint4*>(src + j0 + 32);
  }
  if (tid < 32) {
    // M-RoPE planes of this token (all equal to idx for text)
    const int n = mh * mw;
    int pt = idx, ph = idx, pw = idx;
    if (n > 0 && idx >= mstart) {
      if (idx < mstart + n) {
        const int k = idx - mstart;
        pt = mstart;
        ph = mstart + k / mw;
        pw = mstart + k % mw;
      } else {
        pt = ph = pw = idx - (n - max(mh, mw));
      }
    }
    const int plane = tid % 3;
    const int pos = plane == 0 ? pt : (plane == 1 ? ph : pw);
    // angle = pos * theta^(-j/32) formed in fp64 and reduced to [-pi, pi] there (Cody and
    // Waite's two-constant reduction, with 2 pi as its nearest double plus the remainder, each
    // k * constant taken exactly inside an fma), then sin and cos in fp32 of the reduced angle:
    // a few fp64 operations per angle instead of an fp64 sin/cos (fp64 runs at a small fraction
    // of the fp32 rate on this part)
    const double a = (double)pos * fr.f[tid];
    const double kq = rint(a * 0.15915494309189535);          // 1 / (2 pi)
    double r = fma(-kq, 6.2831853071795860, a);                // 2 pi rounded to double
    r = fma(-kq, 2.4492935982947064e-16, r);                   // 2 pi minus that
    float s, c;
    sincosf((float)r, &s, &c);
    cs[tid] = c;
    sn[tid] = s;
  }
  __syncthreads();
  const bool copy_q = qout != qin, copy_k = kout != kin;
  if (dst) {
    // pairs (j, j + 32) of this thread: x1 from `lo`, x2 from `hi`
    const __half2* l2 = reinterpret_cast<const __half2*>(&lo);
    const __half2* h2 = reinterpret_cast<const __half2*>(&hi);
    uint32_t ol[4], oh[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const float2 x1 = __half22float2(l2[p]), x2 = __half22float2(h2[p]);
      const int j = j0 + 2 * p;
      ol[p] = pack_half2(x1.x * cs[j] - x2.x * sn[j], x1.y * cs[j + 1] - x2.y * sn[j + 1]);
      oh[p] = pack_half2(x2.x * cs[j] + x1.x * sn[j], x2.y * cs[j + 1] + x1.y * sn[j + 1]);
    }
    *reinterpret_cast<uint4*>(dst + j0) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
    *reinterpret_cast<uint4*>(dst + j0 + 32) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
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
      *reinterpret_cast<uint4*>(kout + krow * ldko + head * D + c8) =
          *reinterpret_cast<const uint4*>(kin + tok * ldki + head * D + c8);
    }
  }
}

// ------------------------------------------------------------------------------------------
// tcgen05 flash attention.  CTA = 128 rows (32 positions x the 4 query heads of kv head g, row
// r = 4 * position + head), keys in tiles of 64.
//   warp 0   TMA: K tiles (4 stages, 4 boxes of 64 dims, 128-byte swizzle)
//   warp 2   TMA: V tiles (2 stages), a ring of its own so K runs ahead of V
//   warp 1   MMA: S_j = Q K_j^T (M=128, N=64, 16 steps of K=16; Q from tensor memory) into one
//            of two 64-column S buffers, once P_{j-2} V_{j-2} has released that buffer
//   warp 3   MMA: O += P_j V_j (M=128, N=256, K=64; P_j read from the first 32 columns of its S
//            buffer, V an MN-major shared operand).  The two MMA chains have a thread each: a
//            thread's mbarrier waits complete only after the MMAs it has committed.
//   warps 4-11 first copy Q (rows of 256 dims, after rotary) from global memory into tensor
//            memory; then softmax in two groups that take alternate tiles: warps 4-7 the even
//            tiles (S buffer 0), warps 8-11 the odd ones (buffer 1), one thread per row and all
//            64 keys of its tile (warps w and w+4 share TMEM lanes 32 (w % 4)..).  A thread reads
//            S, masks (diagonal tiles only), takes the tile's max and then, in base 2, the
//            online softmax step against a reference max that passes from group to group once
//            per tile (shared memory and a named arrive / sync barrier, before either group's
//            exponentials, so two tiles' exponentials run at once), and writes P (fp16) over
//            the first 32 columns of its S buffer.  The reference, and with it O (in TMEM, by
//            the row's thread), moves only when a row's max grows by more than 2^8, so P stays
//            below 256; each group keeps its share of the row sum relative to the reference it
//            last used.  The final O is divided by the combined row sum, multiplied by
//            sigmoid(gate) and stored, each thread of a row taking half of its columns.
// Tensor memory (512 columns): O [0,256), S/P buffers [256,320) and [320,384), Q [384,512).
// ------------------------------------------------------------------------------------------
constexpr int TBN = 64;                   // keys per tile
constexpr int KV_BLOCK = TBN * 128;       // 8 KB: [64 keys][64 dims]
constexpr int KV_BYTES = TBN * D * 2;     // 32 KB: 4 blocks
constexpr int KST = 4, VST = 2;           // K and V ring stages
constexpr int OFF_K = 0;
constexpr int OFF_V = OFF_K + KST * KV_BYTES;
constexpr int OFF_BAR = OFF_V + VST * KV_BYTES;
constexpr int NUM_BARS = 1 + 2 * KST + 2 * VST + 2 + 2 + 2 + 2;
constexpr int OFF_SLOT = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_XCH = OFF_SLOT + 16;       // 6 x [128 rows] fp32: reference maxima, row sums
constexpr int FLASH_SMEM = OFF_XCH + 6 * BM * 4 + 1024;
static_assert(FLASH_SMEM <= 232448, "shared memory per CTA");
constexpr int FLASH_THREADS = 384;
constexpr uint32_t S_COL = 256;           // S/P buffers at TMEM columns 256 and 320
constexpr uint32_t Q_COL = 384;           // Q (the S MMAs' A operand): 128 columns of fp16 pairs
constexpr float kRescale = 8.0f;          // lazy rescale threshold (base-2 units)

// 2^x by the hardware's approximate exp2 (PTX ex2.approx.ftz.f32, subnormal results flushed
// to zero): P is rounded to fp16 right after, a far larger error than the approximation's.
// 2^-inf = 0 for masked scores.
__device__ __forceinline__ float ex2_fast(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__global__ void __launch_bounds__(FLASH_THREADS, 1) flash_tc_kernel(
    const __half* __restrict__ q, int64_t ldq, const __grid_constant__ CUtensorMap tk,
    const __grid_constant__ CUtensorMap tv, const __half* __restrict__ gate, int64_t ldg,
    __half* __restrict__ out, int64_t ldo, int L, int pos0, unsigned* status) {
  pdl_trigger();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pblk = gridDim.x - 1 - blockIdx.x;  // heavy (late) position blocks first
  const int p0 = pblk * POS;
  const int g = blockIdx.y % HKV;
  const int b = blockIdx.y / HKV;
  const int tb = b * L;                          // first query row of the request
  const int last_pos = min(p0 + POS, L) - 1;     // query positions are pos0 + local position
  const int nt = (pos0 + last_pos) / TBN + 1;

  const uint32_t bar_q = sb + OFF_BAR;              // Q written into tensor memory
  const uint32_t bar_kf = bar_q + 8;                // [KST] K tile landed
  const uint32_t bar_ke = bar_kf + 8 * KST;         // [KST] S MMAs done with a K stage
  const uint32_t bar_vf = bar_ke + 8 * KST;         // [VST] V tile landed
  const uint32_t bar_ve = bar_vf + 8 * VST;         // [VST] P V MMAs done with a V stage
  const uint32_t bar_s = bar_ve + 8 * VST;          // [2] S_j complete
  const uint32_t bar_p = bar_s + 16;                // [2] P_j written
  const uint32_t bar_pf = bar_p + 16;               // [2] P_j V_j done (S/P buffer free)
  const uint32_t bar_fin = bar_pf + 16;             // the last P V done
  const uint32_t bar_sfin = bar_fin + 8;            // the last S done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_SLOT);

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 8);  // the 8 warps that write Q into tensor memory
    for (int i = 0; i < KST; ++i) {
      mbar_init(bar_kf + 8 * i, 1);
      mbar_init(bar_ke + 8 * i, 1);
    }
    for (int i = 0; i < VST; ++i) {
      mbar_init(bar_vf + 8 * i, 1);
      mbar_init(bar_ve + 8 * i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_s + 8 * i, 1);
      mbar_init(bar_p + 8 * i, 4);   // the 4 warps of the group that owns buffer i
      mbar_init(bar_pf + 8 * i, 1);
    }
    mbar_init(bar_fin, 1);
    mbar_init(bar_sfin, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tk);
    tma_prefetch_desc(&tv);
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

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------------------------ TMA producers
    if (lane == 0) {
      const bool kside = warp == 0;
      const int nst = kside ? KST : VST;
      const uint32_t bf = kside ? bar_kf : bar_vf, be = kside ? bar_ke : bar_ve;
      const uint32_t base = sb + (kside ? OFF_K : OFF_V);
      const CUtensorMap* map = kside ? &tk : &tv;
      int issued = 0;
      for (int j = 0; j < nt; ++j) {
        const int st = j % nst;
        if (j >= nst &&
            !mbar_wait(be + 8 * st, (uint32_t)((j - nst) / nst) & 1, status, DEV_TIMEOUT_TMA))
          break;
        mbar_arrive_expect_tx(bf + 8 * st, KV_BYTES);
        for (int blk = 0; blk < 4; ++blk)
          tma_load_4d(base + st * KV_BYTES + blk * KV_BLOCK, map, bf + 8 * st, blk * 64, g,
                      j * TBN, b);
        issued = j + 1;
      }
      // copies still in flight land before the CTA may exit (no later phase of these barriers
      // can complete, so the parity tests are unambiguous)
      for (int j = issued > nst ? issued - nst : 0; j < issued; ++j)
        mbar_wait(bf + 8 * (j % nst), (uint32_t)(j / nst) & 1, status, DEV_TIMEOUT_TMA);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ S MMAs
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16_f32(128, TBN);
      bool ok = mbar_wait(bar_q, 0, status, DEV_TIMEOUT_MMA);
      for (int j = 0; j < nt && ok; ++j) {
        const int sk = j % KST, s = j & 1;
        ok = mbar_wait(bar_kf + 8 * sk, (uint32_t)(j / KST) & 1, status, DEV_TIMEOUT_MMA);
        // buffer s holds P_{j-2} until P_{j-2} V_{j-2} is done (P_j V_j cannot be done yet, so
        // the parity test is unambiguous)
        if (ok && j >= 2)
          ok = mbar_wait(bar_pf + 8 * s, (uint32_t)((j - 2) >> 1) & 1, status, DEV_TIMEOUT_MMA);
        if (!ok) break;
        tc_fence_after();
        // one descriptor per tile, the 16 slices by constant offsets of its start-address field
        // (building each from the address costs the issuing thread more than an N = 64 MMA runs)
        const uint64_t kd = sdesc_k_sw128(sb + OFF_K + sk * KV_BYTES);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          tc_mma_f16_ts(tmem + S_COL + s * TBN, tmem + Q_COL + kk * 8,
                        kd + (uint64_t)(((kk >> 2) * KV_BLOCK + (kk & 3) * 32) >> 4), idesc_s, kk != 0);
        tc_commit(bar_s + 8 * s);
        tc_commit(bar_ke + 8 * sk);
      }
      // tensor memory is freed only after every MMA issued here has completed
      tc_commit(bar_sfin);
      mbar_wait(bar_sfin, 0, status, DEV_TIMEOUT_MMA);
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------------ P V MMAs
    if (lane == 0) {
      constexpr uint32_t idesc_o = idesc_f16_f32(128, D, 0, 1);
      bool ok = true;
      for (int j = 0; j < nt && ok; ++j) {
        const int sv = j % VST, s = j & 1;
        ok = mbar_wait(bar_p + 8 * s, (uint32_t)(j >> 1) & 1, status, DEV_TIMEOUT_MMA) &&
             mbar_wait(bar_vf + 8 * sv, (uint32_t)(j / VST) & 1, status, DEV_TIMEOUT_MMA);
        if (!ok) break;
        tc_fence_after();
        const uint64_t vd = sdesc_mn_sw128(sb + OFF_V + sv * KV_BYTES, KV_BLOCK, 1024);
#pragma unroll
        for (int kk = 0; kk < TBN / 16; ++kk)
          tc_mma_f16_ts(tmem, tmem + S_COL + s * TBN + kk * 8, vd + (uint64_t)((kk * 16 * 128) >> 4),
                        idesc_o, (j | kk) != 0);
        tc_commit(bar_pf + 8 * s);
        tc_commit(bar_ve + 8 * sv);
      }
      // the epilogue waits for the last P V; tensor memory is freed only after every MMA
      // issued here has completed
      tc_commit(bar_fin);
      mbar_wait(bar_fin, 0, status, DEV_TIMEOUT_MMA);
    }
  } else if (warp >= 4) {
    const int quarter = warp & 3;
    const int grp = (warp - 4) >> 2;                   // 0: even tiles (S buffer 0), 1: odd tiles
    const int r = quarter * 32 + lane;                 // row of this thread
    const int pos = p0 + (r >> 2);
    const uint32_t tl = tmem + ((uint32_t)(quarter * 32) << 16);
    float* xm = reinterpret_cast<float*>(smem + OFF_XCH);   // [row] reference max handed over
    float* xl = xm + BM;                                     // [group][row] row sums
    float* xr = xl + 2 * BM;                                 // [group][row] their references
    float* xf = xr + 2 * BM;                                 // [row] reference after the last tile
    const float sl2 = 0.0625f * 1.4426950408889634f;  // 1/sqrt(256) in base 2
    // named barriers of the two warps on lane quarter q (64 threads): 1 + q both ways at the
    // end; 5 + q carries the reference max from the even-tile group to the odd-tile group,
    // 9 + q back
    const int bar_send = (grp == 0 ? 5 : 9) + quarter;
    const int bar_recv = (grp == 0 ? 9 : 5) + quarter;
    auto pair_sync = [&]() { asm volatile("bar.sync %0, 64;" ::"r"(1 + quarter) : "memory"); };
    {
      // Q into tensor memory: row r, column Q_COL + c holds dims 2c, 2c+1 (the A-operand layout
      // of kind::f16); this thread writes its row's dims 128 grp .. 128 grp + 127
      const bool valid = pos < L;
      const __half* qrow = q + ((int64_t)tb + (valid ? pos : 0)) * ldq + (4 * g + (r & 3)) * D + grp * 128;
#pragma unroll 1
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t qv[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 d = valid ? __ldg(reinterpret_cast<const uint4*>(qrow + 2 * c0) + i)
                                : make_uint4(0u, 0u, 0u, 0u);
          qv[4 * i] = d.x;
          qv[4 * i + 1] = d.y;
          qv[4 * i + 2] = d.z;
          qv[4 * i + 3] = d.w;
        }
        tmem_st_32x32b_x32(tl + Q_COL + grp * 64 + c0, qv);
      }
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_q);
    }
    // keys of tiles before this one are all at or before the CTA's first position: no mask
    const int p_first = pos0 + p0;
    const int qpos = pos0 + pos;                        // this row's position in the request
    float m_ref = -INFINITY;   // reference max of the raw scores (P = 2^((s - m_ref) sl2))
    float m_l = -INFINITY;     // the reference this group's row sum is relative to
    float lsum = 0.f;
    // Both warps of a lane quarter pass the same named barriers whatever happens: a failed
    // (timed-out) wait only turns the rest of the work off (ok is warp-uniform).
    bool ok = true;
    for (int j = grp; j < nt; j += 2) {
      const int s = grp;                                // tile j's S/P buffer
      ok = ok && mbar_wait(bar_s + 8 * s, (uint32_t)(j >> 1) & 1, status, DEV_TIMEOUT_EPILOGUE);
      ok = __all_sync(0xffffffffu, ok);
      uint32_t sv0[32], sv1[32];                        // keys 0..31 and 32..63 of the tile
      float mt = -INFINITY;
      if (ok) {
        tc_fence_after();
        tmem_ld_32x32b_x32(tl + S_COL + s * TBN, sv0);
        tmem_ld_32x32b_x32(tl + S_COL + s * TBN + 32, sv1);
        tc_wait_ld();
        const int key0 = j * TBN;
        if (key0 + TBN - 1 > p_first) {
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (key0 + c > qpos) sv0[c] = __float_as_uint(-INFINITY);
            if (key0 + 32 + c > qpos) sv1[c] = __float_as_uint(-INFINITY);
          }
        }
        // four independent max chains
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          m4[(c >> 1) & 1] = fmaxf(m4[(c >> 1) & 1], fmaxf(__uint_as_float(sv0[c]), __uint_as_float(sv0[c + 1])));
          m4[2 + ((c >> 1) & 1)] = fmaxf(m4[2 + ((c >> 1) & 1)],
                                        fmaxf(__uint_as_float(sv1[c]), __uint_as_float(sv1[c + 1])));
        }
        mt = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      }
      // the reference after tile j - 1, from the other group
      if (j >= 1) {
        asm volatile("bar.sync %0, 64;" ::"r"(bar_recv) : "memory");
        m_ref = xm[r];
      }
      const float m_prev = m_ref;                       // the reference O is relative to
      const float m_new = fmaxf(m_prev, mt);
      const bool need = ok && (m_new - m_prev) * sl2 > kRescale;
      if (need) m_ref = m_new;
      // the other group's next tile may start its exponentials now
      if (j + 1 < nt) {
        xm[r] = m_ref;
        asm volatile("bar.arrive %0, 64;" ::"r"(bar_send) : "memory");
      }
      if (!ok) continue;
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O may only be rescaled once P_{j-1} V_{j-1} has landed in it (P_j V_j cannot have
        // been issued yet, so the parity test is unambiguous)
        const int jp = j - 1;
        ok = __all_sync(0xffffffffu, mbar_wait(bar_pf + 8 * (jp & 1), (uint32_t)(jp >> 1) & 1,
                                               status, DEV_TIMEOUT_EPILOGUE));
        if (!ok) continue;
        tc_fence_after();
        const float f = need ? exp2f((m_prev - m_new) * sl2) : 1.f;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          uint32_t ov[32];
          tmem_ld_32x32b_x32(tl + c0, ov);
          tc_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * f);
          tmem_st_32x32b_x32(tl + c0, ov);
        }
        tc_wait_st();
      }
      // this group's row sum follows the reference
      if (m_ref != m_l) {
        if (lsum > 0.f) lsum *= exp2f((m_l - m_ref) * sl2);
        m_l = m_ref;
      }
      // P = 2^(s sl2 - m_ref sl2): one FFMA and one exp2 per score
      const float moff = -m_ref * sl2;
      uint32_t pk[32];
      float rs[4] = {0.f, 0.f, 0.f, 0.f};   // four independent sum chains
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const float e0 = ex2_fast(fmaf(__uint_as_float(sv0[2 * c]), sl2, moff));
        const float e1 = ex2_fast(fmaf(__uint_as_float(sv0[2 * c + 1]), sl2, moff));
        const float e2 = ex2_fast(fmaf(__uint_as_float(sv1[2 * c]), sl2, moff));
        const float e3 = ex2_fast(fmaf(__uint_as_float(sv1[2 * c + 1]), sl2, moff));
        rs[c & 1] += e0 + e1;
        rs[2 + (c & 1)] += e2 + e3;
        pk[c] = pack_half2(e0, e1);
        pk[16 + c] = pack_half2(e2, e3);
      }
      lsum += (rs[0] + rs[1]) + (rs[2] + rs[3]);
      tmem_st_32x32b_x32(tl + S_COL + s * TBN, pk);
      tc_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p + 8 * s);
    }
    // the two groups' row sums, each brought to the reference of the last tile (the one O is
    // relative to); then O / l * sigmoid(gate), each thread of a row taking half of its columns
    if (grp == ((nt - 1) & 1)) xf[r] = m_ref;
    xl[grp * BM + r] = lsum;
    xr[grp * BM + r] = m_l;
    pair_sync();
    const float m_fin = xf[r];
    float l = 0.f;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const float lh = xl[h * BM + r];
      if (lh > 0.f) l += lh * exp2f((xr[h * BM + r] - m_fin) * sl2);
    }
    if (ok && mbar_wait(bar_fin, 0, status, DEV_TIMEOUT_EPILOGUE)) {
      tc_fence_after();
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int hq = 4 * g + (r & 3);
      const int64_t row = (int64_t)tb + pos;
#pragma unroll 1
      for (int c0 = grp * (D / 2); c0 < (grp + 1) * (D / 2); c0 += 32) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tl + c0, ov);
        tc_wait_ld();
        if (pos < L) {
          uint32_t pkd[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            float a0 = __uint_as_float(ov[2 * c]) * inv, a1 = __uint_as_float(ov[2 * c + 1]) * inv;
            if (gate) {
              const float2 gf = __half22float2(
                  *reinterpret_cast<const __half2*>(gate + row * ldg + hq * D + c0 + 2 * c));
              a0 *= sigmoid_f(gf.x);
              a1 *= sigmoid_f(gf.y);
            }
            pkd[c] = pack_half2(a0, a1);
          }
          uint4* dst = reinterpret_cast<uint4*>(out + row * ldo + hq * D + c0);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            dst[c] = make_uint4(pkd[4 * c], pkd[4 * c + 1], pkd[4 * c + 2], pkd[4 * c + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Rows of one request chunk into a cache: dst row (request * dctx + pos0 + t) <- src row
// (request * L + t), `cols` fp16 per row (a multiple of 8), 16 bytes per thread.
__global__ void kv_store_kernel(const __half* __restrict__ src, int64_t lds, __half* __restrict__ dst,
                                int64_t ldd, int64_t M, int L, int pos0, int64_t dctx, int cols) {
  pdl_trigger();
  pdl_wait();
  const int per_row = cols / 8;
  const int64_t n = M * per_row;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tok = i / per_row;
    const int c8 = (int)(i % per_row) * 8;
    const int64_t drow = (tok / L) * dctx + pos0 + tok % L;
    *reinterpret_cast<uint4*>(dst + drow * ldd + c8) =
        *reinterpret_cast<const uint4*>(src + tok * lds + c8);
  }
}

}  // namespace attn

clef_status rope_launch(const __half* qin, int64_t ldqi, __half* qout, int64_t ldqo,
                        const __half* kin, int64_t ldki, __half* kout, int64_t ldko, int64_t M,
                        int64_t L, int64_t pos0, int64_t kctx, cudaStream_t stream,
                        const MRope& mr) {
  if (M == 0) return CLEF_OK;
  static const attn::RopeFreq fr = [] {
    attn::RopeFreq f;
    for (int j = 0; j < 32; ++j) f.f[j] = std::exp(-(double)j * (std::log(1e7) / 32.0));
    return f;
  }();
  // rows are read and written with 16-byte accesses
  const auto mis = [](const void* p, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(p) & 15) != 0 || (ld & 7) != 0;
  };
  if (mis(qin, ldqi) || mis(qout, ldqo) || mis(kin, ldki) || mis(kout, ldko)) return CLEF_E_ALIGN;
  TraceScope ts(stream, "rope", 0.0, M * (20.0 * 64 * 2 * 2));
  CLEF_CUDA_CHECK(launch_pdl(attn::rope_kernel, dim3((unsigned)M), dim3(96), 0, stream,
       qin, ldqi, qout, ldqo, kin, ldki, kout, ldko,
       (int)L, (int)pos0, kctx, (int)mr.start,
       (int)mr.h, (int)mr.w, fr));
  return CLEF_OK;
}

clef_status flash_launch(const __half* q, int64_t ldq, const __half* k, int64_t ldk,
                         const __half* v, int64_t ldv, const __half* gate, int64_t ldg, __half* out,
                         int64_t ldo, int64_t B, int64_t L, int64_t pos0, int64_t kv_req,
                         cudaStream_t stream) {
  if (B == 0 || L == 0) return CLEF_OK;
  static std::atomic<uint64_t> attr{0};
  CLEF_CUDA_CHECK(smem_opt_in((const void*)attn::flash_tc_kernel, attn::FLASH_SMEM, &attr));
  // Q rows are read with 16-byte loads; K and V by TMA (row strides a multiple of 16 bytes)
  if ((reinterpret_cast<uintptr_t>(q) & 15) != 0 || (ldq & 7) != 0 ||
      (reinterpret_cast<uintptr_t>(k) & 15) != 0 || (ldk & 7) != 0 ||
      (reinterpret_cast<uintptr_t>(v) & 15) != 0 || (ldv & 7) != 0)
    return CLEF_E_ALIGN;
  CUtensorMap mk, mv;
  {
    // keys and values [B][kv_req rows][4 heads][256]; only positions below pos0 + L are in the
    // map, so a key tile's rows past them read zero
    const uint64_t dims[4] = {256, 4, (uint64_t)(pos0 + L), (uint64_t)B};
    const uint32_t box[4] = {64, 1, attn::TBN, 1};
    const uint64_t stk[3] = {512, (uint64_t)ldk * 2, (uint64_t)kv_req * ldk * 2};
    const uint64_t stv[3] = {512, (uint64_t)ldv * 2, (uint64_t)kv_req * ldv * 2};
    if (tma_encode(&mk, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, k, dims, stk, box,
                   CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess ||
        tma_encode(&mv, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, v, dims, stv, box,
                   CU_TENSOR_MAP_SWIZZLE_128B) != cudaSuccess)
      return CLEF_E_CUDA;
  }
  dim3 grid((unsigned)((L + attn::POS - 1) / attn::POS), (unsigned)(B * attn::HKV));
  TraceScope ts(stream, "flash_attn",
                4.0 * attn::D * attn::HQ * (double)B * ((double)L * pos0 + (double)L * (L + 1) / 2.0),
                (double)B * L * (16 + 16 + 16) * attn::D * 2.0 + (double)B * (pos0 + L) * 8 * attn::D * 2.0);
  CLEF_CUDA_CHECK(launch_pdl(attn::flash_tc_kernel, dim3(grid), dim3(attn::FLASH_THREADS), attn::FLASH_SMEM, stream,
       q, ldq, mk, mv, gate, ldg, out, ldo, (int)L, (int)pos0, status_word_ptr()));
  return CLEF_OK;
}

clef_status kv_store_launch(const __half* src, int64_t lds, __half* dst, int64_t ldd, int64_t M,
                            int64_t L, int64_t pos0, int64_t dctx, int cols, cudaStream_t stream) {
  if (M == 0) return CLEF_OK;
  TraceScope ts(stream, "kv_store", 0.0, (double)M * cols * 4.0);
  const int64_t n = M * (cols / 8);
  const unsigned grid = (unsigned)std::min<int64_t>((n + 255) / 256, 4096);
  CLEF_CUDA_CHECK(launch_pdl(attn::kv_store_kernel, dim3(grid), dim3(256), 0, stream,
       src, lds, dst, ldd, M, (int)L, (int)pos0, dctx, cols));
  return CLEF_OK;
}

}  // namespace clef
