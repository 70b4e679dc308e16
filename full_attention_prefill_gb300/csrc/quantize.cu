// LUT-6 quantiser: fp16 weight W [n, k] -> packed 6-bit indices + an fp16 table of 64 values for
// each block of 16 output channels ("Clef-Flash-ANE-LUT6" model card, section "LUT-6 text weights": per 16-row
// group, 40 k-means iterations in one dimension from 64 initial centroids, 32 quantiles of the
// group and 32 equal steps from its smallest to its largest weight).
//
// GB300 design.  Every fp16 value maps to a 16-bit key that orders like the value (negative
// patterns reversed below the positive ones), so a group's weights are summarised exactly by a
// histogram over the 65,536 keys.  One thread-block cluster of 4 CTAs owns a group: CTA q keeps
// the counts of keys [16384 q, 16384 q + 16384) in its shared memory (64 KB) with exclusive
// prefix counts and prefix sums per 32-key block, and reads the other quarters through
// distributed shared memory.  With that summary every step of the method is a handful of
// lookups instead of a pass over the weights:
//   * the order statistics behind the quantiles: a binary search over the block prefixes, then
//     a scan of one block;
//   * a k-means round: with ascending centroids the cell of centroid j is the key range between
//     the first keys above the midpoints of its neighbours, so the count and the sum of its
//     members are two prefix lookups.  Sums are exact integers (fp16 values are multiples of
//     2^-24), so the new centroid fl(fl(S) / count) * 2^-24 has one rounding, as in the oracle.
//     A run of equal centroids gives all its cells to its first member, which moves alone, so
//     the 64 centroids are sorted again (stable) after every round;
//   * the final indices: one pass over the group, each weight's index found among 63 sorted
//     threshold keys, packed four to three bytes.
// The weights are read from HBM twice per group (histogram, then indices; the second read mostly
// hits L2) and written once as 0.75 bytes per weight.  The 40 rounds are latency bound (a few
// shared-memory and DSMEM lookups and 64 fp64 divisions each) and run in CTA 0 of the cluster
// alone; 76 KB of shared memory per CTA lets CTAs of three clusters share an SM to hide that
// latency.  This part's fp64 pipe is narrow, so comparisons of centroids use integer keys.
#include <cooperative_groups.h>

#include "common.cuh"

namespace cg = cooperative_groups;

namespace clef {
namespace quant {

constexpr int CL = 4;                   // CTAs per cluster, one key quarter each
constexpr int QKEYS = 16384;            // keys per quarter
constexpr int BK = 32;                  // keys per prefix block
constexpr int NB = QKEYS / BK;          // 512 prefix blocks per quarter
constexpr int THREADS = 256;
constexpr int UNR = 4;                  // 16-byte loads in flight per thread in the histogram pass
constexpr int ROUNDS = 40;
constexpr int TS = 64;                  // table entries
constexpr uint32_t KEY_END = 65536u;

struct Smem {
  uint32_t hist[QKEYS];                 // counts of this CTA's quarter
  uint32_t bcnt[NB + 1];                // exclusive prefix counts of 32-key blocks; [NB] = total
  long long bsum[NB + 1];               // exclusive prefix sums (units of 2^-24)
  double c[2][TS];                      // centroids, ascending; moved centroids
  long long okey[2][TS];                // integer order keys of c[0], of the moved centroids
  double seed[TS];
  uint32_t fcnt[TS + 1];                // prefix count at the cell thresholds
  long long fsum[TS + 1];
  uint32_t qcnt[CL + 1];                // counts below each quarter; [CL] = n
  long long qsum[CL + 1];
  uint32_t wcnt[THREADS / 32];          // scan scratch
  long long wsum[THREADS / 32];
  double xval[2 * (TS / 2) + 2];        // order statistics for the seeds
  uint32_t pcnt[TS];                    // the (count, sum) each centroid was last computed from
  long long psum[TS];                   // (count ~0: none, or its slot has changed since)
  uint16_t tkey[TS];                    // final thresholds
  uint8_t first[TS];                    // first index of each run of equal table values
  int nonfinite;
};

// three CTAs per SM: 233,472 bytes of shared memory per SM, 1 KB reserved per CTA
static_assert(sizeof(Smem) + 1024 <= 233472 / 3, "three CTAs per SM");

// ---- keys ----
__device__ __forceinline__ uint32_t key_of(uint32_t h) {
  return (h & 0x8000u) ? (0xFFFFu - h) : (h + 0x8000u);
}
__device__ __forceinline__ uint32_t bits_of(uint32_t key) {
  return key >= 0x8000u ? key - 0x8000u : 0xFFFFu - key;
}
// value in units of 2^-24 (exact integer for every finite fp16)
__device__ __forceinline__ long long key_fixed(uint32_t key) {
  const uint32_t h = bits_of(key);
  const uint32_t e = (h >> 10) & 31u, m = h & 1023u;
  const long long mag = e ? ((long long)(1024u | m) << (e - 1)) : (long long)m;
  return (h & 0x8000u) ? -mag : mag;
}
// A 32-key block never crosses an fp16 binade, so inside it the value is linear in the key:
// key_fixed(key0 + i) = key_fixed(key0) + i * key_step(key0) (both signs, subnormals included).
__device__ __forceinline__ long long key_step(uint32_t key0) {
  const uint32_t e = (bits_of(key0) >> 10) & 31u;
  return e >= 2 ? (1ll << (e - 1)) : 1ll;
}
__device__ __forceinline__ double key_value(uint32_t key) {
  return (double)__half2float(__ushort_as_half((unsigned short)bits_of(key)));
}
// The first key whose value is above b (|b| <= 65504), from the bits of b with integer
// operations only: t = the largest fp16 magnitude <= |b| (the significand cut to 10 bits, or to
// units of 2^-24 below 2^-14), exact when nothing was cut.  b > 0: the key after +t.  b < 0: the
// key of -t (its value is above b) unless -t == b, then the one after; -0 and +0 share one value.
__device__ __forceinline__ uint32_t first_key_above(double b) {
  const unsigned long long bits = (unsigned long long)__double_as_longlong(b);
  const unsigned long long m52 = bits & ((1ull << 52) - 1);
  const int ebits = (int)((bits >> 52) & 0x7FF);
  if (ebits == 0 && m52 == 0) return 0x8001u;
  const int E = ebits - 1023;
  uint32_t t;
  bool exact;
  if (E >= -14) {
    if (E > 15) {
      t = 0x7BFFu;
      exact = false;
    } else {
      t = ((uint32_t)(E + 15) << 10) | (uint32_t)(m52 >> 42);
      exact = (m52 & ((1ull << 42) - 1)) == 0;
    }
  } else {
    const unsigned long long sig = (1ull << 52) | m52;
    const int shift = 28 - E;
    if (shift >= 64) {
      t = 0;
      exact = false;
    } else {
      t = (uint32_t)(sig >> shift);
      exact = (sig & ((1ull << shift) - 1)) == 0;
    }
  }
  if (!(bits >> 63)) return t + 0x8000u + 1u;
  if (t == 0) return 0x7FFFu;
  const uint32_t k = 0xFFFFu - (0x8000u | t);
  return exact ? k + 1u : k;
}

// Integer key ordered like the double x, with -0 and +0 equal (sorting on the fp64 pipe of
// this part would cost ~16 cycles per warp compare).
__device__ __forceinline__ long long order_key(double x) {
  long long b = __double_as_longlong(x);
  if (b == (long long)0x8000000000000000ull) b = 0;
  return b < 0 ? (b ^ 0x7FFFFFFFFFFFFFFFll) : b;
}

// Address of `p`'s counterpart in the shared memory of cluster CTA q (distributed shared memory).
template <class T>
__device__ __forceinline__ const T* in_cta(const T* p, uint32_t q) {
  return cg::this_cluster().map_shared_rank(const_cast<T*>(p), q);
}

// Count and sum of the group's weights with key < u (u in [0, 65536]).
__device__ __forceinline__ void prefix_at(const Smem& sm, uint32_t u,
                                          uint32_t& cnt, long long& sum) {
  if (u >= KEY_END) {
    cnt = sm.qcnt[CL];
    sum = sm.qsum[CL];
    return;
  }
  const uint32_t q = u >> 14, local = u & (QKEYS - 1), b = local >> 5, off = local & 31u;
  cnt = sm.qcnt[q] + in_cta(sm.bcnt, q)[b];
  sum = sm.qsum[q] + in_cta(sm.bsum, q)[b];
  const uint4* blk = reinterpret_cast<const uint4*>(in_cta(sm.hist, q) + b * BK);
  uint4 v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = blk[i];
  const uint32_t* c = reinterpret_cast<const uint32_t*>(v);
  uint32_t n = 0, in = 0;   // count and first moment (sum of i * c_i) of keys key0 .. key0 + off - 1
#pragma unroll
  for (uint32_t i = 0; i < 32; ++i) {
    const uint32_t ci = i < off ? c[i] : 0u;
    n += ci;
    in += i * ci;
  }
  const uint32_t key0 = (q << 14) | (b << 5);
  cnt += n;
  sum += key_fixed(key0) * (long long)n + key_step(key0) * (long long)in;
}

// Value of the weight of rank r (0-based) in ascending order.
__device__ __forceinline__ double value_at_rank(const Smem& sm, uint32_t r) {
  // largest global block B (32 keys each, 2048 in all) whose start count is <= r
  uint32_t lo = 0, hi = CL * NB;   // invariant: start(lo) <= r < start(hi) (start(2048) = n)
  while (hi - lo > 1) {
    const uint32_t mid = (lo + hi) >> 1;
    const uint32_t q = mid / NB, b = mid % NB;
    if (sm.qcnt[q] + in_cta(sm.bcnt, q)[b] <= r) lo = mid; else hi = mid;
  }
  const uint32_t q = lo / NB, b = lo % NB;
  uint32_t run = sm.qcnt[q] + in_cta(sm.bcnt, q)[b];
  const uint32_t* h = in_cta(sm.hist, q) + b * BK;
  uint32_t key = lo * BK;
  for (int i = 0; i < BK - 1; ++i) {
    run += h[i];
    if (run <= r) key = lo * BK + i + 1; else break;
  }
  return key_value(key);
}

__global__ void __cluster_dims__(CL, 1, 1) __launch_bounds__(THREADS, 3)
    quantize_kernel(const __half* __restrict__ w, int64_t n, int64_t k, uint8_t* __restrict__ packed,
                    __half* __restrict__ lut, unsigned* status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  cg::cluster_group cl = cg::this_cluster();
  const uint32_t rank = cl.block_rank();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) sm.nonfinite = 0;

  const int64_t groups = n / 16, k4 = k / 4, row_bytes = k4 * 3;
  const int64_t cid = blockIdx.x / CL, ncl = gridDim.x / CL;
  for (int64_t g = cid; g < groups; g += ncl) {
    // every CTA has finished reading the other quarters of the previous group
    cl.sync();
    for (int i = tid; i < QKEYS / 4; i += THREADS)
      reinterpret_cast<uint4*>(sm.hist)[i] = make_uint4(0, 0, 0, 0);
    __syncthreads();

    // ---- histogram of this CTA's quarter ----
    // the group's 16 rows are one contiguous run of 16 k values (2 k 16-byte vectors)
    const __half* wg = w + g * 16 * k;
    const uint4* wv = reinterpret_cast<const uint4*>(wg);
    const int64_t nvec = 2 * k;
    bool bad = false;
    for (int64_t v0 = tid; v0 < nvec; v0 += UNR * THREADS) {
      uint4 d[UNR];
#pragma unroll
      for (int j = 0; j < UNR; ++j) {
        const int64_t v = v0 + (int64_t)j * THREADS;
        d[j] = v < nvec ? wv[v] : make_uint4(0x7C007C00u, 0x7C007C00u, 0x7C007C00u, 0x7C007C00u);
      }
#pragma unroll
      for (int j = 0; j < UNR; ++j) {
        if (v0 + (int64_t)j * THREADS >= nvec) break;
        const uint32_t words[4] = {d[j].x, d[j].y, d[j].z, d[j].w};
#pragma unroll
        for (int x = 0; x < 8; ++x) {
          const uint32_t h = (words[x >> 1] >> (16 * (x & 1))) & 0xFFFFu;
          if ((h & 0x7C00u) == 0x7C00u) { bad = true; continue; }
          const uint32_t key = key_of(h);
          if ((key >> 14) == rank) atomicAdd(&sm.hist[key & (QKEYS - 1)], 1u);
        }
      }
    }
    if (bad) sm.nonfinite = 1;
    __syncthreads();

    // ---- per-block totals (lanes rotate over the block's keys: no bank conflicts) ----
    for (int b = tid; b < NB; b += THREADS) {
      uint32_t cnt = 0, in = 0;
      for (int i = 0; i < BK; ++i) {
        const int j = (i + lane) & (BK - 1);
        const uint32_t c = sm.hist[b * BK + j];
        cnt += c;
        in += (uint32_t)j * c;
      }
      const uint32_t key0 = (rank << 14) | (uint32_t)(b * BK);
      sm.bcnt[b] = cnt;
      sm.bsum[b] = key_fixed(key0) * (long long)cnt + key_step(key0) * (long long)in;
    }
    __syncthreads();
    // ---- exclusive scan of the 512 block totals (2 per thread) ----
    {
      const uint32_t c0 = sm.bcnt[2 * tid], c1 = sm.bcnt[2 * tid + 1];
      const long long s0 = sm.bsum[2 * tid], s1 = sm.bsum[2 * tid + 1];
      uint32_t ic = c0 + c1;
      long long is = s0 + s1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t oc = __shfl_up_sync(0xffffffffu, ic, o);
        const long long os = __shfl_up_sync(0xffffffffu, is, o);
        if (lane >= o) { ic += oc; is += os; }
      }
      if (lane == 31) { sm.wcnt[warp] = ic; sm.wsum[warp] = is; }
      __syncthreads();
      uint32_t bc = 0;
      long long bs = 0;
      for (int i = 0; i < warp; ++i) { bc += sm.wcnt[i]; bs += sm.wsum[i]; }
      const uint32_t ex_c = bc + ic - (c0 + c1);
      const long long ex_s = bs + is - (s0 + s1);
      sm.bcnt[2 * tid] = ex_c;
      sm.bsum[2 * tid] = ex_s;
      sm.bcnt[2 * tid + 1] = ex_c + c0;
      sm.bsum[2 * tid + 1] = ex_s + s0;
      if (tid == THREADS - 1) { sm.bcnt[NB] = bc + ic; sm.bsum[NB] = bs + is; }
    }
    // every quarter's prefixes are complete
    cl.sync();
    if (tid == 0) {
      uint32_t c = 0;
      long long s = 0;
      for (int q = 0; q < CL; ++q) {
        sm.qcnt[q] = c;
        sm.qsum[q] = s;
        c += in_cta(sm.bcnt, q)[NB];
        s += in_cta(sm.bsum, q)[NB];
      }
      sm.qcnt[CL] = c;
      sm.qsum[CL] = s;
    }
    __syncthreads();
    const uint32_t ntot = sm.qcnt[CL];

    // CTA 0 alone finds the table (the others wait): the rounds are latency bound, and
    // repeating them in every CTA would only load the SM's fp64 pipe three more times
    if (rank == 0) {
    if (ntot == 0) {
      // no finite weight: an all-zero table (the status word reports the input)
      if (tid < TS) sm.c[0][tid] = 0.0;
    } else {
      // ---- seeds: order statistics for the 32 quantiles, the minimum and the maximum ----
      // quantile i sits at h = (n - 1)(2i + 1) / 64 between ranks floor(h) and floor(h) + 1
      if (tid < TS + 2) {
        uint32_t r;
        if (tid < TS) {
          const uint64_t num = (uint64_t)(ntot - 1) * (uint64_t)(2 * (tid >> 1) + 1);
          r = (uint32_t)(num >> 6) + (tid & 1);
          if (r > ntot - 1) r = ntot - 1;
        } else {
          r = tid == TS ? 0u : ntot - 1;
        }
        sm.xval[tid] = value_at_rank(sm, r);
      }
      __syncthreads();
      if (tid < TS / 2) {
        const uint64_t num = (uint64_t)(ntot - 1) * (uint64_t)(2 * tid + 1);
        const double f = (double)(num & 63u) * (1.0 / 64.0);
        const double a = sm.xval[2 * tid], b = sm.xval[2 * tid + 1];
        // exact for fp16 data; evaluated as written, also for f = 0, so a zero keeps the sign
        // IEEE addition gives it (-0 + 0 = +0)
        sm.seed[tid] = __dadd_rn(a, __dmul_rn(f, __dsub_rn(b, a)));
      } else if (tid < TS) {
        const int i = tid - TS / 2;
        const double mn = sm.xval[TS], mx = sm.xval[TS + 1];
        const double step = __ddiv_rn(mx - mn, (double)(TS / 2 - 1));
        sm.seed[tid] = i == TS / 2 - 1 ? mx : __dadd_rn(__dmul_rn((double)i, step), mn);
      }
      __syncthreads();
      // stable sort of the 64 seeds (equal values, -0 and +0 too, by position) on integer keys
      if (tid < TS) sm.okey[1][tid] = order_key(sm.seed[tid]);
      __syncthreads();
      if (tid < TS) {
        const long long o = sm.okey[1][tid];
        int pos = 0;
        for (int i = 0; i < TS; ++i) {
          const long long x = sm.okey[1][i];
          pos += (x < o) || (x == o && i < tid);
        }
        sm.c[0][pos] = sm.seed[tid];
        sm.okey[0][pos] = o;
        sm.pcnt[tid] = 0xFFFFFFFFu;
      }
      __syncthreads();

      // ---- 40 rounds of k-means on the histogram ----
      // centroids live in c[0] (ascending) at the start of every round; c[1] takes the moved ones
      for (int it = 0; it < ROUNDS; ++it) {
        double* c = sm.c[0];
        double* cn = sm.c[1];
        if (tid < TS - 1) {
          const double mid = __dmul_rn(__dadd_rn(c[tid], c[tid + 1]), 0.5);
          uint32_t cnt;
          long long sum;
          prefix_at(sm, first_key_above(mid), cnt, sum);
          sm.fcnt[tid + 1] = cnt;
          sm.fsum[tid + 1] = sum;
        } else if (tid == TS - 1) {
          sm.fcnt[0] = 0;
          sm.fsum[0] = 0;
          sm.fcnt[TS] = ntot;
          sm.fsum[TS] = sm.qsum[CL];
        }
        __syncthreads();
        if (tid < TS) {
          // cell j holds the weights between thresholds j and j + 1; a run of equal centroids
          // gives all its cells to its first member
          const double cj = c[tid];
          const long long kj = sm.okey[0][tid];
          double out = cj;
          uint32_t pc = 0xFFFFFFFFu;
          long long ps = 0;
          if (tid == 0 || sm.okey[0][tid - 1] != kj) {
            int e = tid;
            while (e < TS - 1 && sm.okey[0][e + 1] == kj) ++e;
            const uint32_t cnt = sm.fcnt[e + 1] - sm.fcnt[tid];
            const long long sum = sm.fsum[e + 1] - sm.fsum[tid];
            if (cnt) {
              // the same members as when this centroid was computed give the same bits
              if (cnt != sm.pcnt[tid] || sum != sm.psum[tid])
                out = __dmul_rn(__ddiv_rn(__ll2double_rn(sum), (double)cnt), 0x1p-24);
              pc = cnt;
              ps = sum;
            }
          }
          sm.pcnt[tid] = pc;
          sm.psum[tid] = ps;
          cn[tid] = out;
          sm.okey[1][tid] = order_key(out);
        }
        __syncthreads();
        // equal centroids moved only their first member: sort again (stable); usually the
        // order has not changed and the sort is the identity
        const bool unsorted = tid > 0 && tid < TS && sm.okey[1][tid - 1] > sm.okey[1][tid];
        if (!__syncthreads_or(unsorted)) {
          if (tid < TS) {
            c[tid] = cn[tid];
            sm.okey[0][tid] = sm.okey[1][tid];
          }
        } else if (tid < TS) {
          sm.pcnt[tid] = 0xFFFFFFFFu;   // centroids change slots: compute every mean again
          const long long o = sm.okey[1][tid];
          int pos = 0;
          for (int i = 0; i < TS; ++i) {
            const long long x = sm.okey[1][i];
            pos += (x < o) || (x == o && i < tid);
          }
          c[pos] = cn[tid];
          sm.okey[0][pos] = o;
        }
        __syncthreads();
      }
    }

    // ---- table: centroids rounded to fp16; thresholds between neighbouring entries ----
    double* cfin = sm.c[0];
    if (tid < TS) {
      const __half t = __double2half(cfin[tid]);
      cfin[tid] = (double)__half2float(t);
      lut[g * TS + tid] = t;
    }
    __syncthreads();
    if (tid < TS) {
      if (tid < TS - 1)   // exact midpoint of two fp16 values
        sm.tkey[tid] = (uint16_t)min(first_key_above((cfin[tid] + cfin[tid + 1]) * 0.5), 0xFFFFu);
      int f = tid;
      while (f > 0 && cfin[f - 1] == cfin[tid]) --f;
      sm.first[tid] = (uint8_t)f;
    }
    }  // rank 0
    // CTA 0's thresholds are ready; the others copy them
    cl.sync();
    if (rank != 0 && tid < TS) {
      sm.tkey[tid] = in_cta(sm.tkey, 0)[tid];
      sm.first[tid] = in_cta(sm.first, 0)[tid];
    }
    __syncthreads();

    // ---- indices of this CTA's 4 rows, packed four to three bytes ----
    // this CTA's rows 4 rank .. 4 rank + 3 are contiguous in w (4 k values) and in packed (3 k
    // bytes): units of 16 values, two 16-byte loads in, three 4-byte words out
    const uint4* src = reinterpret_cast<const uint4*>(wg + (int64_t)rank * 4 * k);
    uint32_t* dst = reinterpret_cast<uint32_t*>(packed + (g * 16 + (int64_t)rank * 4) * row_bytes);
    for (int64_t u = tid; u < k4; u += THREADS) {
      const uint4 a = src[2 * u], b = src[2 * u + 1];
      const uint32_t words[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      uint32_t q[4] = {0, 0, 0, 0};   // four 24-bit quadruples
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        const uint32_t key = key_of((words[x >> 1] >> (16 * (x & 1))) & 0xFFFFu);
        uint32_t cell = 0;   // number of thresholds <= key (63 sorted thresholds)
#pragma unroll
        for (uint32_t step = 32; step; step >>= 1)
          if (sm.tkey[cell + step - 1] <= key) cell += step;
        q[x >> 2] |= (uint32_t)sm.first[cell] << (6 * (x & 3));
      }
      dst[3 * u + 0] = q[0] | (q[1] << 24);
      dst[3 * u + 1] = (q[1] >> 8) | (q[2] << 16);
      dst[3 * u + 2] = (q[2] >> 16) | (q[3] << 8);
    }
  }
  // no CTA leaves while another may still read its shared memory
  cl.sync();
  if (tid == 0 && sm.nonfinite) report(status, DEV_NONFINITE);
}

}  // namespace quant

clef_status lut6_quantize_launch(const __half* w, int64_t n, int64_t k, uint8_t* packed, __half* lut,
                                 cudaStream_t stream) {
  const int64_t groups = n / 16;
  if (groups == 0) return CLEF_OK;
  const size_t smem = sizeof(quant::Smem);
  static std::atomic<uint64_t> attr{0};
  CLEF_CUDA_CHECK(smem_opt_in((const void*)quant::quantize_kernel, smem, &attr));
  const int64_t clusters = std::min<int64_t>(groups, (int64_t)num_sms() * 3 / quant::CL);
  TraceScope ts(stream, "lut6_quantize", 0.0, 2.0 * n * k * 2.0 + 0.75 * n * k + 128.0 * groups);
  quant::quantize_kernel<<<(unsigned)(clusters * quant::CL), quant::THREADS, smem, stream>>>(
      w, n, k, packed, lut, status_word_ptr());
  CLEF_LAUNCH_CHECK();
  return CLEF_OK;
}

}  // namespace clef

using namespace clef;

extern "C" clef_status clef_lut6_quantize(const uint16_t* w, int64_t n, int64_t k, uint8_t* packed,
                                          uint16_t* lut, clef_stream stream) {
  if (!w || !packed || !lut || n < 0 || k < 0) {
    set_error("clef_lut6_quantize: NULL pointer or negative size");
    return CLEF_E_INVALID;
  }
  if (n % 16 || k % 4 || k == 0 || k > (int64_t)1 << 18) {
    set_error("clef_lut6_quantize: need n %% 16 == 0 and k %% 4 == 0, 0 < k <= 262144 (n=%lld k=%lld)",
              (long long)n, (long long)k);
    return CLEF_E_SHAPE;
  }
  if ((reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(packed) |
       reinterpret_cast<uintptr_t>(lut)) & 15u) {
    set_error("clef_lut6_quantize: device pointers must be 16-byte aligned");
    return CLEF_E_ALIGN;
  }
  if (debug_should_fail()) return CLEF_E_CUDA;
  return lut6_quantize_launch(reinterpret_cast<const __half*>(w), n, k, packed,
                              reinterpret_cast<__half*>(lut), static_cast<cudaStream_t>(stream));
}
