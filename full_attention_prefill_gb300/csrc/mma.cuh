// Warp-level tensor-core helpers (mma.sync m16n8k16 fp16 -> fp32, ldmatrix) for the small
// per-chunk / per-tile products of the Gated DeltaNet scan and the attention kernel.
//
// Fragment layouts (per PTX ISA, m16n8k16 .row.col): with g = lane / 4 and t = lane % 4,
//   A (16x16): a0 = (row g,   k 2t..2t+1)   a1 = (row g+8, k 2t..)
//              a2 = (row g,   k 2t+8..)     a3 = (row g+8, k 2t+8..)
//   B (16x8):  b0 = (k 2t..2t+1, col g)     b1 = (k 2t+8.., col g)
//   C (16x8):  c0,c1 = (row g, cols 2t, 2t+1)   c2,c3 = (row g+8, cols 2t, 2t+1)
#pragma once
#include <cuda_fp16.h>
#include <stdint.h>

namespace clef {

__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// Addresses (byte offsets into a row-major fp16 tile with `ld` elements per row) that lane
// `lane` passes to ldmatrix for each operand form.
// A fragment of rows m0.., k-cols k0.. from a [m][k] tile (k contiguous):      ldsm_x4
__device__ __forceinline__ uint32_t a_addr(uint32_t base, int ld, int m0, int k0, int lane) {
  const int m = m0 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int k = k0 + (lane >> 4) * 8;
  return base + (uint32_t)(m * ld + k) * 2u;
}
// A fragment from a [k][m] tile (m contiguous, i.e. A stored transposed):       ldsm_x4_t
__device__ __forceinline__ uint32_t at_addr(uint32_t base, int ld, int m0, int k0, int lane) {
  const int k = k0 + (lane & 7) + (lane >> 4) * 8;
  const int m = m0 + ((lane >> 3) & 1) * 8;
  return base + (uint32_t)(k * ld + m) * 2u;
}
// B fragments of two n-tiles (n0.., n0+8..) from a [n][k] tile (k contiguous): ldsm_x4
//   -> r[0], r[1] = (b0, b1) of n-tile n0;  r[2], r[3] = of n-tile n0 + 8
__device__ __forceinline__ uint32_t bn_addr(uint32_t base, int ld, int n0, int k0, int lane) {
  const int n = n0 + (lane & 7) + (lane >> 4) * 8;
  const int k = k0 + ((lane >> 3) & 1) * 8;
  return base + (uint32_t)(n * ld + k) * 2u;
}
// B fragments of two n-tiles from a [k][n] tile (n contiguous):                 ldsm_x4_t
__device__ __forceinline__ uint32_t bk_addr(uint32_t base, int ld, int n0, int k0, int lane) {
  const int k = k0 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int n = n0 + (lane >> 4) * 8;
  return base + (uint32_t)(k * ld + n) * 2u;
}

__device__ __forceinline__ uint32_t h2u(float lo, float hi) {
  __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// cp.async 16-byte copy global -> shared (L2-cached), with zero fill when `valid` is false.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

}  // namespace clef
