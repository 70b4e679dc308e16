// A variant of clef_gdn_prefill for callers that cannot allocate device memory.
//
// Some hosts run this library where cudaMalloc is not available to them: a plugin or an
// embedded runtime that owns the device allocator, or code that must not allocate once it is
// running.  They can still hand over their inputs and outputs, but not the scan's scratch.  For
// them the scratch lives in one array with static storage in this file, reserved on every GPU
// that loads the library for as long as the process runs.
//
// The pages describe nothing like this; it is an interface convenience only.  The computation is
// exactly that of clef_gdn_prefill (same kernels, same order), so results are bit-identical.
#include <mutex>

#include "common.cuh"
#include "gdn.cuh"

namespace clef {

// Scratch of the no-allocation scan.  In host code this name is only a stand-in for the device
// variable: its device address is taken with cudaGetSymbolAddress, per device, below.
static constexpr size_t kStaticScratchBytes = CLEF_GDN_NOALLOC_SCRATCH_BYTES;  // 64 MiB
static __device__ __align__(256) uint8_t g_gdn_scratch[kStaticScratchBytes];

// Device address of the scratch array on the current device, resolved once per device.
static void* static_scratch_ptr(clef_status* st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    set_error("clef_gdn_prefill_noalloc: no usable current device");
    *st = CLEF_E_CUDA;
    return nullptr;
  }
  static void* ptrs[64] = {nullptr};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_gdn_scratch);
    if (e != cudaSuccess || p == nullptr) {
      set_error("clef_gdn_prefill_noalloc: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
      *st = CLEF_E_CUDA;
      return nullptr;
    }
    ptrs[dev] = p;
  }
  *st = CLEF_OK;
  return ptrs[dev];
}

}  // namespace clef

using namespace clef;

extern "C" {

clef_status clef_gdn_prefill_noalloc(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                     const float* alpha, const float* beta, const float* s0,
                                     uint16_t* o, float* s_out, int64_t B, int64_t L,
                                     clef_stream stream) {
  // the same size limits as clef_gdn_prefill (B * L <= 2^22 keeps the scratch size query's
  // products in range) before the scratch size is computed
  const clef_status size_st = check_batch_len(B, L);
  if (size_st != CLEF_OK) return size_st;
  const size_t need = gdn_scan_workspace_bytes(B, L, false);
  if (need > kStaticScratchBytes) {
    set_error("clef_gdn_prefill_noalloc: B=%lld, L=%lld needs %zu bytes of scratch, above the "
              "built-in %zu (use clef_gdn_prefill with a workspace instead)",
              (long long)B, (long long)L, need, kStaticScratchBytes);
    return CLEF_E_SHAPE;
  }
  const void* need_ptrs[] = {q, k, v, alpha, beta, o};
  for (const void* p : need_ptrs)
    if (p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u)) {
      set_error("clef_gdn_prefill_noalloc: a pointer is NULL or not 16-byte aligned");
      return p ? CLEF_E_ALIGN : CLEF_E_INVALID;
    }
  if ((s0 && (reinterpret_cast<uintptr_t>(s0) & 15u)) ||
      (s_out && (reinterpret_cast<uintptr_t>(s_out) & 15u))) {
    set_error("clef_gdn_prefill_noalloc: s0 / s_out not 16-byte aligned");
    return CLEF_E_ALIGN;
  }
  clef_status st;
  void* scratch = static_scratch_ptr(&st);
  if (!scratch) return st;
  // Every scratch byte the scan reads is written earlier in the same call (the chunk phase
  // writes g, W and U' of every valid row, the state pass writes U and each chunk's entering
  // state; rows past the end are zero-filled on load, not read), so nothing has to be cleared.
  return gdn_scan_launch(reinterpret_cast<const __half*>(q), reinterpret_cast<const __half*>(k),
                         reinterpret_cast<const __half*>(v), nullptr, alpha, beta, s0, s_out,
                         nullptr, 0, nullptr, reinterpret_cast<__half*>(o), 32 * 128, B, L,
                         scratch, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
