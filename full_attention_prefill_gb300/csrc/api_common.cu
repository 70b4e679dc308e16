// Library plumbing behind the C ABI: error messages, the device status word, TMA descriptor
// encoding, the host-side fault hook, and the LUT-6 entry points.
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "glue.cuh"
#include "lut6.cuh"

namespace clef {

static thread_local char g_err[512] = "";

const char* set_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return g_err;
}

// The device status word: one per device that loads the library (a module-scope variable).
__device__ unsigned g_status_word = 0;

unsigned* status_word_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  static unsigned* ptrs[64] = {nullptr};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return nullptr;
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned*>(p);
  }
  return ptrs[dev];
}

cudaError_t smem_opt_in(const void* func, size_t bytes, std::atomic<uint64_t>* done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = (dev >= 0 && dev < 64) ? (uint64_t)1 << dev : 0;
  if (bit && (done->load(std::memory_order_acquire) & bit)) return cudaSuccess;
  // setting the same value twice (two threads racing here) is harmless
  e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && bit) done->fetch_or(bit, std::memory_order_release);
  return e;
}

clef_status check_batch_len(int64_t B, int64_t L) {
  if (B < 1 || L < 1) {
    set_error("need B >= 1 and L >= 1 (B=%lld L=%lld)", (long long)B, (long long)L);
    return CLEF_E_INVALID;
  }
  if (L > CLEF_MAX_LEN) {
    set_error("L = %lld is above the %d-position limit (refused, never cut)", (long long)L,
              CLEF_MAX_LEN);
    return CLEF_E_TOO_LONG;
  }
  if (B > (((int64_t)1 << 22) / L)) {   // B * L > 2^22, without forming the product
    set_error("B = %lld requests of L = %lld positions is above the supported 4194304 tokens",
              (long long)B, (long long)L);
    return CLEF_E_SHAPE;
  }
  return CLEF_OK;
}

// The lowest non-finite hidden row reported since the last clef_sync_status (one per device).
__device__ unsigned long long g_bad_row_word = ~0ull;

unsigned long long* bad_row_word_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  static unsigned long long* ptrs[64] = {nullptr};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= 64) return nullptr;
  if (!ptrs[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bad_row_word) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned long long*>(p);
  }
  return ptrs[dev];
}

int num_sms() {
  int dev = 0, n = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  return n > 0 ? n : 1;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

cudaError_t tma_encode(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
                       const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                       CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) {
    set_error("cuTensorMapEncodeTiled is not available from the driver");
    return cudaErrorNotSupported;
  }
  cuuint64_t d[5];
  cuuint64_t st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides_bytes[i];
  }
  CUresult r = fn(map, dt, (cuuint32_t)rank, const_cast<void*>(base), d, st, bx, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    set_error("cuTensorMapEncodeTiled failed (%d): rank %d, dims %llu x %llu, box %u x %u", (int)r,
              rank, (unsigned long long)dims[0], (unsigned long long)dims[1], box[0], box[1]);
    return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

cudaError_t tma_encode_2d(CUtensorMap* map, CUtensorMapDataType dt, const void* base, uint64_t inner,
                          uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner,
                          uint32_t box_outer, CUtensorMapSwizzle swz) {
  const uint64_t dims[2] = {inner, outer};
  const uint64_t strides[1] = {row_stride_bytes};
  const uint32_t box[2] = {box_inner, box_outer};
  return tma_encode(map, dt, 2, base, dims, strides, box, swz);
}

// host-side fault hook (tests of error paths without any GPU fault)
static int g_fail_next = 0;
static std::mutex g_fail_mu;
bool debug_should_fail() {
  std::lock_guard<std::mutex> lock(g_fail_mu);
  if (g_fail_next > 0) {
    --g_fail_next;
    set_error("failure injected by clef_debug_fail_next");
    return true;
  }
  return false;
}

// ---- per-kernel-class tracing ----
struct TraceRec {
  cudaEvent_t a, b;
  const char* cls;
  double flops, bytes;
  bool used;
};
static std::mutex g_trace_mu;
static bool g_trace = false;
static std::vector<TraceRec> g_recs;
static size_t g_next = 0;

bool trace_on() { return g_trace; }

int trace_start(cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  if (!g_trace) return -1;
  if (g_next == g_recs.size()) {
    TraceRec r{};
    if (cudaEventCreate(&r.a) != cudaSuccess || cudaEventCreate(&r.b) != cudaSuccess) return -1;
    g_recs.push_back(r);
  }
  const int slot = (int)g_next++;
  g_recs[slot].used = false;
  cudaEventRecord(g_recs[slot].a, s);
  return slot;
}

void trace_stop(int slot, cudaStream_t s, const char* cls, double flops, double bytes) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  if (slot < 0 || (size_t)slot >= g_recs.size()) return;
  TraceRec& r = g_recs[slot];
  cudaEventRecord(r.b, s);
  r.cls = cls;
  r.flops = flops;
  r.bytes = bytes;
  r.used = true;
}

}  // namespace clef

using namespace clef;

static inline bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

extern "C" {

const char* clef_last_error(void) { return g_err; }

int32_t clef_version(void) { return (1 << 16) | 1; }

clef_status clef_trace_begin(void) {
  std::lock_guard<std::mutex> lock(g_trace_mu);
  g_trace = true;
  g_next = 0;
  return CLEF_OK;
}

clef_status clef_trace_end(clef_trace_entry* entries, int32_t max_entries, int32_t* n_entries) {
  if (!n_entries || (max_entries > 0 && !entries)) {
    set_error("clef_trace_end: NULL output");
    return CLEF_E_INVALID;
  }
  std::lock_guard<std::mutex> lock(g_trace_mu);
  g_trace = false;
  CLEF_CUDA_CHECK(cudaDeviceSynchronize());
  int32_t n = 0;
  for (size_t i = 0; i < g_next; ++i) {
    const TraceRec& r = g_recs[i];
    if (!r.used) continue;
    float ms = 0.f;
    CLEF_CUDA_CHECK(cudaEventElapsedTime(&ms, r.a, r.b));
    int32_t j = 0;
    while (j < n && strncmp(entries[j].name, r.cls, sizeof entries[j].name) != 0) ++j;
    if (j == n) {
      if (n == max_entries) continue;
      memset(&entries[n], 0, sizeof entries[n]);
      strncpy(entries[n].name, r.cls, sizeof entries[n].name - 1);
      ++n;
    }
    entries[j].launches += 1;
    entries[j].ms += ms;
    entries[j].flops += r.flops;
    entries[j].bytes += r.bytes;
  }
  g_next = 0;
  *n_entries = n;
  return CLEF_OK;
}

void clef_debug_fail_next(int32_t n_calls) {
  std::lock_guard<std::mutex> lock(g_fail_mu);
  g_fail_next = n_calls > 0 ? n_calls : 0;
}

clef_status clef_sync_status(clef_stream stream) {
  CLEF_CUDA_CHECK(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
  unsigned* p = status_word_ptr();
  if (!p) {
    set_error("cannot resolve the device status word");
    return CLEF_E_CUDA;
  }
  unsigned v = 0, zero = 0;
  CLEF_CUDA_CHECK(cudaMemcpy(&v, p, sizeof v, cudaMemcpyDeviceToHost));
  CLEF_CUDA_CHECK(cudaMemcpy(p, &zero, sizeof zero, cudaMemcpyHostToDevice));
  if (v == DEV_OK) return CLEF_OK;
  if (v == DEV_BAD_TOKEN) {
    set_error("a token id was outside [0, vocab)");
    return CLEF_E_BAD_TOKEN;
  }
  if (v == DEV_NONFINITE) {
    set_error("a weight given to the quantiser was not finite");
    return CLEF_E_NONFINITE;
  }
  if (v == DEV_NONFINITE_HIDDEN) {
    unsigned long long row = ~0ull, none = ~0ull;
    unsigned long long* rp = bad_row_word_ptr();
    if (rp) {
      CLEF_CUDA_CHECK(cudaMemcpy(&row, rp, sizeof row, cudaMemcpyDeviceToHost));
      CLEF_CUDA_CHECK(cudaMemcpy(rp, &none, sizeof none, cudaMemcpyHostToDevice));
    }
    set_error("hidden row %lld (row index b * L + t) is not finite, and maybe later rows: the "
              "request overflowed fp16 and is rejected", (long long)row);
    return CLEF_E_NONFINITE;
  }
  set_error("a device wait ran out (code 0x%x)", v);
  return CLEF_E_DEVICE_TIMEOUT;
}

clef_status clef_check_finite(const uint16_t* x, int64_t rows, int64_t cols, uint8_t* flags,
                              clef_stream stream) {
  if (rows < 0 || cols < 0 || (rows > 0 && !x)) {
    set_error("clef_check_finite: NULL pointer or negative size");
    return CLEF_E_INVALID;
  }
  if (cols % 8) {
    set_error("clef_check_finite: cols = %lld is not a multiple of 8", (long long)cols);
    return CLEF_E_SHAPE;
  }
  if (misaligned(x)) {
    set_error("clef_check_finite: x must be 16-byte aligned");
    return CLEF_E_ALIGN;
  }
  if (debug_should_fail()) return CLEF_E_CUDA;
  return check_finite_launch(reinterpret_cast<const __half*>(x), rows, cols, flags,
                             static_cast<cudaStream_t>(stream));
}

clef_status clef_lut6_pack(const uint8_t* idx, int64_t n, int64_t k, uint8_t* packed) {
  if (!idx || !packed || n < 0 || k < 0) {
    set_error("clef_lut6_pack: NULL pointer or negative size");
    return CLEF_E_INVALID;
  }
  if (k % 4) {
    set_error("clef_lut6_pack: k = %lld is not a multiple of 4", (long long)k);
    return CLEF_E_SHAPE;
  }
  const int64_t quads = n * (k / 4);
  for (int64_t q = 0; q < quads; ++q) {
    const uint8_t* i = idx + 4 * q;
    if ((i[0] | i[1] | i[2] | i[3]) & 0xC0) {
      set_error("clef_lut6_pack: index >= 64 at quadruple %lld", (long long)q);
      return CLEF_E_INVALID;
    }
    const uint32_t w = (uint32_t)i[0] | ((uint32_t)i[1] << 6) | ((uint32_t)i[2] << 12) |
                       ((uint32_t)i[3] << 18);
    packed[3 * q + 0] = (uint8_t)(w & 0xFFu);
    packed[3 * q + 1] = (uint8_t)((w >> 8) & 0xFFu);
    packed[3 * q + 2] = (uint8_t)((w >> 16) & 0xFFu);
  }
  return CLEF_OK;
}

clef_status clef_lut6_unpack(const uint8_t* packed, int64_t n, int64_t k, uint8_t* idx) {
  if (!idx || !packed || n < 0 || k < 0) {
    set_error("clef_lut6_unpack: NULL pointer or negative size");
    return CLEF_E_INVALID;
  }
  if (k % 4) {
    set_error("clef_lut6_unpack: k = %lld is not a multiple of 4", (long long)k);
    return CLEF_E_SHAPE;
  }
  const int64_t quads = n * (k / 4);
  for (int64_t q = 0; q < quads; ++q) {
    const uint32_t w = (uint32_t)packed[3 * q] | ((uint32_t)packed[3 * q + 1] << 8) |
                       ((uint32_t)packed[3 * q + 2] << 16);
    for (int j = 0; j < 4; ++j) idx[4 * q + j] = (uint8_t)((w >> (6 * j)) & 63u);
  }
  return CLEF_OK;
}

clef_status clef_lut6_dequant(const uint8_t* packed, const uint16_t* lut, int64_t n, int64_t k,
                              uint16_t* w, clef_stream stream) {
  if (!packed || !lut || !w || n < 0 || k < 0) {
    set_error("clef_lut6_dequant: NULL pointer or negative size");
    return CLEF_E_INVALID;
  }
  if (n % 16 || k % 4) {
    set_error("clef_lut6_dequant: need n %% 16 == 0 and k %% 4 == 0 (n=%lld k=%lld)", (long long)n,
              (long long)k);
    return CLEF_E_SHAPE;
  }
  if (misaligned(lut) || misaligned(w)) {
    set_error("clef_lut6_dequant: device pointers must be 16-byte aligned");
    return CLEF_E_ALIGN;
  }
  if (debug_should_fail()) return CLEF_E_CUDA;
  return lut6_dequant_launch(packed, reinterpret_cast<const __half*>(lut), n, k,
                             reinterpret_cast<__half*>(w), static_cast<cudaStream_t>(stream));
}

clef_status clef_lut6_tile(const uint8_t* packed, int64_t n, int64_t k, uint8_t* tiled,
                           clef_stream stream) {
  if (!packed || !tiled || n < 0 || k < 0) {
    set_error("clef_lut6_tile: NULL pointer or negative size");
    return CLEF_E_INVALID;
  }
  if (n % 16 || k % 64) {
    set_error("clef_lut6_tile: need n %% 16 == 0 and k %% 64 == 0 (n=%lld k=%lld)", (long long)n,
              (long long)k);
    return CLEF_E_SHAPE;
  }
  if (debug_should_fail()) return CLEF_E_CUDA;
  return lut6_tile_launch(packed, n, k, tiled, static_cast<cudaStream_t>(stream));
}

size_t clef_lut6_gemm_canonical_workspace_size(int64_t n, int64_t k) {
  if (n <= 0 || k <= 0 || n % 16 || k % 64) return 0;
  return (size_t)n * (size_t)(k / 4 * 3);
}

clef_status clef_lut6_gemm_canonical(const uint16_t* x, const uint8_t* packed, const uint16_t* lut,
                                     void* y, int32_t y_is_fp32, int64_t m, int64_t n, int64_t k,
                                     void* workspace, size_t workspace_bytes, clef_stream stream) {
  if (m < 0 || n <= 0 || k <= 0) {
    set_error("clef_lut6_gemm_canonical: bad size");
    return CLEF_E_INVALID;
  }
  if (m == 0) return CLEF_OK;
  if (!packed || !workspace) {
    set_error("clef_lut6_gemm_canonical: NULL pointer");
    return CLEF_E_INVALID;
  }
  if (n % 16 || k % 64) {
    set_error("clef_lut6_gemm_canonical: need n %% 16 == 0 and k %% 64 == 0 (n=%lld k=%lld)",
              (long long)n, (long long)k);
    return CLEF_E_SHAPE;
  }
  if (workspace_bytes < clef_lut6_gemm_canonical_workspace_size(n, k)) {
    set_error("clef_lut6_gemm_canonical: workspace of %zu bytes, need %zu", workspace_bytes,
              clef_lut6_gemm_canonical_workspace_size(n, k));
    return CLEF_E_WORKSPACE;
  }
  if (misaligned(workspace)) {
    set_error("clef_lut6_gemm_canonical: workspace must be 16-byte aligned");
    return CLEF_E_ALIGN;
  }
  const clef_status st = clef_lut6_tile(packed, n, k, static_cast<uint8_t*>(workspace), stream);
  if (st != CLEF_OK) return st;
  return clef_lut6_gemm(x, static_cast<const uint8_t*>(workspace), lut, y, y_is_fp32, m, n, k,
                        stream);
}

clef_status clef_lut6_gemm(const uint16_t* x, const uint8_t* packed, const uint16_t* lut, void* y,
                           int32_t y_is_fp32, int64_t m, int64_t n, int64_t k, clef_stream stream) {
  if (m < 0 || n <= 0 || k <= 0 || (y_is_fp32 != 0 && y_is_fp32 != 1)) {
    set_error("clef_lut6_gemm: bad size or bad y_is_fp32");
    return CLEF_E_INVALID;
  }
  if (m == 0) return CLEF_OK;  /* nothing to compute; x and y may be NULL */
  if (!x || !packed || !lut || !y) {
    set_error("clef_lut6_gemm: NULL pointer");
    return CLEF_E_INVALID;
  }
  if (n % 16 || k % 64) {
    set_error("clef_lut6_gemm: need n %% 16 == 0 and k %% 64 == 0 (n=%lld k=%lld)", (long long)n,
              (long long)k);
    return CLEF_E_SHAPE;
  }
  if (m > (int64_t)INT32_MAX / 2 || n > (1 << 24) || k > (1 << 20)) {
    set_error("clef_lut6_gemm: size out of the supported range");
    return CLEF_E_SHAPE;
  }
  if (misaligned(x) || misaligned(packed) || misaligned(lut) || misaligned(y)) {
    set_error("clef_lut6_gemm: device pointers must be 16-byte aligned");
    return CLEF_E_ALIGN;
  }
  if (debug_should_fail()) return CLEF_E_CUDA;
  return lut6_gemm_launch(reinterpret_cast<const __half*>(x), packed,
                          reinterpret_cast<const __half*>(lut), y, n, m, n, k,
                          y_is_fp32 ? EPI_F32 : EPI_F16, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
