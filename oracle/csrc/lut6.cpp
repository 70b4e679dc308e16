// LUT-6 weight format and the LUT-6 linear, oracle side (test infrastructure only).
//
// "Clef-Flash-ANE-LUT6" model card, Weight precision and LUT-6 text weights: each large linear
// stores a 6-bit index per weight and, for every block of 16 output channels, a table of 64 FP16
// values; four indices go into three bytes in the little-endian order Core ML uses; with the
// tables a layer of 4,096 inputs costs about 6.02 bits per weight.
//
// Reading of "little-endian" (no page prints the bytes): the indices form one bit stream over
// the weight matrix, row-major with the input index fastest, least significant bit first; four
// indices i0..i3 are the 24-bit word w = i0 | i1 << 6 | i2 << 12 | i3 << 18, stored as the bytes
// w & 255, (w >> 8) & 255, w >> 16.  With k % 4 == 0 no byte holds bits of two rows.
#include <stdarg.h>
#include <stdio.h>

#include <memory>

#include "internal.h"

namespace orc {

static thread_local char g_msg[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return code;
}

// The dot products of x rows i, i + 1 with W rows j, j + 1, each summed exactly as orc::dot
// sums (eight interleaved partial sums, lane k % 8, added pairwise): the four outputs share
// their loads, nothing else.  On x86 the compiler also builds AVX2 and AVX-512 copies and picks
// one at load time; with no fused multiply-adds formed (-ffp-contract=off) every copy rounds
// the same way.
#if defined(__x86_64__) && defined(__GNUC__) && !defined(__clang__)
__attribute__((target_clones("avx512f", "avx2", "default")))
#endif
static void dot_2x2(const double* x0, const double* x1, const double* w0, const double* w1,
                    int64_t n, double* y00, double* y01, double* y10, double* y11) {
  v8d a00 = {0, 0, 0, 0, 0, 0, 0, 0}, a01 = a00, a10 = a00, a11 = a00;
  int64_t k = 0;
  for (; k + 8 <= n; k += 8) {
    const v8d X0 = load8(x0 + k), X1 = load8(x1 + k), W0 = load8(w0 + k), W1 = load8(w1 + k);
    a00 += X0 * W0;
    a01 += X0 * W1;
    a10 += X1 * W0;
    a11 += X1 * W1;
  }
  for (int l = 0; k < n; ++k, ++l) {
    a00[l] += x0[k] * w0[k];
    a01[l] += x0[k] * w1[k];
    a10[l] += x1[k] * w0[k];
    a11[l] += x1[k] * w1[k];
  }
  *y00 = lane_total(a00);
  *y01 = lane_total(a01);
  *y10 = lane_total(a10);
  *y11 = lane_total(a11);
}

void dense_linear(const double* x, int64_t m, int64_t k, const double* W, int64_t n, double* y) {
  // Every y[i][j] is one dot product of x row i and W row j over all k, summed as orc::dot sums.
  // Outputs are taken in bands of 512 weight rows (kept in the shared cache while every x row
  // passes under them), within a band 32 rows x 32 columns at a time and 2 x 2 within that.
  // That changes which outputs are computed together, never how any one is computed.
  const int64_t RB = 32, CB = 32, BAND = 512;
  const int64_t rblocks = (m + RB - 1) / RB;
  for (int64_t b0 = 0; b0 < n; b0 += BAND) {
    const int64_t b1 = std::min(n, b0 + BAND);
    const int64_t cblocks = (b1 - b0 + CB - 1) / CB;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int64_t rb = 0; rb < rblocks; ++rb)
      for (int64_t cb = 0; cb < cblocks; ++cb) {
        const int64_t i1 = std::min(m, (rb + 1) * RB), j1 = std::min(b1, b0 + (cb + 1) * CB);
        for (int64_t i = rb * RB; i < i1; i += 2)
          for (int64_t j = b0 + cb * CB; j < j1; j += 2) {
            // a ragged last row or column pairs with itself; its duplicate result is dropped
            const int64_t i2 = std::min(i + 1, i1 - 1), j2 = std::min(j + 1, j1 - 1);
            double r00, r01, r10, r11;
            dot_2x2(x + i * k, x + i2 * k, W + j * k, W + j2 * k, k, &r00, &r01, &r10, &r11);
            y[i * n + j] = r00;
            if (j2 != j) y[i * n + j2] = r01;
            if (i2 != i) y[i2 * n + j] = r10;
            if (i2 != i && j2 != j) y[i2 * n + j2] = r11;
          }
      }
  }
}

}  // namespace orc

using namespace orc;

extern "C" {

const char* orc_last_error(void) { return g_msg; }

int32_t orc_num_threads(void) {
  int32_t n = 1;
#ifdef _OPENMP
#pragma omp parallel
#pragma omp single
  n = (int32_t)omp_get_num_threads();
#endif
  return n;
}

int orc_lut6_pack(const uint8_t* idx, int64_t n, int64_t k, uint8_t* packed) {
  if (n < 0 || k < 0 || k % 4) return fail(-1, "pack: k must be a multiple of 4");
  for (int64_t i = 0; i < n * k; ++i)
    if (idx[i] >= 64) return fail(-2, "pack: index %d >= 64 at %lld", idx[i], (long long)i);
  for (int64_t q = 0; q < n * k / 4; ++q) {
    const uint8_t* i4 = idx + 4 * q;
    const uint32_t w = (uint32_t)i4[0] | (uint32_t)i4[1] << 6 | (uint32_t)i4[2] << 12 |
                       (uint32_t)i4[3] << 18;
    packed[3 * q + 0] = (uint8_t)(w & 255u);
    packed[3 * q + 1] = (uint8_t)((w >> 8) & 255u);
    packed[3 * q + 2] = (uint8_t)(w >> 16);
  }
  return 0;
}

int orc_lut6_unpack(const uint8_t* packed, int64_t n, int64_t k, uint8_t* idx) {
  if (n < 0 || k < 0 || k % 4) return fail(-1, "unpack: k must be a multiple of 4");
  for (int64_t q = 0; q < n * k / 4; ++q) {
    // the 24-bit word of the quadruple, then index j = bits 6j .. 6j + 5
    const uint32_t w = (uint32_t)packed[3 * q] | (uint32_t)packed[3 * q + 1] << 8 |
                       (uint32_t)packed[3 * q + 2] << 16;
    for (int j = 0; j < 4; ++j) idx[4 * q + j] = (uint8_t)((w >> (6 * j)) & 63u);
  }
  return 0;
}

int orc_lut6_dequant_f16(const uint8_t* packed, const uint16_t* lut, int64_t n, int64_t k,
                         uint16_t* w) {
  if (n < 0 || n % 16 || k < 0 || k % 4) return fail(-1, "dequant: need n %% 16 == 0, k %% 4 == 0");
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    std::vector<uint8_t> idx((size_t)k);
    orc_lut6_unpack(packed + r * (k / 4) * 3, 1, k, idx.data());
    const uint16_t* table = lut + (r / 16) * 64;           // the table of row r's 16-row group
    for (int64_t c = 0; c < k; ++c) w[r * k + c] = table[idx[(size_t)c]];
  }
  return 0;
}

int orc_lut6_dequant(const uint8_t* packed, const uint16_t* lut, int64_t n, int64_t k, double* w) {
  if (n < 0 || n % 16 || k < 0 || k % 4) return fail(-1, "dequant: need n %% 16 == 0, k %% 4 == 0");
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < n; ++r) {
    std::vector<uint8_t> idx((size_t)k);
    orc_lut6_unpack(packed + r * (k / 4) * 3, 1, k, idx.data());
    double table[64];                                       // row r's group table, widened
    for (int j = 0; j < 64; ++j) table[j] = half_to_double(lut[(r / 16) * 64 + j]);
    for (int64_t c = 0; c < k; ++c) w[r * k + c] = table[idx[(size_t)c]];
  }
  return 0;
}

int orc_lut6_linear(const double* x, int64_t m, int64_t k, const uint8_t* packed,
                    const uint16_t* lut, int64_t n, double* y) {
  if (m < 0 || n < 0 || n % 16 || k < 0 || k % 4) return fail(-1, "linear: bad shape");
  std::unique_ptr<double[]> W(new double[(size_t)(n * k)]);  // every entry written below
  orc_lut6_dequant(packed, lut, n, k, W.get());
  dense_linear(x, m, k, W.get(), n, y);
  return 0;
}

int64_t orc_lut6_storage_bits(int64_t n, int64_t k) {
  const int64_t packed_bytes = n * (k * 3 / 4);
  const int64_t table_bytes = (n / 16) * 64 * 2;
  return 8 * (packed_bytes + table_bytes);
}

}  // extern "C"
