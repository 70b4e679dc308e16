// Helpers shared by the oracle's translation units (oracle side only).
#pragma once

#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <cmath>
#include <limits>
#include <vector>

#include "oracle.h"

#ifdef _OPENMP
#include <omp.h>
#endif

namespace orc {

int fail(int code, const char* fmt, ...);   // records the message; returns code

// IEEE 754 binary16 -> binary64, from the format's definition (1 sign bit, 5 exponent bits with
// bias 15, 10 fraction bits); exact.
inline double half_to_double(uint16_t h) {
  const int e = (h >> 10) & 0x1F, f = h & 0x3FF;
  double mag;
  if (e == 0)
    mag = std::ldexp((double)f, -24);                       // zero and subnormals: f * 2^-24
  else if (e == 31)
    mag = f ? std::numeric_limits<double>::quiet_NaN() : std::numeric_limits<double>::infinity();
  else
    mag = std::ldexp((double)(0x400 | f), e - 25);          // (1 + f / 1024) * 2^(e - 15)
  return (h & 0x8000) ? -mag : mag;
}

// binary64 -> the nearest binary16, ties to even.
inline uint16_t double_to_half(double x) {
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  if (std::isnan(x)) return sign | 0x7E00;
  const double a = std::fabs(x);
  if (a >= 65520.0) return sign | 0x7C00;                   // past the midpoint above 65504
  if (a == 0.0) return sign;
  int E = 0;
  std::frexp(a, &E);                                        // a in [2^(E-1), 2^E)
  const int b = std::max(E - 1, -14);                       // subnormals: the lowest binade's step
  const double step = std::ldexp(1.0, b - 10);
  const double n = std::nearbyint(a / step);                // default mode: ties to even
  const double v = n * step;
  if (v < std::ldexp(1.0, -14)) return sign | (uint16_t)n;  // subnormal
  std::frexp(v, &E);
  const int eb = E - 1;
  const uint16_t frac = (uint16_t)(std::ldexp(v, 10 - eb) - 1024.0);
  return sign | (uint16_t)((eb + 15) << 10) | frac;
}

inline std::vector<double> widen(const uint16_t* h, int64_t n) {
  std::vector<double> out((size_t)n);
  for (int64_t i = 0; i < n; ++i) out[(size_t)i] = half_to_double(h[i]);
  return out;
}

// Eight doubles as one value (a GCC vector extension: portable, lowered to whatever vector
// width the target has); lane l holds the partial sum over k % 8 == l.
typedef double v8d __attribute__((vector_size(64)));

inline v8d load8(const double* p) {
  v8d v;
  __builtin_memcpy(&v, p, sizeof v);
  return v;
}

// The lanes of a partial-sum vector added pairwise: ((0 + 1) + (2 + 3)) + ((4 + 5) + (6 + 7)).
inline double lane_total(v8d a) {
  return ((a[0] + a[1]) + (a[2] + a[3])) + ((a[4] + a[5]) + (a[6] + a[7]));
}

// sum_k a[k] b[k] in fp64, accumulated in eight interleaved partial sums (lane k % 8) that are
// added pairwise at the end: a fixed order, the same on every machine and thread count.
inline double dot(const double* a, const double* b, int64_t n) {
  v8d acc = {0, 0, 0, 0, 0, 0, 0, 0};
  int64_t k = 0;
  for (; k + 8 <= n; k += 8) acc += load8(a + k) * load8(b + k);
  for (int l = 0; k < n; ++k, ++l) acc[l] += a[k] * b[k];
  return lane_total(acc);
}

inline double silu(double x) { return x / (1.0 + std::exp(-x)); }
inline double sigmoid(double x) { return 1.0 / (1.0 + std::exp(-x)); }
// log(1 + e^x), written so that neither branch overflows
inline double softplus(double x) { return std::max(x, 0.0) + std::log1p(std::exp(-std::fabs(x))); }

// y [m, n] = x [m, k] . W^T for a dense fp64 W [n, k]
void dense_linear(const double* x, int64_t m, int64_t k, const double* W, int64_t n, double* y);

constexpr double kRmsEps = 1e-6;
constexpr double kL2Eps = 1e-6;
constexpr double kRopeTheta = 1.0e7;
constexpr int64_t kRopeDims = 64;

}  // namespace orc
