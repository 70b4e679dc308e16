// The LUT-6 quantiser, oracle side (fp64 with exact integer sums; test infrastructure only).
//
// "Clef-Flash-ANE-LUT6" model card, LUT-6 text weights: each group of 16 output channels gets a
// 64-value table found by 40 rounds of one-dimensional k-means; half of the starting values are
// quantiles of the group's weights, the other half are spread evenly between its minimum and
// maximum.
//
// Readings where the card is silent (each a plain choice the rest of the card allows):
//   * quantiles: the 32 probabilities (i + 1/2) / 32, each between the two neighbouring order
//     statistics by linear interpolation, x[lo] + f (x[lo+1] - x[lo]) with h = p (n - 1),
//     lo = floor(h), f = h - lo (exact in fp64 for fp16 weights);
//   * evenly spread: min + i * step, step = (max - min) / 31, i = 0..30, rounded after the
//     division, the product and the sum; the 32nd value is max itself;
//   * the 64 starting centroids (quantiles first, then the spread values) are sorted ascending by
//     a stable sort, and again after every round: equal centroids share their members with the
//     first of them, which moves alone, so the order is not kept by itself (sorting only
//     relabels; the set of centroids, and every later round, stays the same);
//   * a round gives each weight to its nearest centroid: with ascending centroids, the cell
//     between the midpoints fl(c_j + c_j+1) / 2 of its neighbours; a weight exactly on a midpoint
//     goes to the lower index, and a weight whose nearest value several equal centroids hold goes
//     to the first of them.  A centroid with members moves to their mean; one without stays;
//   * the mean is rounded once: fp16 weights are integer multiples of 2^-24, so their sum S is an
//     exact integer (in units of 2^-24) and the centroid is fl(fl(S) / count) * 2^-24;
//   * after the rounds the table is the centroids rounded to fp16 (nearest, ties to even), and
//     each weight's index is its nearest table entry, ties (a midpoint, or equal entries) to the
//     lower index;
//   * weights must be finite.
#include "internal.h"

using namespace orc;

namespace {

constexpr int64_t kHalf = 32;                 // quantile seeds, and evenly spread seeds
constexpr double kFix = 16777216.0;           // 2^24: fp16 values are integer multiples of 2^-24

void stable_ascending(double* c, int64_t nc) {
  std::stable_sort(c, c + nc, [](double a, double b) { return a < b; });
}

}  // namespace

extern "C" {

void orc_quant_quantiles(const double* values, int64_t n, double* out) {
  std::vector<double> x(values, values + n);
  std::sort(x.begin(), x.end());
  for (int64_t i = 0; i < kHalf; ++i) {
    const double h = (i + 0.5) / (double)kHalf * (double)(n - 1);
    const int64_t lo = (int64_t)std::floor(h);
    const int64_t hi = std::min(lo + 1, n - 1);
    const double f = h - (double)lo;
    out[i] = x[(size_t)lo] + f * (x[(size_t)hi] - x[(size_t)lo]);
  }
}

void orc_quant_spread(const double* values, int64_t n, double* out) {
  // the smallest and the largest value; a zero maximum keeps +0 over -0 when both occur
  double lo = values[0], hi = values[0];
  for (int64_t i = 1; i < n; ++i) {
    if (values[i] < lo) lo = values[i];
    if (values[i] > hi || (values[i] == hi && !std::signbit(values[i]))) hi = values[i];
  }
  const double step = (hi - lo) / (double)(kHalf - 1);
  for (int64_t i = 0; i < kHalf - 1; ++i) out[i] = (double)i * step + lo;
  out[kHalf - 1] = hi;
}

void orc_quant_initial_table(const double* values, int64_t n, double* out) {
  orc_quant_quantiles(values, n, out);
  orc_quant_spread(values, n, out + kHalf);
  stable_ascending(out, 2 * kHalf);
}

void orc_quant_assign(const double* values, int64_t n, const double* c, int64_t nc, int64_t* cell) {
  std::vector<double> mid((size_t)(nc - 1));
  for (int64_t j = 0; j + 1 < nc; ++j) mid[(size_t)j] = (c[j] + c[j + 1]) / 2.0;
  // first[j]: the lowest index holding the value c[j] (the number of centroids below it)
  std::vector<int64_t> first((size_t)nc);
  for (int64_t j = 0; j < nc; ++j)
    first[(size_t)j] = std::lower_bound(c, c + nc, c[j]) - c;
  for (int64_t i = 0; i < n; ++i) {
    // the number of midpoints strictly below the value: its cell among the ascending centroids
    const int64_t m = std::lower_bound(mid.begin(), mid.end(), values[i]) - mid.begin();
    cell[i] = first[(size_t)m];
  }
}

void orc_quant_kmeans_round(const double* values, int64_t n, double* c, int64_t nc) {
  std::vector<int64_t> cell((size_t)n);
  orc_quant_assign(values, n, c, nc, cell.data());
  std::vector<int64_t> total((size_t)nc, 0), count((size_t)nc, 0);
  for (int64_t i = 0; i < n; ++i) {
    total[(size_t)cell[i]] += (int64_t)std::nearbyint(values[i] * kFix);   // exact for fp16 data
    count[(size_t)cell[i]] += 1;
  }
  for (int64_t j = 0; j < nc; ++j)
    if (count[(size_t)j]) c[j] = ((double)total[(size_t)j] / (double)count[(size_t)j]) / kFix;
  stable_ascending(c, nc);
}

void orc_quant_group(const double* values, int64_t n, int32_t rounds, uint16_t* table,
                     uint8_t* idx) {
  double c[2 * kHalf];
  orc_quant_initial_table(values, n, c);
  for (int32_t r = 0; r < rounds; ++r) orc_quant_kmeans_round(values, n, c, 2 * kHalf);
  double t[2 * kHalf];
  for (int64_t j = 0; j < 2 * kHalf; ++j) {
    table[j] = double_to_half(c[j]);
    t[j] = half_to_double(table[j]);
  }
  std::vector<int64_t> cell((size_t)n);
  orc_quant_assign(values, n, t, 2 * kHalf, cell.data());
  for (int64_t i = 0; i < n; ++i) idx[i] = (uint8_t)cell[(size_t)i];
}

int orc_lut6_quantize(const uint16_t* w, int64_t n, int64_t k, int32_t rounds, uint8_t* packed,
                      uint16_t* lut) {
  if (n < 0 || n % 16 || k <= 0 || k % 4)
    return fail(-1, "quantize: n must be a multiple of 16 and k a positive multiple of 4");
  for (int64_t i = 0; i < n * k; ++i)
    if ((w[i] & 0x7C00) == 0x7C00) return fail(-2, "quantize: weights must be finite");
  std::vector<uint8_t> idx((size_t)(n * k));
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t g = 0; g < n / 16; ++g) {
    // the group's 16 rows, row-major
    const std::vector<double> v = widen(w + g * 16 * k, 16 * k);
    orc_quant_group(v.data(), 16 * k, rounds, lut + g * 64, idx.data() + g * 16 * k);
  }
  return orc_lut6_pack(idx.data(), n, k, packed);
}

}  // extern "C"
