// Building blocks of the clef-flash decoder layers, oracle side (fp64, test infrastructure only).
//
// Each function states the passage it follows.  Where the pages are silent the plainest reading
// is taken and named.
#include "internal.h"

using namespace orc;

extern "C" {

void orc_silu(const double* x, int64_t n, double* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = silu(x[i]);
}

void orc_sigmoid(const double* x, int64_t n, double* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = sigmoid(x[i]);
}

void orc_softplus(const double* x, int64_t n, double* y) {
  for (int64_t i = 0; i < n; ++i) y[i] = softplus(x[i]);
}

// RMSNorm.  "Clef-Flash-ANE-LUT6", Weight precision: the normalisation weights are FP16 text
// weights; "clef-flash-LiteRT", Host contract: the output is the final RMSNorm's, per position.
// Reading (no page gives them): eps = 1e-6 and the plain form x * r * w, r = 1 / sqrt(mean x^2 + eps).
void orc_rmsnorm(const double* x, int64_t rows, int64_t d, const double* w, double eps, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const double* xr = x + r * d;
    double ss = 0.0;
    for (int64_t i = 0; i < d; ++i) ss += xr[i] * xr[i];
    const double inv = 1.0 / std::sqrt(ss / (double)d + eps);
    for (int64_t i = 0; i < d; ++i) y[r * d + i] = xr[i] * inv * (w ? w[i] : 1.0);
  }
}

// The per-head L2 normalisation of the Gated DeltaNet's q and k (eps 1e-6, a reading).
void orc_l2norm(const double* x, int64_t rows, int64_t d, double eps, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const double* xr = x + r * d;
    double ss = 0.0;
    for (int64_t i = 0; i < d; ++i) ss += xr[i] * xr[i];
    const double den = std::sqrt(ss + eps);
    for (int64_t i = 0; i < d; ++i) y[r * d + i] = xr[i] / den;
  }
}

// Short causal convolution + SiLU.  "Clef-Flash-ANE-LUT6", Weight precision names the short
// convolution; "clef-flash - Core AI", Core AI shape carries a conv state [24, 1, 8192, 3] per
// GDN layer: 8,192 channels and 3 + 1 = 4 taps.
//   c[t][ch] = SiLU( sum_{j = 0 .. taps-1} w[ch][j] * x[t - (taps - 1) + j][ch] ),
// with zero history before position 0 (a prefill starts from a zeroed state).
void orc_conv_silu(const double* x, int64_t L, int64_t C, const double* w, int64_t taps, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < L; ++t)
    for (int64_t ch = 0; ch < C; ++ch) {
      double acc = 0.0;
      for (int64_t j = 0; j < taps; ++j) {
        const int64_t src = t - (taps - 1) + j;
        if (src >= 0) acc += w[ch * taps + j] * x[src * C + ch];
      }
      y[t * C + ch] = silu(acc);
    }
}

// Decay and write strength per value head.  "Clef-Flash-ANE-LUT6", Weight precision keeps the
// small gate projections and the decay parameters in FP16.  Reading (standard Gated DeltaNet
// gating): alpha = exp(-exp(A_log) * softplus(a + dt_bias)), beta = sigmoid(b).
void orc_gdn_gates(const double* a, const double* b, int64_t L, int64_t H, const double* A_log,
                   const double* dt_bias, double* alpha, double* beta) {
  for (int64_t t = 0; t < L; ++t)
    for (int64_t h = 0; h < H; ++h) {
      alpha[t * H + h] = std::exp(-std::exp(A_log[h]) * softplus(a[t * H + h] + dt_bias[h]));
      beta[t * H + h] = sigmoid(b[t * H + h]);
    }
}

// The gated delta rule as a per-token recurrence (no chunking).
// "Clef-Flash-ANE-LUT6", Model architecture: Gated DeltaNet layers with 16 key and 32 value
// heads of size 128; "clef-flash - Core AI", Core AI shape: a recurrent state [.., 32, 128, 128]
// per layer carried across positions.  For value head h (key head h / (Hv / Hk)):
//   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T
//   o_t = S_t q_t / sqrt(dk)
// S is [dv][dk]; the output is read from the updated state (reading: the updated state maps k
// to v, so it is the state after position t) and scaled by 1 / sqrt(dk) (reading).
int orc_gated_delta_rule(const double* q, const double* k, const double* v, const double* alpha,
                         const double* beta, const double* s0, int64_t L, int64_t Hk, int64_t Hv,
                         int64_t dk, int64_t dv, double* o, double* s_out) {
  if (Hk < 1 || Hv % Hk) return fail(-1, "delta rule: Hv must be a multiple of Hk");
  const int64_t rep = Hv / Hk;
  const double scale = 1.0 / std::sqrt((double)dk);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t h = 0; h < Hv; ++h) {
    const int64_t g = h / rep;
    std::vector<double> S((size_t)(dv * dk), 0.0), Sk((size_t)dv);
    if (s0)
      for (int64_t i = 0; i < dv * dk; ++i) S[(size_t)i] = s0[h * dv * dk + i];
    for (int64_t t = 0; t < L; ++t) {
      const double* kt = k + (t * Hk + g) * dk;
      const double* qt = q + (t * Hk + g) * dk;
      const double* vt = v + (t * Hv + h) * dv;
      const double a = alpha[t * Hv + h], b = beta[t * Hv + h];
      for (int64_t i = 0; i < dv; ++i) {                      // S_{t-1} k_t
        double s = 0.0;
        for (int64_t j = 0; j < dk; ++j) s += S[(size_t)(i * dk + j)] * kt[j];
        Sk[(size_t)i] = s;
      }
      for (int64_t i = 0; i < dv; ++i) {                      // the update, row by row
        const double u = b * (vt[i] - a * Sk[(size_t)i]);
        for (int64_t j = 0; j < dk; ++j)
          S[(size_t)(i * dk + j)] = a * S[(size_t)(i * dk + j)] + u * kt[j];
      }
      for (int64_t i = 0; i < dv; ++i) {                      // o_t = S_t q_t / sqrt(dk)
        double s = 0.0;
        for (int64_t j = 0; j < dk; ++j) s += S[(size_t)(i * dk + j)] * qt[j];
        o[(t * Hv + h) * dv + i] = s * scale;
      }
    }
    if (s_out)
      for (int64_t i = 0; i < dv * dk; ++i) s_out[h * dv * dk + i] = S[(size_t)i];
  }
  return 0;
}

// Output gate of the GDN mixer: RMSNorm over each head's dv values, times w (shared by the
// heads), times SiLU(z).
void orc_zgated_norm(const double* o, const double* z, int64_t L, int64_t H, int64_t d,
                     const double* w, double eps, double* y) {
  orc_rmsnorm(o, L * H, d, w, eps, y);
  for (int64_t i = 0; i < L * H * d; ++i) y[i] = y[i] * silu(z[i]);
}

// Rotary embedding on the first rot_dims dims of each head, rotate-half pairing.
// "clef-flash-coreml" README: the decoder parts take cos / sin [L, 64]; "clef-flash-LiteRT",
// Host contract: theta = 1e7, and text tokens sit at (i, i, i), so the three M-RoPE planes
// collapse to one 1-D rotary.  Pair (j, j + rot_dims/2), j < rot_dims/2, turns by the angle
// pos * theta^(-2j / rot_dims); the other dims pass through.
void orc_rope(const double* x, int64_t L, int64_t H, int64_t D, const double* pos,
              int64_t rot_dims, double theta, double* y) {
  const int64_t half = rot_dims / 2;
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < L; ++t)
    for (int64_t h = 0; h < H; ++h) {
      const double* xr = x + (t * H + h) * D;
      double* yr = y + (t * H + h) * D;
      for (int64_t i = rot_dims; i < D; ++i) yr[i] = xr[i];
      for (int64_t j = 0; j < half; ++j) {
        const double ang = pos[t] * std::pow(theta, -(double)(2 * j) / (double)rot_dims);
        const double c = std::cos(ang), s = std::sin(ang);
        yr[j] = xr[j] * c - xr[j + half] * s;
        yr[j + half] = xr[j + half] * c + xr[j] * s;
      }
    }
}

// "clef-flash-LiteRT", Host contract: three planes with sections 11 / 11 / 10, interleaved.
// Reading: frequency pair j takes plane j mod 3, which gives exactly 11, 11 and 10 pairs.
void orc_mrope_planes(int64_t rot_dims, int64_t* planes) {
  for (int64_t j = 0; j < rot_dims / 2; ++j) planes[j] = j % 3;
}

// Positions (t, h, w) of a request holding at most one picture block of grid_h x grid_w tokens
// at index image_start.  "clef-flash-LiteRT", Host contract: text tokens at (i, i, i), picture
// tokens at their row and column, padding goes on from the last position; "clef-flash - Core
// AI", Core AI shape: image token k at row k / W, column k % W, and from the <|vision_end|>
// index (start + N) on the positions move back by N - max(H, W).  Reading: image token k has
// (s, s + k / W, s + k % W), so the token after the block continues at s + max(H, W).
int orc_mrope_positions(int64_t L, int64_t s, int64_t grid_h, int64_t grid_w, int64_t* pos3) {
  if (L < 0 || s < 0 || grid_h < 0 || grid_w < 0) return fail(-1, "mrope positions: negative size");
  const int64_t n = grid_h * grid_w;
  for (int64_t i = 0; i < L; ++i) {
    int64_t* p = pos3 + 3 * i;
    if (n == 0 || i < s) {
      p[0] = p[1] = p[2] = i;
    } else if (i < s + n) {
      const int64_t kk = i - s;
      p[0] = s;
      p[1] = s + kk / grid_w;
      p[2] = s + kk % grid_w;
    } else {
      const int64_t shifted = i - (n - std::max(grid_h, grid_w));
      p[0] = p[1] = p[2] = shifted;
    }
  }
  return 0;
}

// M-RoPE ("clef-flash-LiteRT", Host contract: cos / sin [L, 64] of the three-plane positions,
// theta 1e7): as orc_rope, pair j turning by pos3[t][plane(j)] * theta^(-2j / rot_dims).
void orc_mrope(const double* x, int64_t L, int64_t H, int64_t D, const int64_t* pos3,
               int64_t rot_dims, double theta, double* y) {
  const int64_t half = rot_dims / 2;
  std::vector<int64_t> planes((size_t)half);
  orc_mrope_planes(rot_dims, planes.data());
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < L; ++t)
    for (int64_t h = 0; h < H; ++h) {
      const double* xr = x + (t * H + h) * D;
      double* yr = y + (t * H + h) * D;
      for (int64_t i = rot_dims; i < D; ++i) yr[i] = xr[i];
      for (int64_t j = 0; j < half; ++j) {
        const double p = (double)pos3[3 * t + planes[(size_t)j]];
        const double ang = p * std::pow(theta, -(double)(2 * j) / (double)rot_dims);
        const double c = std::cos(ang), s = std::sin(ang);
        yr[j] = xr[j] * c - xr[j + half] * s;
        yr[j + half] = xr[j + half] * c + xr[j] * s;
      }
    }
}

// Causal softmax attention with grouped keys and values, one explicit softmax per query row.
// "clef-flash-LiteRT", Provenance: attention as batched products with an additive mask, the
// grouped keys and values repeated to the query heads.  Query head h reads kv head
// h / (Hq / Hkv); the logits are q.k / sqrt(D); row t attends to positions 0..t:
//   l_j = q_t . k_j / sqrt(D),  m = max_j l_j,  p_j = exp(l_j - m),  o_t = sum_j (p_j / sum p) v_j.
// Rows are worked on 16 at a time (one head) only so that each key and value row is loaded once
// for all of them; every row's arithmetic is exactly the per-row softmax above, in key order.
int orc_causal_attention(const double* q, const double* k, const double* v, int64_t L, int64_t Hq,
                         int64_t Hkv, int64_t D, int64_t row0, int64_t row1, double* o) {
  if (Hkv < 1 || Hq % Hkv) return fail(-1, "attention: Hq must be a multiple of Hkv");
  if (row0 < 0 || row1 > L || row0 > row1) return fail(-1, "attention: bad row range");
  const int64_t rep = Hq / Hkv, RB = 16;
  const double scale = 1.0 / std::sqrt((double)D);
  const int64_t nblk = (row1 - row0 + RB - 1) / RB;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int64_t h = 0; h < Hq; ++h)
    for (int64_t bi = nblk - 1; bi >= 0; --bi) {              // long rows first
      const int64_t g = h / rep;
      const int64_t t0 = row0 + bi * RB, t1 = std::min(row1, t0 + RB);
      const int64_t nk = t1;                                  // keys 0 .. t1 - 1 cover the block
      std::vector<double> logit((size_t)((t1 - t0) * nk));
      for (int64_t j = 0; j < nk; ++j) {
        const double* kj = k + (j * Hkv + g) * D;
        for (int64_t t = std::max(t0, j); t < t1; ++t)
          logit[(size_t)((t - t0) * nk + j)] = dot(q + (t * Hq + h) * D, kj, D) * scale;
      }
      std::vector<double> wsum((size_t)(t1 - t0));
      for (int64_t t = t0; t < t1; ++t) {
        double* lr = logit.data() + (t - t0) * nk;
        double m = -std::numeric_limits<double>::infinity();
        for (int64_t j = 0; j <= t; ++j) m = std::max(m, lr[j]);
        double sum = 0.0;
        for (int64_t j = 0; j <= t; ++j) {
          lr[j] = std::exp(lr[j] - m);
          sum += lr[j];
        }
        wsum[(size_t)(t - t0)] = sum;
        double* orow = o + ((t - row0) * Hq + h) * D;
        for (int64_t d = 0; d < D; ++d) orow[d] = 0.0;
      }
      for (int64_t j = 0; j < nk; ++j) {
        const double* vj = v + (j * Hkv + g) * D;
        for (int64_t t = std::max(t0, j); t < t1; ++t) {
          const double pj = logit[(size_t)((t - t0) * nk + j)] / wsum[(size_t)(t - t0)];
          double* orow = o + ((t - row0) * Hq + h) * D;
          for (int64_t d = 0; d < D; ++d) orow[d] += pj * vj[d];
        }
      }
    }
  return 0;
}

}  // extern "C"
