// The joint schema head on the hidden states of one request, oracle side (fp64; test
// infrastructure only).
//
// What the pages fix ("clef-flash - Core AI" README, Readout contract and Core AI shape, Head):
//   * the head's inputs: the request's final-norm hidden rows; each question's and each option's
//     span mean (q_avg, o_avg: 1 / len on the span), the last real token as a global vector
//     (g_avg), each option's mean lm_head row (lexical), which question each option belongs to
//     (member), the question types, and validity flags for keys, questions and options;
//   * one logit per option out, and each question's probabilities a softmax over its options
//     (computed in float32 there; in fp64 here);
//   * its size ("Clef-Flash-ANE-LUT6", Model architecture: 4 layers of width 1,024 with 16 heads
//     and 2 routing layers; "clef-flash-LiteRT", Host contract step 7: 2 routing layers and 4
//     decoder layers over the request's tokens).
// What is a reading (the pages do not give the layers; synthetic weights only):
//   * slots: one row per question, per option and one global row, each its span mean (global:
//     the last token) projected 4096 -> 1024 (w_in), options plus their lexical row projected by
//     w_lex, questions plus a type embedding, options and the global row plus their own;
//   * the request's tokens projected 4096 -> 1024 (w_mem) are the memory the decoder layers read;
//   * decoder layer: s += CrossAttention(rmsnorm(s), memory) (16 heads of 64, keys with
//     key_valid only, scale 1/8), then s += SwiGLU MLP (1024 -> 4096 -> 1024) of rmsnorm(s);
//   * routing layer: the same with the slots attending to the valid slots (questions, options,
//     the global row) in place of the memory;
//   * after a final rmsnorm, option o's logit is (f_o W_opt^T) . (c_o W_qst^T) / sqrt(1024), c_o
//     the row of the question it belongs to (sum_q member[q][o] f_q); invalid options get 0;
//   * RMSNorm eps 1e-6; a row with no valid key gets a zero attention output.
#include "internal.h"

using namespace orc;

namespace {

constexpr int64_t HID = 4096, D = 1024, NH = 16, DH = 64, FF = 4096;

// y [rows, n] = x [rows, k] . W^T for fp16 W [n, k]
std::vector<double> proj(const double* x, int64_t rows, int64_t k, const uint16_t* W, int64_t n) {
  const std::vector<double> w = widen(W, n * k);
  std::vector<double> y((size_t)(rows * n));
  dense_linear(x, rows, k, w.data(), n, y.data());
  return y;
}

std::vector<double> norm_rows(const std::vector<double>& x, int64_t rows, const uint16_t* w) {
  const std::vector<double> ww = widen(w, D);
  std::vector<double> y(x.size());
  orc_rmsnorm(x.data(), rows, D, ww.data(), kRmsEps, y.data());
  return y;
}

// Multi-head attention of S query rows (q [S, D]) over keys / values [Tk, D] with a validity
// flag per key: per head, one explicit softmax per query row over the valid keys.
std::vector<double> attend(const std::vector<double>& q, int64_t S, const std::vector<double>& k,
                           const std::vector<double>& v, int64_t Tk, const uint8_t* valid) {
  std::vector<double> o((size_t)(S * D), 0.0);
  const double scale = 1.0 / std::sqrt((double)DH);
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int64_t h = 0; h < NH; ++h)
    for (int64_t s = 0; s < S; ++s) {
      std::vector<double> l((size_t)Tk);
      double m = -std::numeric_limits<double>::infinity();
      for (int64_t t = 0; t < Tk; ++t)
        if (valid[t]) {
          l[(size_t)t] = dot(&q[(size_t)(s * D + h * DH)], &k[(size_t)(t * D + h * DH)], DH) * scale;
          m = std::max(m, l[(size_t)t]);
        }
      if (m == -std::numeric_limits<double>::infinity()) continue;  // no valid key: zero
      double sum = 0.0;
      for (int64_t t = 0; t < Tk; ++t)
        if (valid[t]) {
          l[(size_t)t] = std::exp(l[(size_t)t] - m);
          sum += l[(size_t)t];
        }
      double* orow = &o[(size_t)(s * D + h * DH)];
      for (int64_t t = 0; t < Tk; ++t)
        if (valid[t]) {
          const double p = l[(size_t)t] / sum;
          for (int64_t d = 0; d < DH; ++d) orow[d] += p * v[(size_t)(t * D + h * DH + d)];
        }
    }
  return o;
}

// One layer on the slots s [S, D]: attention (to `mem` [Tk, D] with mem_valid, or to the slots
// themselves when mem is NULL) and the SwiGLU MLP, each a pre-norm residual step.
void layer(std::vector<double>& s, int64_t S, const orc_head_layer& L, const std::vector<double>* mem,
           int64_t Tk, const uint8_t* mem_valid, const uint8_t* slot_valid) {
  const std::vector<double> a = norm_rows(s, S, L.norm1);
  const std::vector<double> q = proj(a.data(), S, D, L.wq, D);
  const std::vector<double>& src = mem ? *mem : a;
  const int64_t n = mem ? Tk : S;
  const std::vector<double> k = proj(src.data(), n, D, L.wk, D);
  const std::vector<double> v = proj(src.data(), n, D, L.wv, D);
  const std::vector<double> o = attend(q, S, k, v, n, mem ? mem_valid : slot_valid);
  const std::vector<double> y = proj(o.data(), S, D, L.wo, D);
  for (size_t i = 0; i < s.size(); ++i) s[i] += y[i];
  const std::vector<double> b = norm_rows(s, S, L.norm2);
  std::vector<double> g = proj(b.data(), S, D, L.wg, FF);
  const std::vector<double> u = proj(b.data(), S, D, L.wu, FF);
  for (size_t i = 0; i < g.size(); ++i) g[i] = silu(g[i]) * u[i];
  const std::vector<double> dn = proj(g.data(), S, FF, L.wd, D);
  for (size_t i = 0; i < s.size(); ++i) s[i] += dn[i];
}

}  // namespace

extern "C" int orc_joint_head(const double* hidden, const uint8_t* key_valid, int64_t T,
                              const double* q_avg, const double* o_avg, const double* g_avg,
                              const double* lexical, const uint8_t* member, const int32_t* type_ids,
                              const uint8_t* q_valid, const uint8_t* o_valid, int64_t Q, int64_t O,
                              const orc_head* w, double* logits, double* probs) {
  if (T < 1 || Q < 1 || O < 1) return fail(-1, "joint head: need T, Q, O >= 1");
  for (int64_t q = 0; q < Q; ++q)
    if (type_ids[q] < 0 || type_ids[q] > 2) return fail(-2, "joint head: type id outside 0..2");
  const int64_t S = Q + O + 1;
  // span means and the global row: u = [q_avg; o_avg; g_avg] . hidden  [S, 4096]
  std::vector<double> pool((size_t)(S * T));
  std::copy(q_avg, q_avg + Q * T, pool.begin());
  std::copy(o_avg, o_avg + O * T, pool.begin() + Q * T);
  std::copy(g_avg, g_avg + T, pool.begin() + (Q + O) * T);
  std::vector<double> u((size_t)(S * HID), 0.0);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < S; ++r)
    for (int64_t t = 0; t < T; ++t) {
      const double p = pool[(size_t)(r * T + t)];
      if (p != 0.0)
        for (int64_t c = 0; c < HID; ++c) u[(size_t)(r * HID + c)] += p * hidden[t * HID + c];
    }
  // slots
  std::vector<double> s = proj(u.data(), S, HID, w->w_in, D);
  const std::vector<double> lex = proj(lexical, O, HID, w->w_lex, D);
  const std::vector<double> e_q = widen(w->e_qtype, 3 * D), e_o = widen(w->e_opt, D),
                            e_g = widen(w->e_glob, D);
  for (int64_t q = 0; q < Q; ++q)
    for (int64_t c = 0; c < D; ++c) s[(size_t)(q * D + c)] += e_q[(size_t)(type_ids[q] * D + c)];
  for (int64_t o = 0; o < O; ++o)
    for (int64_t c = 0; c < D; ++c)
      s[(size_t)((Q + o) * D + c)] += lex[(size_t)(o * D + c)] + e_o[(size_t)c];
  for (int64_t c = 0; c < D; ++c) s[(size_t)((Q + O) * D + c)] += e_g[(size_t)c];
  // the memory: the request's tokens at the head's width
  const std::vector<double> mem = proj(hidden, T, HID, w->w_mem, D);
  std::vector<uint8_t> slot_valid((size_t)S);
  for (int64_t q = 0; q < Q; ++q) slot_valid[(size_t)q] = q_valid[q] ? 1 : 0;
  for (int64_t o = 0; o < O; ++o) slot_valid[(size_t)(Q + o)] = o_valid[o] ? 1 : 0;
  slot_valid[(size_t)(Q + O)] = 1;
  for (int l = 0; l < 4; ++l) layer(s, S, w->dec[l], &mem, T, key_valid, nullptr);
  for (int l = 0; l < 2; ++l) layer(s, S, w->route[l], nullptr, 0, nullptr, slot_valid.data());
  const std::vector<double> f = norm_rows(s, S, w->norm_f);
  // option o's question row c_o = sum_q member[q][o] f_q
  std::vector<double> c((size_t)(O * D), 0.0);
  for (int64_t o = 0; o < O; ++o)
    for (int64_t q = 0; q < Q; ++q)
      if (member[q * O + o])
        for (int64_t d = 0; d < D; ++d) c[(size_t)(o * D + d)] += f[(size_t)(q * D + d)];
  const std::vector<double> a = proj(&f[(size_t)(Q * D)], O, D, w->w_opt, D);
  const std::vector<double> b = proj(c.data(), O, D, w->w_qst, D);
  for (int64_t o = 0; o < O; ++o)
    logits[o] = o_valid[o] ? dot(&a[(size_t)(o * D)], &b[(size_t)(o * D)], D) / std::sqrt((double)D)
                           : 0.0;
  // each valid question's softmax over its valid options
  for (int64_t o = 0; o < O; ++o) probs[o] = 0.0;
  for (int64_t q = 0; q < Q; ++q) {
    if (!q_valid[q]) continue;
    double m = -std::numeric_limits<double>::infinity();
    for (int64_t o = 0; o < O; ++o)
      if (member[q * O + o] && o_valid[o]) m = std::max(m, logits[o]);
    if (m == -std::numeric_limits<double>::infinity()) continue;
    double sum = 0.0;
    for (int64_t o = 0; o < O; ++o)
      if (member[q * O + o] && o_valid[o]) sum += std::exp(logits[o] - m);
    for (int64_t o = 0; o < O; ++o)
      if (member[q * O + o] && o_valid[o]) probs[o] = std::exp(logits[o] - m) / sum;
  }
  return 0;
}
