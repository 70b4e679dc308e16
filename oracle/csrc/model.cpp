// The clef-flash decoder layers and the 32-layer hybrid prefill, oracle side (fp64, test
// infrastructure only).
//
// "Clef-Flash-ANE-LUT6", Model architecture: 32 layers, hidden size 4,096, MLP 12,288; 24 Gated
// DeltaNet layers (16 key and 32 value heads of 128) and 8 full-attention layers (16 query and
// 4 key-value heads of 256), full attention every fourth layer.  Reading of the phase: layers
// 3, 7, ..., 31 are the attention layers (three Gated DeltaNet layers, then one attention layer,
// eight times).  Every large linear is LUT-6 (Weight precision).  Each layer is a pre-norm
// residual block (reading; the pages are silent):  h = x + mixer(rmsnorm(x)),
// y = h + mlp(rmsnorm(h)).  The end-to-end activations have no page to be checked against
// (parity unpinned beyond the pins of the parts and of their composition).
#include <stdio.h>
#include <stdlib.h>

#include "internal.h"

using namespace orc;

namespace {

constexpr int64_t GDN_HK = 16, GDN_HV = 32, GDN_D = 128, GDN_TAPS = 4;
constexpr int64_t ATT_HQ = 16, ATT_HKV = 4, ATT_D = 256;

bool verbose() {
  static const bool v = getenv("ORACLE_VERBOSE") != nullptr;
  return v;
}

int lin(const double* x, int64_t L, int64_t k, const orc_lut6_weight& w, std::vector<double>& y,
        const char* name) {
  if (!w.packed || !w.lut) return fail(-3, "missing LUT-6 weight %s", name);
  if (w.k != k) return fail(-1, "%s: weight has k = %lld, input has %lld", name, (long long)w.k,
                            (long long)k);
  y.assign((size_t)(L * w.n), 0.0);
  return orc_lut6_linear(x, L, k, w.packed, w.lut, w.n, y.data());
}

#define TRY(expr)              \
  do {                         \
    const int _rc = (expr);    \
    if (_rc != 0) return _rc;  \
  } while (0)

}  // namespace

extern "C" {

// SwiGLU MLP: down(SiLU(x W_gate^T) * (x W_up^T)); all three LUT-6 ("Clef-Flash-ANE-LUT6",
// Weight precision lists MLP gate / up / down among the LUT-6 layers).
int orc_swiglu_mlp(const double* xn, int64_t L, int64_t hidden, const orc_layer* w, double* y) {
  std::vector<double> g, u, out;
  TRY(lin(xn, L, hidden, w->gate, g, "mlp gate"));
  TRY(lin(xn, L, hidden, w->up, u, "mlp up"));
  if (w->gate.n != w->up.n) return fail(-1, "mlp: gate and up differ in size");
  for (size_t i = 0; i < g.size(); ++i) g[i] = silu(g[i]) * u[i];
  TRY(lin(g.data(), L, w->gate.n, w->down, out, "mlp down"));
  if (w->down.n != hidden) return fail(-1, "mlp: down must give the hidden size");
  std::copy(out.begin(), out.end(), y);
  return 0;
}

// Gated DeltaNet mixer of one request, xn the normalised input [L, hidden].
// QKV (hidden -> 8192 = q 2048 | k 2048 | v 4096) and Z (-> 4096) are LUT-6; the gate
// projections a, b (-> 32 each) are FP16 ("Clef-Flash-ANE-LUT6", Weight precision).  Conv + SiLU
// on all 8,192 QKV channels, per-head L2 norm of q and k, the gates, the delta rule, the
// z-gated RMSNorm, then the LUT-6 output projection (4096 -> hidden).
int orc_gdn_mixer(const double* xn, int64_t L, int64_t hidden, const orc_layer* w, double* y) {
  const int64_t QK = GDN_HK * GDN_D, V = GDN_HV * GDN_D, C = 2 * QK + V;
  if (!w->a_w || !w->b_w || !w->A_log || !w->dt_bias || !w->conv_w || !w->o_norm)
    return fail(-3, "gdn mixer: a missing FP16 weight");
  std::vector<double> qkv, z;
  TRY(lin(xn, L, hidden, w->qkv, qkv, "gdn qkv"));
  TRY(lin(xn, L, hidden, w->z, z, "gdn z"));
  if (w->qkv.n != C || w->z.n != V) return fail(-1, "gdn mixer: projection sizes");
  // a = xn . W_a^T, b = xn . W_b^T with the FP16 weights widened
  const std::vector<double> a_w = widen(w->a_w, GDN_HV * hidden), b_w = widen(w->b_w, GDN_HV * hidden);
  std::vector<double> a((size_t)(L * GDN_HV)), b((size_t)(L * GDN_HV));
  dense_linear(xn, L, hidden, a_w.data(), GDN_HV, a.data());
  dense_linear(xn, L, hidden, b_w.data(), GDN_HV, b.data());
  // conv + SiLU over the 8,192 channels
  const std::vector<double> conv_w = widen(w->conv_w, C * GDN_TAPS);
  std::vector<double> c((size_t)(L * C));
  orc_conv_silu(qkv.data(), L, C, conv_w.data(), GDN_TAPS, c.data());
  // split: q = c[:, 0:2048], k = c[:, 2048:4096] (each [L, 16, 128], L2-normalised per head),
  // v = c[:, 4096:8192] ([L, 32, 128])
  std::vector<double> q((size_t)(L * QK)), k((size_t)(L * QK)), v((size_t)(L * V));
  for (int64_t t = 0; t < L; ++t) {
    std::copy(c.begin() + t * C, c.begin() + t * C + QK, q.begin() + t * QK);
    std::copy(c.begin() + t * C + QK, c.begin() + t * C + 2 * QK, k.begin() + t * QK);
    std::copy(c.begin() + t * C + 2 * QK, c.begin() + (t + 1) * C, v.begin() + t * V);
  }
  orc_l2norm(q.data(), L * GDN_HK, GDN_D, kL2Eps, q.data());
  orc_l2norm(k.data(), L * GDN_HK, GDN_D, kL2Eps, k.data());
  const std::vector<double> A_log = widen(w->A_log, GDN_HV), dt_bias = widen(w->dt_bias, GDN_HV);
  std::vector<double> alpha((size_t)(L * GDN_HV)), beta((size_t)(L * GDN_HV));
  orc_gdn_gates(a.data(), b.data(), L, GDN_HV, A_log.data(), dt_bias.data(), alpha.data(),
                beta.data());
  std::vector<double> o((size_t)(L * V));
  TRY(orc_gated_delta_rule(q.data(), k.data(), v.data(), alpha.data(), beta.data(), nullptr, L,
                           GDN_HK, GDN_HV, GDN_D, GDN_D, o.data(), nullptr));
  const std::vector<double> o_norm = widen(w->o_norm, GDN_D);
  std::vector<double> yg((size_t)(L * V));
  orc_zgated_norm(o.data(), z.data(), L, GDN_HV, GDN_D, o_norm.data(), kRmsEps, yg.data());
  std::vector<double> out;
  TRY(lin(yg.data(), L, V, w->out, out, "gdn out"));
  if (w->out.n != hidden) return fail(-1, "gdn mixer: out projection size");
  std::copy(out.begin(), out.end(), y);
  return 0;
}

// Gated full-attention mixer of one request, xn [L, hidden].
// Q-proj hidden -> 8192 holds the 16 query heads (columns 0..4095) and the 16 output-gate heads
// (4096..8191): the reading of "gated full-attention layers" ("clef-flash-LiteRT", Provenance)
// that makes the model's stored LUT-6 size match the 4.86 GiB of text programs the
// "Clef-Flash-ANE-LUT6" card gives.  K, V hidden -> 1024 (4 heads x 256); rotary on the first
// 64 dims of q and k; causal GQA softmax; o * sigmoid(gate); O-proj 4096 -> hidden.
int orc_attention_mixer(const double* xn, int64_t L, int64_t hidden, const orc_layer* w,
                        const double* pos, const int64_t* pos3, double* y) {
  const int64_t QD = ATT_HQ * ATT_D, KD = ATT_HKV * ATT_D;
  std::vector<double> qg, kk, vv;
  TRY(lin(xn, L, hidden, w->q, qg, "attention q"));
  TRY(lin(xn, L, hidden, w->k, kk, "attention k"));
  TRY(lin(xn, L, hidden, w->v, vv, "attention v"));
  if (w->q.n != 2 * QD || w->k.n != KD || w->v.n != KD) return fail(-1, "attention: projection sizes");
  std::vector<double> q((size_t)(L * QD)), gate((size_t)(L * QD));
  for (int64_t t = 0; t < L; ++t) {
    std::copy(qg.begin() + t * 2 * QD, qg.begin() + t * 2 * QD + QD, q.begin() + t * QD);
    std::copy(qg.begin() + t * 2 * QD + QD, qg.begin() + (t + 1) * 2 * QD, gate.begin() + t * QD);
  }
  std::vector<double> qr(q.size()), kr(kk.size());
  if (pos3) {
    orc_mrope(q.data(), L, ATT_HQ, ATT_D, pos3, kRopeDims, kRopeTheta, qr.data());
    orc_mrope(kk.data(), L, ATT_HKV, ATT_D, pos3, kRopeDims, kRopeTheta, kr.data());
  } else {
    std::vector<double> ramp((size_t)L);
    for (int64_t t = 0; t < L; ++t) ramp[(size_t)t] = pos ? pos[t] : (double)t;
    orc_rope(q.data(), L, ATT_HQ, ATT_D, ramp.data(), kRopeDims, kRopeTheta, qr.data());
    orc_rope(kk.data(), L, ATT_HKV, ATT_D, ramp.data(), kRopeDims, kRopeTheta, kr.data());
  }
  std::vector<double> o((size_t)(L * QD));
  TRY(orc_causal_attention(qr.data(), kr.data(), vv.data(), L, ATT_HQ, ATT_HKV, ATT_D, 0, L,
                           o.data()));
  for (size_t i = 0; i < o.size(); ++i) o[i] = o[i] * sigmoid(gate[i]);
  std::vector<double> out;
  TRY(lin(o.data(), L, QD, w->o, out, "attention o"));
  if (w->o.n != hidden) return fail(-1, "attention: O projection size");
  std::copy(out.begin(), out.end(), y);
  return 0;
}

// One pre-norm residual decoder layer on one request: x [L, hidden] -> y [L, hidden].
int orc_decoder_layer(const double* x, int64_t L, int64_t hidden, const orc_layer* w,
                      const double* pos, const int64_t* pos3, double* y) {
  if (!w->attn_norm || !w->mlp_norm) return fail(-3, "decoder layer: missing norm weight");
  const std::vector<double> attn_norm = widen(w->attn_norm, hidden);
  const std::vector<double> mlp_norm = widen(w->mlp_norm, hidden);
  const size_t n = (size_t)(L * hidden);
  std::vector<double> xn(n), mix(n), h(n);
  orc_rmsnorm(x, L, hidden, attn_norm.data(), kRmsEps, xn.data());
  if (w->attention)
    TRY(orc_attention_mixer(xn.data(), L, hidden, w, pos, pos3, mix.data()));
  else
    TRY(orc_gdn_mixer(xn.data(), L, hidden, w, mix.data()));
  for (size_t i = 0; i < n; ++i) h[i] = x[i] + mix[i];
  orc_rmsnorm(h.data(), L, hidden, mlp_norm.data(), kRmsEps, xn.data());
  TRY(orc_swiglu_mlp(xn.data(), L, hidden, w, mix.data()));
  for (size_t i = 0; i < n; ++i) y[i] = h[i] + mix[i];
  return 0;
}

int32_t orc_is_attention_layer(int64_t layer) { return layer % 4 == 3 ? 1 : 0; }

// The hybrid prefill of one request.  "clef-flash-LiteRT", Host contract: the embedding rows of
// the request's ids in, every position's output of the final RMSNorm out, each call from an
// empty state.  A request with a picture passes the picture's rows in place of the embedding
// rows where its image tokens sit, and its M-RoPE positions.
int orc_prefill(const double* embed_rows, int64_t L, int64_t hidden, const orc_layer* layers,
                int64_t n_layers, const uint16_t* final_norm, const double* pos,
                const int64_t* pos3, double* hidden_out) {
  if (!final_norm) return fail(-3, "prefill: missing final norm weight");
  std::vector<double> x(embed_rows, embed_rows + L * hidden), next((size_t)(L * hidden));
  for (int64_t l = 0; l < n_layers; ++l) {
    if (layers[l].attention != orc_is_attention_layer(l))
      return fail(-2, "prefill: layer %lld is a %s layer, its weights are for the other kind",
                  (long long)l, orc_is_attention_layer(l) ? "full-attention" : "Gated DeltaNet");
    TRY(orc_decoder_layer(x.data(), L, hidden, &layers[l], pos, pos3, next.data()));
    x.swap(next);
    if (verbose()) fprintf(stderr, "oracle prefill: layer %lld of %lld done\n", (long long)l + 1,
                           (long long)n_layers);
  }
  const std::vector<double> w = widen(final_norm, hidden);
  orc_rmsnorm(x.data(), L, hidden, w.data(), kRmsEps, hidden_out);
  return 0;
}

}  // extern "C"
