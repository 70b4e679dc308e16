/*
 * The oracle's C ABI: a plain, slow, fp64 CPU restatement of the clef-flash hybrid prefill.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the CPU legs of bench.py
 * load liboracle.so (through oracle/_lib.py).  It shares no code with the CUDA library: no
 * header, helper, table or constant generator of either side is used by the other.
 *
 * Conventions.  Floating-point inputs and outputs are double (fp16 weights are passed as their
 * IEEE binary16 bit patterns, uint16_t, and widened exactly).  Arrays are dense, row-major, and
 * owned by the caller; nothing here keeps a pointer past the call.  Functions that can fail
 * return 0 on success and a negative code on bad sizes or missing weights (-1 shape, -2 value,
 * -3 missing weight), with a message in orc_last_error().
 *
 * Sources, cited by page title and section:
 *   "Clef-Flash-ANE-LUT6" (Hugging Face model card): Model architecture (32 layers, hidden
 *     4,096, MLP 12,288, 24 Gated DeltaNet + 8 full-attention layers, full attention every fourth
 *     layer); Weight precision (which weights are LUT-6 and which FP16); LUT-6 text weights (the
 *     format, the 6.02 bits per weight, the 40-round k-means quantiser).
 *   "clef-flash - Core AI" (README): Core AI shape (decoder inputs, the conv and recurrent
 *     states, 64-position calls, the final hidden rows).
 *   "clef-flash-LiteRT" (README): Host contract (rotary theta 1e7, the three M-RoPE planes,
 *     text positions (i, i, i), the final norm's output per position); Provenance (the
 *     GatedDeltaNet recurrence, grouped keys/values repeated, gated full-attention layers).
 */
#ifndef CLEF_ORACLE_H
#define CLEF_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

const char* orc_last_error(void);
int32_t orc_num_threads(void);

/* ------------------------------------------------------------------ LUT-6 ("LUT-6 text weights")
 * Four 6-bit indices i0..i3 make the 24-bit word w = i0 | i1 << 6 | i2 << 12 | i3 << 18, stored
 * as the bytes w & 255, (w >> 8) & 255, w >> 16 (the card's "little-endian, as Core ML does",
 * read as one LSB-first bit stream over W row-major, input index fastest); table g (64 fp16
 * values) serves output rows 16g .. 16g + 15. */
int orc_lut6_pack(const uint8_t* idx, int64_t n, int64_t k, uint8_t* packed);
int orc_lut6_unpack(const uint8_t* packed, int64_t n, int64_t k, uint8_t* idx);
int orc_lut6_dequant(const uint8_t* packed, const uint16_t* lut, int64_t n, int64_t k, double* w);
int orc_lut6_dequant_f16(const uint8_t* packed, const uint16_t* lut, int64_t n, int64_t k,
                         uint16_t* w);
/* y [m, n] = x [m, k] . W^T, W the dequantised [n, k] weight, every product and sum in fp64 */
int orc_lut6_linear(const double* x, int64_t m, int64_t k, const uint8_t* packed,
                    const uint16_t* lut, int64_t n, double* y);
/* bits stored for an n x k layer: 6 per weight plus 64 fp16 entries per 16 rows */
int64_t orc_lut6_storage_bits(int64_t n, int64_t k);

/* ------------------------------------------------------------------ element-wise and norms */
void orc_silu(const double* x, int64_t n, double* y);
void orc_sigmoid(const double* x, int64_t n, double* y);
void orc_softplus(const double* x, int64_t n, double* y);
/* per row of d: x / sqrt(mean(x^2) + eps) * w (w may be NULL: 1) */
void orc_rmsnorm(const double* x, int64_t rows, int64_t d, const double* w, double eps, double* y);
/* per row of d: x / sqrt(sum(x^2) + eps) */
void orc_l2norm(const double* x, int64_t rows, int64_t d, double eps, double* y);

/* ------------------------------------------------------------------ Gated DeltaNet pieces */
/* causal depthwise conv (taps per channel, zero history) then SiLU; x, y [L, C]; w [C, taps] */
void orc_conv_silu(const double* x, int64_t L, int64_t C, const double* w, int64_t taps, double* y);
/* alpha = exp(-exp(A_log) softplus(a + dt_bias)), beta = sigmoid(b); a, b, alpha, beta [L, H] */
void orc_gdn_gates(const double* a, const double* b, int64_t L, int64_t H, const double* A_log,
                   const double* dt_bias, double* alpha, double* beta);
/* The per-token recurrence, value head h reading key head h / (Hv / Hk):
 *   S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,  o_t = S_t q_t / sqrt(dk)
 * q, k [L, Hk, dk]; v [L, Hv, dv]; alpha, beta [L, Hv]; s0 [Hv, dv, dk] or NULL (zero);
 * o [L, Hv, dv]; s_out [Hv, dv, dk] or NULL. */
int orc_gated_delta_rule(const double* q, const double* k, const double* v, const double* alpha,
                         const double* beta, const double* s0, int64_t L, int64_t Hk, int64_t Hv,
                         int64_t dk, int64_t dv, double* o, double* s_out);
/* per head of d values: rmsnorm(o, w) * SiLU(z); o, z, y [L, H, d]; w [d] */
void orc_zgated_norm(const double* o, const double* z, int64_t L, int64_t H, int64_t d,
                     const double* w, double eps, double* y);

/* ------------------------------------------------------------------ rotary and attention */
/* 1-D rotary on the first rot_dims dims of each head: pair (j, j + rot_dims / 2) turns by
 * pos[t] * theta^(-2j / rot_dims); x, y [L, H, D] */
void orc_rope(const double* x, int64_t L, int64_t H, int64_t D, const double* pos,
              int64_t rot_dims, double theta, double* y);
/* plane (0 = t, 1 = h, 2 = w) of each frequency pair: j mod 3 */
void orc_mrope_planes(int64_t rot_dims, int64_t* planes);
/* [L, 3] positions of a request holding at most one grid_h x grid_w picture block at
 * image_start (grid_h * grid_w == 0: text only) */
int orc_mrope_positions(int64_t L, int64_t image_start, int64_t grid_h, int64_t grid_w,
                        int64_t* pos3);
/* M-RoPE: pair j turns by pos3[t][plane(j)] * theta^(-2j / rot_dims) */
void orc_mrope(const double* x, int64_t L, int64_t H, int64_t D, const int64_t* pos3,
               int64_t rot_dims, double theta, double* y);
/* causal softmax attention, one explicit softmax per query row; query head h reads kv head
 * h / (Hq / Hkv); logits q.k / sqrt(D); row t sees keys 0..t.  Only query rows row0 .. row1 - 1
 * are computed: o is [row1 - row0, Hq, D]. */
int orc_causal_attention(const double* q, const double* k, const double* v, int64_t L, int64_t Hq,
                         int64_t Hkv, int64_t D, int64_t row0, int64_t row1, double* o);

/* ------------------------------------------------------------------ the decoder */
typedef struct {
  const uint8_t* packed;  /* [n, k * 3 / 4] canonical 4-in-3 packing */
  const uint16_t* lut;    /* [n / 16, 64] fp16 bits */
  int64_t n, k;
} orc_lut6_weight;

/* One decoder layer's weights (fp16 bit patterns; NULL / zero-sized where unused). */
typedef struct {
  int32_t attention;                 /* 0: Gated DeltaNet layer, 1: gated full-attention layer */
  const uint16_t* attn_norm;         /* [hidden] */
  const uint16_t* mlp_norm;          /* [hidden] */
  /* Gated DeltaNet: QKV (q 2048 | k 2048 | v 4096), Z, out; a/b projections [32, hidden];
   * A_log, dt_bias [32]; conv [8192, 4]; o_norm [128] */
  orc_lut6_weight qkv, z, out;
  const uint16_t *a_w, *b_w, *A_log, *dt_bias, *conv_w, *o_norm;
  /* attention: Q (16 query heads | 16 gate heads, x 256), K, V (4 heads x 256), O */
  orc_lut6_weight q, k, v, o;
  /* SwiGLU MLP */
  orc_lut6_weight gate, up, down;
} orc_layer;

/* Rotary positions of an attention layer: pos [L] (1-D), or pos3 [L, 3] (M-RoPE planes), or
 * neither (0 .. L - 1). */
int orc_swiglu_mlp(const double* xn, int64_t L, int64_t hidden, const orc_layer* w, double* y);
int orc_gdn_mixer(const double* xn, int64_t L, int64_t hidden, const orc_layer* w, double* y);
int orc_attention_mixer(const double* xn, int64_t L, int64_t hidden, const orc_layer* w,
                        const double* pos, const int64_t* pos3, double* y);
int orc_decoder_layer(const double* x, int64_t L, int64_t hidden, const orc_layer* w,
                      const double* pos, const int64_t* pos3, double* y);
/* 1 where layer l is a full-attention layer (l % 4 == 3), else 0 */
int32_t orc_is_attention_layer(int64_t layer);
/* The prefill of one request: embedding rows [L, hidden] in, every position's final-norm
 * hidden state [L, hidden] out.  layers[l].attention must agree with orc_is_attention_layer. */
int orc_prefill(const double* embed_rows, int64_t L, int64_t hidden, const orc_layer* layers,
                int64_t n_layers, const uint16_t* final_norm, const double* pos,
                const int64_t* pos3, double* hidden_out);

/* ------------------------------------------------------------------ the LUT-6 quantiser */
/* The 32 quantile seeds and the 32 evenly spread seeds of one group's n values */
void orc_quant_quantiles(const double* values, int64_t n, double* out32);
void orc_quant_spread(const double* values, int64_t n, double* out32);
/* the 64 starting centroids, ascending (stable: quantiles before equal spread values) */
void orc_quant_initial_table(const double* values, int64_t n, double* out64);
/* nearest of the ascending centroids c [nc]: lower index on a tie, first of equal centroids */
void orc_quant_assign(const double* values, int64_t n, const double* c, int64_t nc, int64_t* cell);
/* one k-means round over ascending centroids c [nc] (in place) */
void orc_quant_kmeans_round(const double* values, int64_t n, double* c, int64_t nc);
/* one group: fp16 table [64] (bits) and every value's index */
void orc_quant_group(const double* values, int64_t n, int32_t rounds, uint16_t* table,
                     uint8_t* idx);
/* w [n, k] fp16 bits -> packed [n, k * 3 / 4], lut [n / 16, 64] fp16 bits */
int orc_lut6_quantize(const uint16_t* w, int64_t n, int64_t k, int32_t rounds, uint8_t* packed,
                      uint16_t* lut);

/* ------------------------------------------------------------------ the joint schema head
 * "clef-flash - Core AI" README, Readout contract and Core AI shape (Head): the head reads the
 * final-norm hidden rows of one request; q_avg [Q, T] and o_avg [O, T] average them over each
 * question's and option's span (1 / len on the span), g_avg [T] picks the last real token,
 * lexical [O, 4096] is each option's mean lm_head row, member [Q, O] says which question an
 * option belongs to; the output is one logit per option, and each question's probabilities are
 * a softmax over its options.  "Clef-Flash-ANE-LUT6", Model architecture: 4 layers, width 1,024,
 * 16 heads, 2 routing layers ("clef-flash-LiteRT", Host contract step 7: 2 routing layers and 4
 * decoder layers over the request's tokens).  The layers themselves are not on the pages; their
 * form here is a reading (orc_joint_head in head.cpp states it). */
typedef struct {
  const uint16_t* norm1;             /* [1024] */
  const uint16_t *wq, *wk, *wv, *wo; /* [1024, 1024] */
  const uint16_t* norm2;             /* [1024] */
  const uint16_t *wg, *wu;           /* [4096, 1024] */
  const uint16_t* wd;                /* [1024, 4096] */
} orc_head_layer;

typedef struct {
  const uint16_t *w_mem, *w_in, *w_lex; /* [1024, 4096] */
  const uint16_t* e_qtype;              /* [3, 1024] question types noul / choice / score */
  const uint16_t *e_opt, *e_glob;       /* [1024] */
  orc_head_layer dec[4];                /* decoder layers: slots attend to the request's tokens */
  orc_head_layer route[2];              /* routing layers: slots attend to each other */
  const uint16_t* norm_f;               /* [1024] */
  const uint16_t *w_opt, *w_qst;        /* [1024, 1024] */
} orc_head;

/* hidden [T, 4096]; key_valid [T]; q_avg [Q, T]; o_avg [O, T]; g_avg [T]; lexical [O, 4096];
 * member [Q, O] (0 / 1); type_ids [Q] in 0..2; q_valid [Q]; o_valid [O]; out: logits [O] and
 * probs [O] (0 for an option of no valid question, or an invalid option). */
int orc_joint_head(const double* hidden, const uint8_t* key_valid, int64_t T, const double* q_avg,
                   const double* o_avg, const double* g_avg, const double* lexical,
                   const uint8_t* member, const int32_t* type_ids, const uint8_t* q_valid,
                   const uint8_t* o_valid, int64_t Q, int64_t O, const orc_head* w,
                   double* logits, double* probs);

#ifdef __cplusplus
}
#endif

#endif /* CLEF_ORACLE_H */
