/*
 * clef.h - C ABI of the GB300 (sm_103a) prefill library for the clef-flash hybrid decoder.
 *
 * The model: the clef-flash text backbone ("Clef-Flash-ANE-LUT6" model card, section "Model
 * architecture"): 32 layers of hidden size 4,096 and MLP size 12,288; 24 Gated DeltaNet layers
 * (16 key / 32 value heads of 128) and 8 gated full-attention layers (16 query / 4 kv heads of
 * 256), full attention every fourth layer.  Every large linear is LUT-6 (section "LUT-6 text
 * weights"): a 6-bit index per weight, an fp16 table of 64 values for each block of 16 output
 * channels, 4 indices to 3 bytes.  One call of clef_prefill_forward is one single prefill: token
 * ids in, every position's output of the final RMSNorm out ("clef-flash-LiteRT" README, section "Host
 * contract", steps 3-6; each call starts from an empty state).
 *
 * Conventions of every entry point:
 *   - All buffers are owned by the caller.  The library never allocates device memory; calls
 *     that need scratch take a caller-provided workspace (see the *_workspace_size queries).
 *   - "device" pointers point to memory of the current CUDA device; "host" pointers to host
 *     memory.  fp16 tensors are passed as uint16_t bit patterns (IEEE binary16).
 *   - Tensors are dense and row-major, last index fastest, with the shapes given per call.
 *   - Device calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default stream).
 *     Arguments are validated on the host before anything is launched; on a validation error
 *     nothing is launched and the call returns the error.
 *   - Device pointers must be 16-byte aligned (CLEF_E_ALIGN otherwise).
 *   - Kernels never trap.  A device-side problem (a wait that ran out, a token id outside the
 *     vocabulary) is written to a device status word that clef_sync_status() reads.
 *   - Error messages: clef_last_error() returns the message of the last failing call on the
 *     calling thread.
 *   - Calls are reentrant given distinct output buffers and workspaces.
 */
#ifndef CLEF_H_
#define CLEF_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CLEF_API __attribute__((visibility("default")))
#else
#define CLEF_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  CLEF_OK = 0,
  CLEF_E_INVALID = 1,          /* NULL pointer, negative size, bad enum, index out of range  */
  CLEF_E_SHAPE = 2,            /* a size the call does not support (see each call)           */
  CLEF_E_TOO_LONG = 3,         /* more than CLEF_MAX_LEN positions: refused, never cut       */
  CLEF_E_ALIGN = 4,            /* a device pointer not 16-byte aligned                       */
  CLEF_E_CUDA = 5,             /* a CUDA runtime/driver call failed                          */
  CLEF_E_DEVICE_TIMEOUT = 6,   /* a device wait ran out (from clef_sync_status)              */
  CLEF_E_NONFINITE = 7,        /* not finite: a quantiser weight, or a prefill's hidden row
                                  (from clef_sync_status; see clef_check_finite)             */
  CLEF_E_WORKSPACE = 8,        /* workspace smaller than the size query returned             */
  CLEF_E_BAD_TOKEN = 9         /* a token id outside [0, vocab) (from clef_sync_status)      */
} clef_status;

/* Model constants (clef-flash text backbone). */
#define CLEF_HIDDEN 4096
#define CLEF_INTER 12288
#define CLEF_GDN_HK 16
#define CLEF_GDN_HV 32
#define CLEF_GDN_D 128
#define CLEF_ATT_HQ 16
#define CLEF_ATT_HKV 4
#define CLEF_ATT_D 256
#define CLEF_ROPE_DIMS 64
/* Longest prefill the provider's code reads ("clef-flash-LiteRT" README, section "Limits"). */
#define CLEF_MAX_LEN 16384
/* Rows per block in the interleaved gate/up weight of the SwiGLU MLP (see clef_layer). */
#define CLEF_SWIGLU_BLOCK 16

typedef void* clef_stream; /* a cudaStream_t */

/* Message of the last failing call on this thread ("" if none). */
CLEF_API const char* clef_last_error(void);

/* ABI version: (major << 16) | minor.  1.1 adds the chunked prefill with carried state, the
   LUT-6 quantiser and the picture prefill with M-RoPE to 1.0; nothing of 1.0 changed. */
CLEF_API int32_t clef_version(void);

/* ------------------------------------------------------------------------------------------
 * LUT-6 format ("Clef-Flash-ANE-LUT6" model card, sections "Weight precision" and "LUT-6 text
 * weights").  A weight matrix W [n, k] (n output channels, k inputs) is stored as
 *   packed [n, k*3/4] uint8: the 6-bit indices idx[n][k] as one LSB-first bit stream in
 *          row-major order (k fastest); indices i0..i3 of a quadruple form the 24-bit word
 *          i0 | i1<<6 | i2<<12 | i3<<18, stored as its three little-endian bytes;
 *   lut    [n/16, 64] fp16: table g serves output rows 16g .. 16g+15;
 *   W[r][c] = lut[r/16][idx[r][c]].
 * ------------------------------------------------------------------------------------------ */

/* host: pack idx [n, k] (each < 64; k % 4 == 0) into packed [n, k*3/4].  Host buffers, caller
   owned.  CLEF_E_INVALID for an index >= 64 or a NULL pointer, CLEF_E_SHAPE if k % 4 != 0. */
CLEF_API clef_status clef_lut6_pack(const uint8_t* idx, int64_t n, int64_t k, uint8_t* packed);

/* host: the inverse of clef_lut6_pack. */
CLEF_API clef_status clef_lut6_unpack(const uint8_t* packed, int64_t n, int64_t k, uint8_t* idx);

/* device: w [n, k] fp16 = the dequantised LUT-6 weight (bit-exact table values).  n % 16 == 0,
   k % 4 == 0.  A debugging / parity aid; the GEMM never materialises W. */
CLEF_API clef_status clef_lut6_dequant(const uint8_t* packed, const uint16_t* lut, int64_t n, int64_t k,
                              uint16_t* w, clef_stream stream);

/* device: tiled [n, k*3/4] = the same bytes as `packed` rearranged into the LUT-6 GEMM's operand
   layout (n % 16 == 0, k % 64 == 0; CLEF_E_SHAPE otherwise).  For each 16-row group G and each
   64-wide block kb of k, a 768-byte block at ((G * k/64) + kb) * 768 holds, for t = 0..31, the
   24 bytes t*24 ..: the 3-byte quadruples (16kb + 4j + t%4, j = 0..3) of row 16G + t/4, then of
   row 16G + t/4 + 8.  No bit changes; only whole quadruples move.  Done once per weight. */
CLEF_API clef_status clef_lut6_tile(const uint8_t* packed, int64_t n, int64_t k, uint8_t* tiled,
                                    clef_stream stream);

/* device: quantise an fp16 weight w [n, k] (row-major, k fastest) into the LUT-6 format above:
   packed [n, k*3/4] (the row-major bit stream of clef_lut6_pack) and lut [n/16, 64] fp16
   ("Clef-Flash-ANE-LUT6" model card, section "LUT-6 text weights": per 16-row group, 40 k-means
   iterations in one dimension from 64 initial centroids, 32 quantiles of the group and 32 equal
   steps from its smallest to its largest weight).  Arithmetic, fixed so that the result
   is one exact function of w: quantile i (p = (i + 1/2) / 32) interpolates linearly between the
   order statistics around p (n - 1); spread value i is min + i * ((max - min) / 31), the last
   one max; each round sends a weight to the nearest centroid (cells between midpoints
   fl(c_j + c_j+1) / 2 of the ascending centroids; a tie, or several equal centroids, to the
   lowest index) and moves each centroid with members to fl(S / count), S their exact sum; a
   centroid without members stays; the centroids are then sorted again (stable).  The table is the centroids rounded to fp16, ascending; each
   index points at the nearest table entry (ties to the lowest index).  n % 16 == 0, k % 4 == 0,
   0 < k <= 262144 (CLEF_E_SHAPE otherwise); device pointers, 16-byte aligned, caller owned.
   A non-finite weight is left out of the tables and reported as CLEF_E_NONFINITE by
   clef_sync_status.  Asynchronous on `stream`. */
CLEF_API clef_status clef_lut6_quantize(const uint16_t* w, int64_t n, int64_t k, uint8_t* packed,
                                        uint16_t* lut, clef_stream stream);

/* device: y [m, n] = x [m, k] . W^T, fp32 accumulation; y is fp16 (y_is_fp32 = 0) or fp32
   (y_is_fp32 = 1); W given as `tiled` (clef_lut6_tile) and lut.  The weights are dequantised
   into tensor memory and used there as the A operand of tcgen05 MMAs (Y^T = W X^T); W is never
   written to global memory.  Requirements: m >= 0 (m == 0 is a no-op and x, y may then be NULL),
   n % 16 == 0, k % 64 == 0, k > 0 (CLEF_E_SHAPE otherwise).  x, tiled, lut, y device, 16-byte
   aligned. */
CLEF_API clef_status clef_lut6_gemm(const uint16_t* x, const uint8_t* tiled, const uint16_t* lut,
                                    void* y, int32_t y_is_fp32, int64_t m, int64_t n, int64_t k,
                                    clef_stream stream);

/* device: the same product with W given in the card's own 4-in-3 packing (`packed` [n, k*3/4],
   the row-major bit stream of clef_lut6_pack).  The GEMM's tensor-memory dequantisation reads a
   lane's 32 indices of one k-block as 24 contiguous bytes, which the card's row-major stream
   does not give, so this call first writes the tiled permutation (clef_lut6_tile) into the
   caller's workspace, then runs clef_lut6_gemm on it: one extra pass over the packed bytes per
   call.  A caller that multiplies by the same weight many times should tile it once and call
   clef_lut6_gemm.  workspace: device, >= clef_lut6_gemm_canonical_workspace_size(n, k) bytes,
   16-byte aligned (CLEF_E_WORKSPACE if smaller).  Other requirements as clef_lut6_gemm. */
CLEF_API size_t clef_lut6_gemm_canonical_workspace_size(int64_t n, int64_t k);
CLEF_API clef_status clef_lut6_gemm_canonical(const uint16_t* x, const uint8_t* packed,
                                              const uint16_t* lut, void* y, int32_t y_is_fp32,
                                              int64_t m, int64_t n, int64_t k, void* workspace,
                                              size_t workspace_bytes, clef_stream stream);

/* ------------------------------------------------------------------------------------------
 * Gated DeltaNet scan ("Clef-Flash-ANE-LUT6" section "Model architecture"; "clef-flash - Core
 * AI" README, section "Core AI shape": recurrent state [.., 32, 128, 128] per layer;
 * "clef-flash-LiteRT" section "Provenance": the recurrence evaluated in chunks of 64 positions).
 * For value head h (key head h/2), from S_0 (zero, or s0):
 *     S_t = alpha_t S_{t-1} + beta_t (v_t - alpha_t S_{t-1} k_t) k_t^T,   o_t = S_t q_t / sqrt(128)
 * q, k [B, L, 16, 128] fp16 (already convolved and L2-normalised), v [B, L, 32, 128] fp16,
 * alpha, beta [B, L, 32] fp32 with 0 <= alpha <= 1; o [B, L, 32, 128] fp16.
 * s0 [B, 32, 128, 128] fp32 (row = value dim, column = key dim) or NULL for a zero state;
 * s_out (same shape) receives S_L, or NULL.  L <= CLEF_MAX_LEN.  Needs a workspace of
 * clef_gdn_workspace_size(B, L) bytes (device, 256-byte aligned).
 * ------------------------------------------------------------------------------------------ */
CLEF_API size_t clef_gdn_workspace_size(int64_t B, int64_t L);
CLEF_API clef_status clef_gdn_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                             const float* alpha, const float* beta, const float* s0, uint16_t* o,
                             float* s_out, int64_t B, int64_t L, void* workspace,
                             size_t workspace_bytes, clef_stream stream);

/* The same scan for callers that cannot allocate device memory (no counterpart on the pages; an
 * interface convenience).  Some hosts cannot call cudaMalloc: a plugin inside a runtime that owns
 * the device allocator, or code that must not allocate once it is serving.  This call takes the
 * same inputs and outputs as clef_gdn_prefill but no workspace: its scratch is one array of
 * CLEF_GDN_NOALLOC_SCRATCH_BYTES (64 MiB) with static storage in the library, which every GPU
 * that loads the library keeps reserved until the process exits.  Sizes whose scratch
 * (clef_gdn_workspace_size(B, L), about 37 KB per position) exceeds it are refused with
 * CLEF_E_SHAPE; one request of up to 1,024 positions always fits.  The first call on a device looks up the array's device address (with that device
 * current), so make that first call before any stream capture.  All calls share the one array
 * and it keeps the last call's contents; nothing in it has to start at zero.  Two calls that run
 * on the GPU at the same time (other streams, other threads) race on it: serialise them.
 * Results equal clef_gdn_prefill's bit for bit. */
#define CLEF_GDN_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
CLEF_API clef_status clef_gdn_prefill_noalloc(const uint16_t* q, const uint16_t* k,
                                              const uint16_t* v, const float* alpha,
                                              const float* beta, const float* s0, uint16_t* o,
                                              float* s_out, int64_t B, int64_t L,
                                              clef_stream stream);

/* ------------------------------------------------------------------------------------------
 * Causal GQA attention of a gated full-attention layer ("Clef-Flash-ANE-LUT6" section "Model
 * architecture": 16 query and 4 kv heads of 256; "clef-flash-LiteRT" section "Host contract"
 * step 5: rotary theta 1e7, text positions (i, i, i); "clef-flash-coreml": cos/sin [L, 64]).
 * q [B, L, 16, 256], k, v [B, L, 4, 256] fp16, before rotary; rotary (rotate-half pairs
 * (j, j+32), angle pos * 1e7^(-j/32)) is applied to dims 0..63 of q and k with pos = 0..L-1;
 * query head h reads kv head h/4; P = softmax(q k^T / 16 + causal mask); o = P v.
 * gate [B, L, 16, 256] fp16 or NULL: o <- o * sigmoid(gate).  o [B, L, 16, 256] fp16.
 * q, k, v and gate may be row-strided: row_stride_* is the element distance between positions
 * (e.g. 10240 when they are column slices of one projection output); 0 means packed.
 * Needs a workspace of clef_attn_workspace_size(B, L) bytes (device; the rotated copies of q, k).
 * ------------------------------------------------------------------------------------------ */
CLEF_API size_t clef_attn_workspace_size(int64_t B, int64_t L);
CLEF_API clef_status clef_gqa_attn_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                           const uint16_t* gate, uint16_t* o, int64_t B, int64_t L,
                                           int64_t row_stride_q, int64_t row_stride_kv,
                                           int64_t row_stride_gate, void* workspace,
                                           size_t workspace_bytes, clef_stream stream);

/* ------------------------------------------------------------------------------------------
 * The model.  All pointers are device pointers except `layers` (a host array).
 * ------------------------------------------------------------------------------------------ */
typedef struct {
  const uint8_t* packed; /* [n, k*3/4] in the tiled layout of clef_lut6_tile */
  const uint16_t* lut;   /* [n/16, 64] fp16 */
} clef_lut6;

typedef enum { CLEF_LAYER_GDN = 0, CLEF_LAYER_ATTENTION = 1 } clef_layer_kind;

typedef struct {
  int32_t kind;              /* clef_layer_kind */
  const uint16_t* attn_norm; /* [4096] fp16 pre-mixer RMSNorm weight */
  const uint16_t* mlp_norm;  /* [4096] fp16 pre-MLP RMSNorm weight */
  /* GDN: rows [q 2048 | k 2048 | v 4096 | z 4096] = [12288, 4096].
     attention: rows [query 4096 | gate 4096 | k 1024 | v 1024] = [10240, 4096]. */
  clef_lut6 in_proj;
  clef_lut6 out_proj;        /* [4096, 4096] */
  /* MLP gate and up, interleaved in blocks of CLEF_SWIGLU_BLOCK (16) rows, one table group
     each: rows [32j, 32j+16) are gate rows [16j, 16j+16), rows [32j+16, 32j+32) are up rows
     [16j, 16j+16).  [24576, 4096]. */
  clef_lut6 gate_up;
  clef_lut6 down;            /* [4096, 12288] */
  /* GDN only (NULL for attention layers), fp16: */
  const uint16_t* ab_w;      /* [64, 4096]: rows 0..31 = a projection, 32..63 = b projection */
  const uint16_t* A_log;     /* [32] */
  const uint16_t* dt_bias;   /* [32] */
  const uint16_t* conv_w;    /* [8192, 4] depthwise causal conv taps, tap 3 = current position */
  const uint16_t* o_norm;    /* [128] z-gated RMSNorm weight, shared by the 32 heads */
} clef_layer;

typedef struct {
  int32_t n_layers;          /* 32 for clef-flash; 1..64 accepted */
  const clef_layer* layers;  /* host array [n_layers] */
  const uint16_t* embed;     /* [vocab, 4096] fp16 token embeddings */
  int64_t vocab;             /* 248320 for clef-flash */
  const uint16_t* final_norm;/* [4096] fp16 */
  int32_t flags;             /* 0, or CLEF_MODEL_REPRODUCIBLE */
} clef_model;

/* clef_model.flags: make every run of the same prefill give the same bits.  Short prefills
   split the residual-add projections (out-proj, MLP down) over k-parts to fill the GPU; by
   default each part adds its partial sum into the fp32 residual as it finishes, so the order of
   those fp32 additions (and the last bits of the result) can change from run to run.  With this
   flag each part writes its sums to the workspace and one more kernel adds them in part order.
   Long prefills (no split) are reproducible either way. */
#define CLEF_MODEL_REPRODUCIBLE 1

/* Bytes of workspace clef_prefill_forward / clef_decoder_layer need for B requests of L
   positions. */
CLEF_API size_t clef_prefill_workspace_size(int64_t B, int64_t L);

/* device: the hybrid prefill.  ids [B, L] int32 (device) -> hidden [B, L, 4096] fp16, the final
   RMSNorm's output for each position.  B independent requests of L positions each
   (right-padded to a bucket by the caller: padding rows are computed like real tokens and, by
   causality, never change the real rows).  1 <= L <= CLEF_MAX_LEN (CLEF_E_TOO_LONG above),
   B >= 1.  Ids outside [0, vocab) set CLEF_E_BAD_TOKEN in the device status (their rows are
   zero).  Residual stream in fp32, activations between kernels in fp16.  A hidden row that is
   not finite (an activation overflowed fp16, or an embedding or picture row held inf / NaN)
   sets CLEF_E_NONFINITE in the device status, naming the lowest such row: the request is to be
   rejected, as the pages reject inputs that overflow FP16 (see clef_check_finite). */
CLEF_API clef_status clef_prefill_forward(const clef_model* model, const int32_t* ids, int64_t B, int64_t L,
                                 uint16_t* hidden, void* workspace, size_t workspace_bytes,
                                 clef_stream stream);

/* M-RoPE positions of one request of L tokens holding at most one picture block
   ("clef-flash-LiteRT" README, "Host contract" step 5: three planes, theta = 1e7; text tokens sit
   at (i, i, i) for their index i, picture tokens at their grid row and column;
   "clef-flash - Core AI" README, "Core AI shape": image token k at row k / W, column k % W, and
   from the <|vision_end|> index image_start + N on the positions move back by N - max(H, W)).
   host: pos3 [L][3] int32 (t, h, w), caller owned: image token k (index image_start + k,
   k < N = grid_h * grid_w) gets (image_start, image_start + k / grid_w, image_start + k % grid_w).
   grid_h = grid_w = 0: text only.  CLEF_E_INVALID for bad sizes or a NULL pos3, CLEF_E_SHAPE if
   the picture does not fit in L. */
CLEF_API clef_status clef_mrope_positions(int64_t L, int64_t image_start, int64_t grid_h,
                                          int64_t grid_w, int32_t* pos3);

/* device: clef_prefill_forward for B requests that each hold one picture block of
   grid_h x grid_w tokens at token indices image_start .. image_start + N - 1 (the
   <|image_pad|> tokens; "clef-flash-LiteRT" README, "Host contract" steps 4-5).  Those rows take
   image_rows [B, N, 4096] fp16 (device; the vision tower's merged rows, request-major) instead of
   embedding rows, and the attention layers' rotary uses the M-RoPE positions of
   clef_mrope_positions: frequency pair j (of 32) turns by the position on plane j mod 3
   (sections 11 / 11 / 10, interleaved).  grid_h = grid_w = 0 (image_rows may be NULL) is
   clef_prefill_forward.  Same workspace as clef_prefill_forward.  CLEF_E_INVALID for bad grid
   sizes or a NULL / misaligned image_rows, CLEF_E_SHAPE if the picture does not fit in L. */
CLEF_API clef_status clef_prefill_forward_image(const clef_model* model, const int32_t* ids,
                                                int64_t B, int64_t L, const uint16_t* image_rows,
                                                int64_t image_start, int64_t grid_h,
                                                int64_t grid_w, uint16_t* hidden, void* workspace,
                                                size_t workspace_bytes, clef_stream stream);

/* ------------------------------------------------------------------------------------------
 * Joint schema head on the hidden states of one request ("clef-flash - Core AI" README,
 * sections "Readout contract" and "Core AI shape", Head; "Clef-Flash-ANE-LUT6", section "Model
 * architecture": 4 layers of width 1,024, 16 heads, 2 routing layers; "clef-flash-LiteRT",
 * section "Host contract" step 7).  What the pages fix: the inputs (the request's final-norm
 * hidden rows; the span means q_avg [Q, T] and o_avg [O, T] with 1 / len over each span; g_avg
 * [T] picking the last real token; lexical [O, 4096], each option's mean lm_head row; member
 * [Q, O], which question each option belongs to; question types; validity of keys, questions and
 * options), one logit per option out, and each question's probabilities a float32 softmax over
 * its options.  The layers between are this library's reading (the pages do not give them),
 * with width 1,024 and 16 heads of 64:
 *   slots (Q questions, O options, 1 global row) = span means . W_in^T (4096 -> 1024), plus the
 *     question-type embedding, plus (options) lexical . W_lex^T and an option embedding, plus
 *     (global) a global embedding; memory = hidden . W_mem^T (4096 -> 1024);
 *   4 decoder layers: s += Attention(rmsnorm(s) -> q; memory -> k, v; valid keys only) . W_o^T,
 *     then s += SwiGLU(rmsnorm(s)) (1024 -> 4096 -> 1024);
 *   2 routing layers: the same with the slots attending to the valid slots;
 *   f = rmsnorm(s); logit_o = (f_o W_opt^T) . (f_q(o) W_qst^T) / 32, q(o) the question of o;
 *   RMSNorm eps 1e-6; attention scale 1/8; invalid options get logit 0 and probability 0.
 * Weights: fp16, [out, in] row-major, device, 16-byte aligned, caller owned.
 * hidden [T, 4096] fp16 (the prefill's output for one request); key_valid [T], member [Q][O],
 * q_valid [Q], o_valid [O] uint8 (0 / 1); type_ids [Q] int32 in 0..2 (others clamp); q_avg, o_avg, g_avg,
 * lexical fp32; out logits [O], probs [O] fp32.  All device, caller owned.  1 <= T <=
 * CLEF_MAX_LEN, 1 <= Q <= 16, 1 <= O <= 128 (the pages' head pads to 16 questions and 128
 * options); CLEF_E_SHAPE otherwise.  Workspace: clef_joint_head_workspace_size(T, Q, O) bytes.
 * ------------------------------------------------------------------------------------------ */
typedef struct {
  const uint16_t* norm1;             /* [1024] */
  const uint16_t *wq, *wk, *wv, *wo; /* [1024, 1024] */
  const uint16_t* norm2;             /* [1024] */
  const uint16_t *wg, *wu;           /* [4096, 1024] */
  const uint16_t* wd;                /* [1024, 4096] */
} clef_head_layer;

typedef struct {
  const uint16_t *w_mem, *w_in, *w_lex; /* [1024, 4096] */
  const uint16_t* e_qtype;              /* [3, 1024]: noul, choice, score */
  const uint16_t *e_opt, *e_glob;       /* [1024] */
  clef_head_layer dec[4];               /* decoder layers (slots attend to the tokens) */
  clef_head_layer route[2];             /* routing layers (slots attend to each other) */
  const uint16_t* norm_f;               /* [1024] */
  const uint16_t *w_opt, *w_qst;        /* [1024, 1024] */
} clef_head;

#define CLEF_HEAD_MAX_Q 16
#define CLEF_HEAD_MAX_O 128

CLEF_API size_t clef_joint_head_workspace_size(int64_t T, int64_t Q, int64_t O);
CLEF_API clef_status clef_joint_head(const clef_head* head, const uint16_t* hidden,
                                     const uint8_t* key_valid, int64_t T, const float* q_avg,
                                     const float* o_avg, const float* g_avg, const float* lexical,
                                     const uint8_t* member, const int32_t* type_ids,
                                     const uint8_t* q_valid, const uint8_t* o_valid, int64_t Q,
                                     int64_t O, float* logits, float* probs, void* workspace,
                                     size_t workspace_bytes, clef_stream stream);

/* ------------------------------------------------------------------------------------------
 * Chunked prefill with carried state ("clef-flash - Core AI" README, section "Core AI shape": a
 * request is prefilled as successive calls of 64 positions from zeroed states, each carrying the
 * key and value caches of the attention layers and the conv and recurrent states of the Gated
 * DeltaNet layers to the next; "clef-flash-LiteRT" card, section "Other forms measured": a chunk
 * step of 128 positions carrying caches of 4,096 positions).  Any chunk length works here.  The
 * state of B requests, all device buffers owned by the caller:
 *   conv    fp16 [n_gdn][B][3][8192]      the last three rows of each GDN layer's conv input
 *                                         (the q | k | v projection), oldest first
 *   rec     fp32 [n_gdn][B][32][128][128] each GDN layer's state S (value rows x key columns)
 *   kcache  fp16 [n_attn][B][ctx][4][256] each attention layer's keys after rotary
 *   vcache  fp16 [n_attn][B][ctx][4][256] each attention layer's values
 * n_gdn / n_attn count the model's layers of each kind in order.  Layouts differ from the pages'
 * Core ML states ([.., 8192, 3] conv, fp16 rec, [.., 4, ctx, 256] caches): these are this
 * library's own.  pos = positions already in the state, the same for every request; a state of
 * zeros with pos = 0 is an empty one.
 * ------------------------------------------------------------------------------------------ */
typedef struct {
  uint16_t* conv;
  float* rec;
  uint16_t* kcache;
  uint16_t* vcache;
  int64_t ctx;   /* capacity of the caches in positions, 1..CLEF_MAX_LEN */
  int64_t pos;   /* positions already in the state */
} clef_state;

/* Bytes of workspace clef_prefill_forward_chunk needs for B requests of chunks of L positions. */
CLEF_API size_t clef_prefill_chunk_workspace_size(int64_t B, int64_t L);

/* device: positions pos .. pos + L - 1 of B requests.  ids [B, L] int32 (device) -> hidden
   [B, L, 4096] fp16 (final-norm hidden states of these positions), reading and updating the
   state; on success state->pos += L (host side, before any device work completes).  Calls with
   pos = 0, L1, L1 + L2, .. give the rows of one clef_prefill_forward of the whole request (up
   to rounding).  pos + L > ctx: CLEF_E_TOO_LONG; L < 1 or B < 1: CLEF_E_INVALID.  Calls on one
   state must not overlap on the device. */
CLEF_API clef_status clef_prefill_forward_chunk(const clef_model* model, const int32_t* ids,
                                                int64_t B, int64_t L, clef_state* state,
                                                uint16_t* hidden, void* workspace,
                                                size_t workspace_bytes, clef_stream stream);

/* device: one decoder layer on the fp32 residual stream x [B, L, 4096], updated in place:
   x <- h + mlp(rmsnorm(h)),  h = x + mixer(rmsnorm(x)).  Same workspace as the forward. */
CLEF_API clef_status clef_decoder_layer(const clef_layer* layer, float* x, int64_t B, int64_t L,
                               void* workspace, size_t workspace_bytes, clef_stream stream);

/* Wait for `stream`, then read and clear the device status word.  Returns CLEF_OK,
   CLEF_E_DEVICE_TIMEOUT, CLEF_E_BAD_TOKEN, CLEF_E_NONFINITE or CLEF_E_CUDA.  For a non-finite
   hidden row the message names the lowest such row index (b * L + t). */
CLEF_API clef_status clef_sync_status(clef_stream stream);

/* device: which rows of an fp16 array x [rows, cols] hold an inf or a NaN.  The analogue of the
   pages' rejection of FP16 overflow ("Clef-Flash-ANE-LUT6", section "Vision weights": the
   largest residual met, about 12,400, is within FP16's range, and inputs that overflow are
   rejected rather than answered).  flags [rows] (device, caller owned, may be NULL) receives 1
   for such a row and 0 otherwise; if any row is flagged, the status word reports
   CLEF_E_NONFINITE with the lowest row (clef_sync_status).  Every prefill entry point already
   checks its final-norm output this way (without the per-row flags).  cols % 8 == 0, x 16-byte
   aligned.  Asynchronous on `stream`. */
CLEF_API clef_status clef_check_finite(const uint16_t* x, int64_t rows, int64_t cols,
                                       uint8_t* flags, clef_stream stream);

/* Per-kernel-class device time.  Between clef_trace_begin() and clef_trace_end(), every kernel
   the library launches (from any thread) is bracketed by CUDA events on its own stream.
   clef_trace_end synchronises the device, then fills up to max_entries entries (one per kernel
   class: launches, summed device milliseconds, and the summed algorithmic flops and bytes of
   those launches) and writes their number to *n_entries.  Adds two event records per launch. */
typedef struct {
  char name[32];
  int64_t launches;
  double ms;
  double flops;
  double bytes;
} clef_trace_entry;
CLEF_API clef_status clef_trace_begin(void);
CLEF_API clef_status clef_trace_end(clef_trace_entry* entries, int32_t max_entries,
                                    int32_t* n_entries);

/* Host-side fault hook for tests of the error paths: the next `n_calls` device entry points fail
   with CLEF_E_CUDA before launching anything.  Affects the calling process only. */
CLEF_API void clef_debug_fail_next(int32_t n_calls);

/* Host only, no device call: the byte offsets from the workspace base at which the gated delta
   rule scan (clef_gdn_prefill, and each GDN layer of the prefill with with_norm = 1) places its
   regions for B requests of L positions, in the order g, exp(g), W, U', decayed keys, Aqk^T,
   carried state (only when the scan runs in pieces), o (only with_norm); -1 for a region not
   used.  offsets: 8 int64, caller owned; *total = the workspace bytes the scan needs.  For tests
   of the carving against the size query.  CLEF_E_INVALID for NULL outputs or B, L < 1. */
CLEF_API clef_status clef_debug_gdn_workspace_layout(int64_t B, int64_t L, int32_t with_norm,
                                                     int64_t* offsets, int64_t* total);

#ifdef __cplusplus
}
#endif
#endif /* CLEF_H_ */
