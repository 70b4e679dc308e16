// The decoder layers and the 32-layer hybrid prefill, plus the C-ABI entry points of the scan,
// the attention and the model.
//
// Layer (pre-norm residual, fp32 residual stream x, fp16 activations between kernels):
//   GDN:        xn = rmsnorm(x); proj = xn W_in^T (q|k|v|z); ab = xn W_ab^T;
//               q,k,v,g,beta = prep(proj, ab); y = zgated_norm(scan(q,k,v,g,beta), z);
//               x += y W_out^T
//   attention:  xn = rmsnorm(x); proj = xn W_in^T (query|gate|k|v); rotary(q, k);
//               y = attention(q, k, v) * sigmoid(gate); x += y W_o^T
//   MLP:        xn = rmsnorm(x); h = SiLU(xn W_gate^T) * (xn W_up^T); x += h W_down^T
// The model: x = embed[ids]; 32 layers (attention every fourth, layers 3, 7, ..); hidden =
// rmsnorm(x) in fp16 ("Clef-Flash-ANE-LUT6" model card, "Model architecture";
// "clef-flash-LiteRT" README, "Host contract" steps 4-6).
#include <algorithm>

#include "attn.cuh"
#include "common.cuh"
#include "gdn.cuh"
#include "glue.cuh"
#include "lut6.cuh"

namespace clef {

constexpr int64_t H = CLEF_HIDDEN;
constexpr int64_t I = CLEF_INTER;
constexpr int64_t GDN_PROJ = 2 * 2048 + 4096 + 4096;     // q | k | v | z
constexpr int64_t ATT_PROJ = 4096 + 4096 + 1024 + 1024;  // query | gate | k | v

static inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

struct FwdWs {
  float* x;
  __half* xn;
  __half* proj;
  __half* q;
  __half* k;
  __half* v;
  float* g;
  float* beta;
  float* abpart;
  __half* mix;
  __half* h;
  void* scan;
  float* part;     // k-part partial sums of the split residual adds (ordered reduction)
};

static size_t fwd_layout(int64_t B, int64_t L, void* base, FwdWs* w) {
  const int64_t M = B * L;
  uint8_t* p = static_cast<uint8_t*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    void* r = p ? p + off : nullptr;
    off += al256(bytes);
    return r;
  };
  FwdWs t;
  t.x = static_cast<float*>(take(M * H * 4));
  t.xn = static_cast<__half*>(take(M * H * 2));
  t.proj = static_cast<__half*>(take(M * GDN_PROJ * 2));
  t.q = static_cast<__half*>(take(M * 2048 * 2));
  t.k = static_cast<__half*>(take(M * 2048 * 2));
  t.v = static_cast<__half*>(take(M * 4096 * 2));
  t.g = static_cast<float*>(take(M * 32 * 4));
  t.beta = static_cast<float*>(take(M * 32 * 4));
  t.abpart = static_cast<float*>(take(ab_proj_scratch_bytes(M)));
  t.mix = static_cast<__half*>(take(M * H * 2));
  t.h = static_cast<__half*>(take(M * I * 2));
  t.scan = take(gdn_scan_workspace_bytes(B, L, true));
  {
    // the residual adds (out-proj K = 4096, down K = 12288, N = 4096) split over k-parts only
    // when there are few tiles; reproducible prefills keep each part's sums here
    const int64_t parts = std::max(lut6_add_split(M, H, H), lut6_add_split(M, H, I));
    t.part = parts > 1 ? static_cast<float*>(take((size_t)parts * M * H * 4)) : nullptr;
  }
  if (w) *w = t;
  return off;
}

#define CLEF_TRY(expr)                 \
  do {                                 \
    clef_status _s = (expr);           \
    if (_s != CLEF_OK) return _s;      \
  } while (0)

// Carried state of one layer for a chunk of positions pos0 .. pos0 + L - 1 (NULL pointers and
// pos0 = 0: a whole prefill from an empty state).
struct LayerState {
  __half* conv = nullptr;   // GDN: [B][3][8192]
  float* rec = nullptr;     // GDN: [B][32][128][128]
  __half* kc = nullptr;     // attention: [B][ctx][4][256]
  __half* vc = nullptr;
  int64_t ctx = 0;
  int64_t pos0 = 0;
  MRope mr;                 // picture block of every request (M-RoPE); h * w == 0: text only
};

static clef_status run_layer(const clef_layer& ly, const FwdWs& w, int64_t B, int64_t L,
                             cudaStream_t s, const LayerState& st = LayerState(),
                             bool reproducible = false) {
  const int64_t M = B * L;
  float* part = reproducible ? w.part : nullptr;
  const __half* attn_norm = reinterpret_cast<const __half*>(ly.attn_norm);
  CLEF_TRY(rmsnorm_launch(w.x, attn_norm, w.xn, M, s));
  const __half* in_lut = reinterpret_cast<const __half*>(ly.in_proj.lut);
  if (ly.kind == CLEF_LAYER_GDN) {
    CLEF_TRY(lut6_gemm_launch(w.xn, ly.in_proj.packed, in_lut, w.proj, GDN_PROJ, M, GDN_PROJ, H,
                              EPI_F16, s));
    CLEF_TRY(ab_proj_launch(w.xn, reinterpret_cast<const __half*>(ly.ab_w),
                            reinterpret_cast<const __half*>(ly.A_log),
                            reinterpret_cast<const __half*>(ly.dt_bias), w.g, w.beta, w.abpart, M,
                            s));
    CLEF_TRY(gdn_prep_launch(w.proj, GDN_PROJ, reinterpret_cast<const __half*>(ly.conv_w),
                             st.conv, w.q, w.k, w.v, M, L, s));
    if (st.conv) CLEF_TRY(conv_state_launch(w.proj, GDN_PROJ, st.conv, B, L, s));
    // the recurrent state enters from and returns to st.rec (each CTA reads its slice first)
    CLEF_TRY(gdn_scan_launch(w.q, w.k, w.v, w.g, nullptr, w.beta, st.rec, st.rec,
                             w.proj + 8192, GDN_PROJ, reinterpret_cast<const __half*>(ly.o_norm),
                             w.mix, H, B, L, w.scan, s));
  } else {
    CLEF_TRY(lut6_gemm_launch(w.xn, ly.in_proj.packed, in_lut, w.proj, ATT_PROJ, M, ATT_PROJ, H,
                              EPI_F16, s));
    __half* qp = w.proj;
    __half* gp = w.proj + 4096;
    __half* kp = w.proj + 8192;
    __half* vp = w.proj + 9216;
    if (st.kc) {
      // rotated keys and the values go into the caches at positions pos0 ..; attention reads
      // positions 0 .. pos0 + L - 1 from there
      constexpr int64_t KV = 4 * 256;
      CLEF_TRY(rope_launch(qp, ATT_PROJ, qp, ATT_PROJ, kp, ATT_PROJ, st.kc, KV, M, L, st.pos0,
                           st.ctx, s, st.mr));
      CLEF_TRY(kv_store_launch(vp, ATT_PROJ, st.vc, KV, M, L, st.pos0, st.ctx, (int)KV, s));
      CLEF_TRY(flash_launch(qp, ATT_PROJ, st.kc, KV, st.vc, KV, gp, ATT_PROJ, w.mix, H, B, L,
                            st.pos0, st.ctx, s));
    } else {
      CLEF_TRY(rope_launch(qp, ATT_PROJ, qp, ATT_PROJ, kp, ATT_PROJ, kp, ATT_PROJ, M, L, 0, L, s,
                           st.mr));
      CLEF_TRY(flash_launch(qp, ATT_PROJ, kp, ATT_PROJ, vp, ATT_PROJ, gp, ATT_PROJ, w.mix, H, B, L,
                            0, L, s));
    }
  }
  CLEF_TRY(lut6_gemm_launch(w.mix, ly.out_proj.packed,
                            reinterpret_cast<const __half*>(ly.out_proj.lut), w.x, H, M, H, H,
                            EPI_ADD_F32, s, part));
  // MLP
  CLEF_TRY(rmsnorm_launch(w.x, reinterpret_cast<const __half*>(ly.mlp_norm), w.xn, M, s));
  CLEF_TRY(lut6_gemm_launch(w.xn, ly.gate_up.packed, reinterpret_cast<const __half*>(ly.gate_up.lut),
                            w.h, I, M, 2 * I, H, EPI_SWIGLU_F16, s));
  CLEF_TRY(lut6_gemm_launch(w.h, ly.down.packed, reinterpret_cast<const __half*>(ly.down.lut), w.x,
                            H, M, H, I, EPI_ADD_F32, s, part));
  return CLEF_OK;
}

static bool bad_ptr(const void* p) {
  return p == nullptr || (reinterpret_cast<uintptr_t>(p) & 15u) != 0;
}

static clef_status check_layer(const clef_layer* ly, int idx) {
  if (!ly) {
    set_error("layer %d: NULL", idx);
    return CLEF_E_INVALID;
  }
  if (ly->kind != CLEF_LAYER_GDN && ly->kind != CLEF_LAYER_ATTENTION) {
    set_error("layer %d: bad kind %d", idx, ly->kind);
    return CLEF_E_INVALID;
  }
  const void* need[] = {ly->attn_norm, ly->mlp_norm, ly->in_proj.packed, ly->in_proj.lut,
                        ly->out_proj.packed, ly->out_proj.lut, ly->gate_up.packed, ly->gate_up.lut,
                        ly->down.packed, ly->down.lut};
  for (const void* p : need)
    if (bad_ptr(p)) {
      set_error("layer %d: a weight pointer is NULL or not 16-byte aligned", idx);
      return p ? CLEF_E_ALIGN : CLEF_E_INVALID;
    }
  if (ly->kind == CLEF_LAYER_GDN) {
    const void* g[] = {ly->ab_w, ly->A_log, ly->dt_bias, ly->conv_w, ly->o_norm};
    for (const void* p : g)
      if (bad_ptr(p)) {
        set_error("layer %d: a GDN weight pointer is NULL or not 16-byte aligned", idx);
        return p ? CLEF_E_ALIGN : CLEF_E_INVALID;
      }
  }
  return CLEF_OK;
}

static clef_status check_bl(int64_t B, int64_t L) { return check_batch_len(B, L); }

// The whole prefill of B requests (ids [B][L]); with image_rows, rows mr.start .. of every
// request are the picture's rows ([B][h * w][4096] fp16) and the rotary uses M-RoPE planes.
static clef_status prefill_impl(const char* who, const clef_model* model, const int32_t* ids,
                                int64_t B, int64_t L, const __half* image_rows, const MRope& mr,
                                uint16_t* hidden, void* workspace, size_t workspace_bytes,
                                clef_stream stream) {
  CLEF_TRY(check_bl(B, L));
  if (!model || !model->layers || model->n_layers < 1 || model->n_layers > 64 ||
      model->vocab < 1) {
    set_error("%s: bad model (layers, n_layers in 1..64, vocab >= 1)", who);
    return CLEF_E_INVALID;
  }
  if (bad_ptr(ids) || bad_ptr(hidden) || bad_ptr(workspace) || bad_ptr(model->embed) ||
      bad_ptr(model->final_norm)) {
    set_error("%s: a pointer is NULL or not 16-byte aligned", who);
    return CLEF_E_INVALID;
  }
  for (int i = 0; i < model->n_layers; ++i) CLEF_TRY(check_layer(&model->layers[i], i));
  if (workspace_bytes < fwd_layout(B, L, nullptr, nullptr)) {
    set_error("%s: workspace of %zu bytes, need %zu", who, workspace_bytes,
              fwd_layout(B, L, nullptr, nullptr));
    return CLEF_E_WORKSPACE;
  }
  if (debug_should_fail()) return CLEF_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  FwdWs w;
  fwd_layout(B, L, workspace, &w);
  const int64_t M = B * L;
  CLEF_TRY(embed_launch(ids, reinterpret_cast<const __half*>(model->embed), model->vocab, w.x, M, s));
  if (image_rows) CLEF_TRY(image_rows_launch(image_rows, w.x, B, L, mr.start, mr.h * mr.w, s));
  LayerState ls;
  ls.mr = mr;
  const bool repro = (model->flags & CLEF_MODEL_REPRODUCIBLE) != 0;
  for (int i = 0; i < model->n_layers; ++i)
    CLEF_TRY(run_layer(model->layers[i], w, B, L, s, ls, repro));
  return rmsnorm_launch(w.x, reinterpret_cast<const __half*>(model->final_norm),
                        reinterpret_cast<__half*>(hidden), M, s, /*check_finite=*/true);
}

}  // namespace clef

using namespace clef;

extern "C" {

size_t clef_gdn_workspace_size(int64_t B, int64_t L) {
  if (B < 1 || L < 1) return 0;
  return gdn_scan_workspace_bytes(B, L, false);
}

clef_status clef_gdn_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                             const float* alpha, const float* beta, const float* s0, uint16_t* o,
                             float* s_out, int64_t B, int64_t L, void* workspace,
                             size_t workspace_bytes, clef_stream stream) {
  CLEF_TRY(check_bl(B, L));
  const void* need[] = {q, k, v, alpha, beta, o, workspace};
  for (const void* p : need)
    if (bad_ptr(p)) {
      set_error("clef_gdn_prefill: a pointer is NULL or not 16-byte aligned");
      return p ? CLEF_E_ALIGN : CLEF_E_INVALID;
    }
  if ((s0 && bad_ptr(s0)) || (s_out && bad_ptr(s_out))) {
    set_error("clef_gdn_prefill: s0 / s_out not 16-byte aligned");
    return CLEF_E_ALIGN;
  }
  if (workspace_bytes < gdn_scan_workspace_bytes(B, L, false)) {
    set_error("clef_gdn_prefill: workspace of %zu bytes, need %zu", workspace_bytes,
              gdn_scan_workspace_bytes(B, L, false));
    return CLEF_E_WORKSPACE;
  }
  if (debug_should_fail()) return CLEF_E_CUDA;
  return gdn_scan_launch(reinterpret_cast<const __half*>(q), reinterpret_cast<const __half*>(k),
                         reinterpret_cast<const __half*>(v), nullptr, alpha, beta, s0, s_out,
                         nullptr, 0, nullptr, reinterpret_cast<__half*>(o), 32 * 128, B, L,
                         workspace, static_cast<cudaStream_t>(stream));
}

size_t clef_attn_workspace_size(int64_t B, int64_t L) {
  if (B < 1 || L < 1) return 0;
  return al256((size_t)B * L * 16 * 256 * 2) + al256((size_t)B * L * 4 * 256 * 2);
}

clef_status clef_gqa_attn_prefill(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                  const uint16_t* gate, uint16_t* o, int64_t B, int64_t L,
                                  int64_t row_stride_q, int64_t row_stride_kv,
                                  int64_t row_stride_gate, void* workspace, size_t workspace_bytes,
                                  clef_stream stream) {
  CLEF_TRY(check_bl(B, L));
  const void* need[] = {q, k, v, o, workspace};
  for (const void* p : need)
    if (bad_ptr(p)) {
      set_error("clef_gqa_attn_prefill: a pointer is NULL or not 16-byte aligned");
      return p ? CLEF_E_ALIGN : CLEF_E_INVALID;
    }
  if (gate && bad_ptr(gate)) {
    set_error("clef_gqa_attn_prefill: gate not 16-byte aligned");
    return CLEF_E_ALIGN;
  }
  const int64_t ldq = row_stride_q ? row_stride_q : 16 * 256;
  const int64_t ldkv = row_stride_kv ? row_stride_kv : 4 * 256;
  const int64_t ldg = row_stride_gate ? row_stride_gate : 16 * 256;
  if (ldq < 16 * 256 || ldkv < 4 * 256 || ldg < 16 * 256 || ldq % 8 || ldkv % 8 || ldg % 8) {
    set_error("clef_gqa_attn_prefill: row strides must cover a row and be multiples of 8");
    return CLEF_E_SHAPE;
  }
  if (workspace_bytes < clef_attn_workspace_size(B, L)) {
    set_error("clef_gqa_attn_prefill: workspace of %zu bytes, need %zu", workspace_bytes,
              clef_attn_workspace_size(B, L));
    return CLEF_E_WORKSPACE;
  }
  if (debug_should_fail()) return CLEF_E_CUDA;
  const int64_t M = B * L;
  __half* qr = static_cast<__half*>(workspace);
  __half* kr = reinterpret_cast<__half*>(static_cast<uint8_t*>(workspace) + al256((size_t)M * 16 * 256 * 2));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  CLEF_TRY(rope_launch(reinterpret_cast<const __half*>(q), ldq, qr, 16 * 256,
                       reinterpret_cast<const __half*>(k), ldkv, kr, 4 * 256, M, L, 0, L, s));
  return flash_launch(qr, 16 * 256, kr, 4 * 256, reinterpret_cast<const __half*>(v), ldkv,
                      reinterpret_cast<const __half*>(gate), ldg, reinterpret_cast<__half*>(o),
                      16 * 256, B, L, 0, L, s);
}

size_t clef_prefill_workspace_size(int64_t B, int64_t L) {
  if (B < 1 || L < 1) return 0;
  return fwd_layout(B, L, nullptr, nullptr);
}

clef_status clef_decoder_layer(const clef_layer* layer, float* x, int64_t B, int64_t L,
                               void* workspace, size_t workspace_bytes, clef_stream stream) {
  CLEF_TRY(check_bl(B, L));
  CLEF_TRY(check_layer(layer, 0));
  if (bad_ptr(x) || bad_ptr(workspace)) {
    set_error("clef_decoder_layer: x / workspace NULL or not 16-byte aligned");
    return CLEF_E_INVALID;
  }
  if (workspace_bytes < fwd_layout(B, L, nullptr, nullptr)) {
    set_error("clef_decoder_layer: workspace of %zu bytes, need %zu", workspace_bytes,
              fwd_layout(B, L, nullptr, nullptr));
    return CLEF_E_WORKSPACE;
  }
  if (debug_should_fail()) return CLEF_E_CUDA;
  FwdWs w;
  fwd_layout(B, L, workspace, &w);
  w.x = x;  // the layer works on the caller's residual stream in place
  return run_layer(*layer, w, B, L, static_cast<cudaStream_t>(stream));
}

clef_status clef_prefill_forward(const clef_model* model, const int32_t* ids, int64_t B, int64_t L,
                                 uint16_t* hidden, void* workspace, size_t workspace_bytes,
                                 clef_stream stream) {
  return prefill_impl("clef_prefill_forward", model, ids, B, L, nullptr, MRope(), hidden,
                      workspace, workspace_bytes, stream);
}

clef_status clef_prefill_forward_image(const clef_model* model, const int32_t* ids, int64_t B,
                                       int64_t L, const uint16_t* image_rows, int64_t image_start,
                                       int64_t grid_h, int64_t grid_w, uint16_t* hidden,
                                       void* workspace, size_t workspace_bytes,
                                       clef_stream stream) {
  if (grid_h < 0 || grid_w < 0 || (grid_h == 0) != (grid_w == 0) || image_start < 0) {
    set_error("clef_prefill_forward_image: need grid_h, grid_w both 0 or both >= 1 and "
              "image_start >= 0");
    return CLEF_E_INVALID;
  }
  const int64_t n = grid_h * grid_w;
  if (n > 0 && (image_start + n > L)) {
    set_error("clef_prefill_forward_image: the picture's %lld tokens from index %lld do not fit "
              "in L = %lld", (long long)n, (long long)image_start, (long long)L);
    return CLEF_E_SHAPE;
  }
  if (n > 0 && bad_ptr(image_rows)) {
    set_error("clef_prefill_forward_image: image_rows NULL or not 16-byte aligned");
    return CLEF_E_INVALID;
  }
  MRope mr;
  mr.start = n > 0 ? image_start : 0;
  mr.h = grid_h;
  mr.w = grid_w;
  return prefill_impl("clef_prefill_forward_image", model, ids, B, L,
                      n > 0 ? reinterpret_cast<const __half*>(image_rows) : nullptr, mr, hidden,
                      workspace, workspace_bytes, stream);
}

clef_status clef_mrope_positions(int64_t L, int64_t image_start, int64_t grid_h, int64_t grid_w,
                                 int32_t* pos3) {
  if (!pos3 || L < 0 || grid_h < 0 || grid_w < 0 || (grid_h == 0) != (grid_w == 0) ||
      image_start < 0) {
    set_error("clef_mrope_positions: NULL output or bad sizes");
    return CLEF_E_INVALID;
  }
  const int64_t n = grid_h * grid_w;
  if (n > 0 && image_start + n > L) {
    set_error("clef_mrope_positions: the picture does not fit in L");
    return CLEF_E_SHAPE;
  }
  for (int64_t i = 0; i < L; ++i) {
    int64_t p[3] = {i, i, i};
    if (n > 0 && i >= image_start) {
      if (i < image_start + n) {
        const int64_t k = i - image_start;
        p[0] = image_start;
        p[1] = image_start + k / grid_w;
        p[2] = image_start + k % grid_w;
      } else {
        p[0] = p[1] = p[2] = i - (n - std::max(grid_h, grid_w));
      }
    }
    for (int c = 0; c < 3; ++c) pos3[3 * i + c] = (int32_t)p[c];
  }
  return CLEF_OK;
}

size_t clef_prefill_chunk_workspace_size(int64_t B, int64_t L) {
  return clef_prefill_workspace_size(B, L);
}

clef_status clef_prefill_forward_chunk(const clef_model* model, const int32_t* ids, int64_t B,
                                       int64_t L, clef_state* state, uint16_t* hidden,
                                       void* workspace, size_t workspace_bytes,
                                       clef_stream stream) {
  CLEF_TRY(check_bl(B, L));
  if (!model || !model->layers || model->n_layers < 1 || model->n_layers > 64 ||
      model->vocab < 1 || !state) {
    set_error("clef_prefill_forward_chunk: bad model (layers, n_layers in 1..64, vocab >= 1) or "
              "NULL state");
    return CLEF_E_INVALID;
  }
  if (bad_ptr(ids) || bad_ptr(hidden) || bad_ptr(workspace) || bad_ptr(model->embed) ||
      bad_ptr(model->final_norm)) {
    set_error("clef_prefill_forward_chunk: a pointer is NULL or not 16-byte aligned");
    return CLEF_E_INVALID;
  }
  int n_gdn = 0, n_attn = 0;
  for (int i = 0; i < model->n_layers; ++i) {
    CLEF_TRY(check_layer(&model->layers[i], i));
    (model->layers[i].kind == CLEF_LAYER_GDN ? n_gdn : n_attn) += 1;
  }
  if (state->ctx < 1 || state->ctx > CLEF_MAX_LEN || state->pos < 0) {
    set_error("clef_prefill_forward_chunk: state ctx must be in 1..%d and pos >= 0", CLEF_MAX_LEN);
    return CLEF_E_INVALID;
  }
  if (state->pos + L > state->ctx) {
    set_error("clef_prefill_forward_chunk: pos %lld + L %lld is above the state's %lld positions "
              "(refused, never cut)", (long long)state->pos, (long long)L, (long long)state->ctx);
    return CLEF_E_TOO_LONG;
  }
  if ((n_gdn && (bad_ptr(state->conv) || bad_ptr(state->rec))) ||
      (n_attn && (bad_ptr(state->kcache) || bad_ptr(state->vcache)))) {
    set_error("clef_prefill_forward_chunk: a state buffer is NULL or not 16-byte aligned");
    return CLEF_E_INVALID;
  }
  if (workspace_bytes < fwd_layout(B, L, nullptr, nullptr)) {
    set_error("clef_prefill_forward_chunk: workspace of %zu bytes, need %zu", workspace_bytes,
              fwd_layout(B, L, nullptr, nullptr));
    return CLEF_E_WORKSPACE;
  }
  if (debug_should_fail()) return CLEF_E_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  FwdWs w;
  fwd_layout(B, L, workspace, &w);
  const int64_t M = B * L;
  CLEF_TRY(embed_launch(ids, reinterpret_cast<const __half*>(model->embed), model->vocab, w.x, M, s));
  int gi = 0, ai = 0;
  for (int i = 0; i < model->n_layers; ++i) {
    LayerState ls;
    ls.ctx = state->ctx;
    ls.pos0 = state->pos;
    if (model->layers[i].kind == CLEF_LAYER_GDN) {
      ls.conv = reinterpret_cast<__half*>(state->conv) + (size_t)gi * B * 3 * 8192;
      ls.rec = state->rec + (size_t)gi * B * 32 * 128 * 128;
      ++gi;
    } else {
      const size_t per_layer = (size_t)B * state->ctx * 4 * 256;
      ls.kc = reinterpret_cast<__half*>(state->kcache) + (size_t)ai * per_layer;
      ls.vc = reinterpret_cast<__half*>(state->vcache) + (size_t)ai * per_layer;
      ++ai;
    }
    CLEF_TRY(run_layer(model->layers[i], w, B, L, s, ls,
                       (model->flags & CLEF_MODEL_REPRODUCIBLE) != 0));
  }
  CLEF_TRY(rmsnorm_launch(w.x, reinterpret_cast<const __half*>(model->final_norm),
                          reinterpret_cast<__half*>(hidden), M, s, /*check_finite=*/true));
  state->pos += L;
  return CLEF_OK;
}

}  // extern "C"
