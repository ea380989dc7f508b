// libhe: engine state, workspace, and the launch sequence of one generation.
//
// Host C++ only (kernels live in gemm_tc.cu, gemm_simt.cu, attn.cu, rows.cu).
// The engine records the caller's weight pointers (one model instance), owns a
// workspace taken through the caller's allocator (KV cache + activations), and
// enqueues every step of generation on the caller's stream.  No host
// synchronisation happens inside he_generate: the token chosen at step k is
// embedded on the device by the head kernel for step k + 1.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/he.h"
#include "../../include/he_ops.h"
#include "kernels.h"

using namespace he;

namespace {

thread_local std::string g_err;

he_status fail(he_status s, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

void *default_alloc(size_t bytes, void *, void *) {
  void *p = nullptr;
  return cudaMalloc(&p, bytes) == cudaSuccess ? p : nullptr;
}
void default_free(void *p, size_t, void *, void *) { cudaFree(p); }

struct Buf {
  void *p = nullptr;
  size_t bytes = 0;
};

constexpr int kMaxGemmSplit = 16;
constexpr int kMaxAttnSplit = 32;
constexpr int kClasses = 8;

}  // namespace

namespace he {
bool g_pdl = true;

// Sets the calling thread's he_last_error message (used by entry points in other files).
he_status set_error(he_status s, const char *msg) {
  g_err = msg ? msg : "";
  return s;
}
}  // namespace he

struct he_engine {
  he_config cfg{};
  int device = 0, num_sms = 0;
  size_t elem = 4;
  const void *tok_emb = nullptr, *pos_emb = nullptr, *lnf_g = nullptr, *lnf_b = nullptr;
  std::vector<he_layer_weights> layers;
  // BF16 while fused: the merged fp16 projections in the tiled layout, one per
  // (layer, projection), inside `restore`; generation reads these instead of w[]
  std::vector<const void *> fused_w;
  // he_set_weight_format: HE_WEIGHTS_FP8 keeps E4M3 codes and row scales next to
  // fused_w (which then holds the same codes as fp16 values, for the prefill GEMMs)
  int wfmt = HE_WEIGHTS_F16;
  std::vector<const void *> fused_w8;
  std::vector<const float *> fused_scale;
  he_allocator alloc{};

  bool taken = false, fused = false;
  bool tiled = false;  // projections hold the tiled layout (bf16 path while fused)
  int act = 0;         // activation type of the generation in flight (ActType)
  unsigned prof_mask = 0;
  // workspace (released / retaken together)
  Buf kc, vc, x, h, q, ctx, mid, partial, logits, attn_part, ids_in, ids_out, lp_out, logmap;
  // held for the engine's lifetime
  Buf err;
  Buf tilecnt;  // per-tile arrival counters of the stream-K fix-up (zero between GEMMs)
  Buf attncnt;  // per-(sequence, head) counters of the decode attention's slice merge
  // LoRA restore copy (held while fused)
  Buf restore;
  // BF16 without LoRA fused: the caller's projections as fp16 in the tiled layout,
  // rewritten at the start of every generation (taken with the workspace)
  Buf base;

  he_stats stats{};
  cudaEvent_t ph[7] = {};  // generate begin/prefill end/end, fuse begin/end, unfuse begin/end
  // sampling (he_set_sampling): temperature 0 = greedy
  float temperature = 0.f, top_p = 1.f;
  unsigned long long seed = 0;
  // CUDA-graph generation (he_set_cuda_graph): one captured generation per shape and
  // buffer set, replayed on the caller's stream
  bool graph_on = false, capturing = false;
  cudaStream_t cap_stream = nullptr;
  cudaGraphExec_t gexec = nullptr;
  std::vector<const void *> gkey;  // shape, activation type and every buffer address
  unsigned long long glaunches = 0;  // kernel launches in the captured generation
  struct Pair { cudaEvent_t a, b; };
  std::vector<Pair> prof_pool[kClasses];
  size_t prof_used[kClasses] = {};
  bool stats_pending = false, fuse_pending = false, unfuse_pending = false;

  size_t kv_layer_elems() const {
    return (size_t)cfg.max_batch * cfg.n_heads * cfg.max_seq * (cfg.d_model / cfg.n_heads);
  }
};

namespace {

he_status cuda_fail(cudaError_t e, const char *what) {
  return fail(HE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool get(he_engine *h, Buf &b, size_t bytes, cudaStream_t st) {
  b.bytes = bytes;
  b.p = bytes ? h->alloc.alloc(bytes, st, h->alloc.ctx) : nullptr;
  if (bytes && !b.p) {
    b.bytes = 0;
    return false;
  }
  return true;
}

void put(he_engine *h, Buf &b, cudaStream_t st) {
  if (b.p) h->alloc.free(b.p, b.bytes, st, h->alloc.ctx);
  b.p = nullptr;
  b.bytes = 0;
}

// Stream-K tile counters: one int per 128-row tile of the widest projection.
size_t tilecnt_bytes(const he_config &c) {
  size_t wide = (size_t)(3 * c.d_model > c.ffn ? 3 * c.d_model : c.ffn);
  if ((size_t)c.vocab > wide) wide = c.vocab;
  return (wide + 127) / 128 * sizeof(int);
}

// Attention slice-merge counters: one int per (sequence, head) pair.
size_t attncnt_bytes(const he_config &c) { return (size_t)c.max_batch * c.n_heads * sizeof(int); }

void free_workspace(he_engine *h, cudaStream_t st) {
  Buf *all[] = {&h->kc, &h->vc, &h->x, &h->h, &h->q, &h->ctx, &h->mid, &h->partial,
                &h->logits, &h->attn_part, &h->ids_in, &h->ids_out, &h->lp_out, &h->logmap,
                &h->base};
  for (Buf *b : all) put(h, *b, st);
  if (!h->fused) {
    h->fused_w.clear();
    h->fused_w8.clear();
    h->fused_scale.clear();
    h->tiled = false;
  }
  h->taken = false;
  h->stats.workspace_bytes = 0;
  h->stats.kv_bytes = 0;
}

he_status take_workspace(he_engine *h, cudaStream_t st) {
  const he_config &c = h->cfg;
  const size_t e = h->elem, hd = c.d_model / c.n_heads;
  size_t max_tok = (size_t)c.max_batch * c.max_seq;
  // decode buffers hold a padded token tile when they are row-tiled
  if (c.dtype == HE_DTYPE_BF16 && (size_t)sk_token_tile(c.max_batch) > max_tok)
    max_tok = sk_token_tile(c.max_batch);
  const size_t kv = (size_t)c.n_layers * h->kv_layer_elems() * e;
  size_t wide = (size_t)(3 * c.d_model > c.ffn ? 3 * c.d_model : c.ffn);
  if ((size_t)c.vocab > wide) wide = c.vocab;  // LM-head slices
  wide = (wide + 127) / 128 * 128;             // tile-contiguous slices: whole 128-wide tiles
  size_t part = max_tok * c.d_model;
  if ((size_t)kMaxGemmSplit * c.max_batch * wide > part) part = (size_t)kMaxGemmSplit * c.max_batch * wide;
  struct {
    Buf *b;
    size_t bytes;
  } want[] = {
      {&h->kc, kv},
      {&h->vc, kv},
      {&h->x, max_tok * c.d_model * 4},
      {&h->h, max_tok * c.d_model * e},
      {&h->q, max_tok * c.d_model * e},
      {&h->ctx, max_tok * c.d_model * e},
      {&h->mid, max_tok * c.ffn * e},
      {&h->partial, part * 4},
      {&h->logits, (size_t)c.max_batch * c.vocab * 4},
      {&h->attn_part, (size_t)c.max_batch * c.n_heads * kMaxAttnSplit * (hd + 2) * 4},
      {&h->ids_in, max_tok * 4},
      {&h->ids_out, max_tok * 4},
      {&h->lp_out, max_tok * 4},
      {&h->logmap, max_tok * 4},
  };
  size_t total = 0;
  for (auto &w : want) {
    if (!get(h, *w.b, w.bytes, st)) {
      free_workspace(h, st);
      return fail(HE_ERR_OOM, "workspace allocation of %zu bytes failed", w.bytes);
    }
    total += w.bytes;
  }
  h->taken = true;
  h->stats.workspace_bytes = total;
  h->stats.kv_bytes = 2 * kv;
  return HE_OK;
}

// ---- profiling helpers -----------------------------------------------------
struct Timed {
  he_engine *h;
  int cls;
  cudaStream_t st;
  he_engine::Pair *p = nullptr;
  Timed(he_engine *h_, int c, cudaStream_t s) : h(h_), cls(c), st(s) {
    if (!((h->prof_mask >> cls) & 1u)) return;
    auto &pool = h->prof_pool[cls];
    if (h->prof_used[cls] == pool.size()) {
      he_engine::Pair np{};
      cudaEventCreate(&np.a);
      cudaEventCreate(&np.b);
      pool.push_back(np);
    }
    p = &pool[h->prof_used[cls]++];
    cudaEventRecord(p->a, st);
  }
  ~Timed() {
    if (p) cudaEventRecord(p->b, st);
  }
};

void ensure_phase_events(he_engine *h) {
  if (!h->ph[0])
    for (auto &e : h->ph) cudaEventCreate(&e);
}

// ---- the generation sequence -------------------------------------------------
struct Ctx {
  he_engine *h;
  cudaStream_t st;
  cudaError_t e = cudaSuccess;
  void check(cudaError_t r, int launches) {
    if (e == cudaSuccess && r != cudaSuccess) e = r;
    h->stats.launches += launches;
  }
};

inline char *at(void *p, size_t off) { return static_cast<char *>(p) + off; }

// Decode projections on bf16 run the persistent stream-K kernel when the shape
// allows (whole 128 x 64 tiles, one token tile).
bool use_stream_k(const he_engine *h, int M, int N, int K, bool decode, bool tiled_w) {
  return decode && h->cfg.dtype == HE_DTYPE_BF16 && M <= 256 && K % 64 == 0 &&
         (!tiled_w || N % 128 == 0);
}

// Rows of the row-tiled decode activation buffers (0 = row-major).
int act_rows(const he_engine *h, int B, bool decode) {
  return decode && h->cfg.dtype == HE_DTYPE_BF16 ? sk_token_tile(B) : 0;
}

// One projection GEMM.  Element-wise epilogues (QKV, ReLU, logits) are completed
// here (stream-K: inside the GEMM by the last run of each tile; split-K: slices
// reduced by a second kernel); for EPI_PARTIAL the
// fp32 slices stay in h->partial and the returned SliceInfo tells the row
// consumer how to add them.
// With fp8 weights (w8 and scales per row group, w the same codes as fp16 values):
// the decode projections stream the fp8 codes through the stream-K kernel when it
// takes them (at most 128 tokens, K % 256 == 0); every other GEMM reads the fp16
// codes and applies the row scales in its epilogue.
SliceInfo gemm(Ctx &c, int cls, const void *x, int ldx, const void *const *w, int n_groups,
               int group_rows, int M, int K, Epi epi, bool decode, bool tiled_w, int act,
               const void *const *w8 = nullptr, const float *const *scales = nullptr) {
  he_engine *h = c.h;
  GemmArgs a{};
  a.dtype = h->cfg.dtype;
  a.act = act;
  a.x = x;
  a.ldx = ldx;
  for (int g = 0; g < n_groups; ++g) a.w[g] = w[g];
  if (scales)
    for (int g = 0; g < n_groups; ++g) a.w_scale[g] = scales[g];
  a.n_groups = n_groups;
  a.group_rows = group_rows;
  a.M = M;
  a.N = n_groups * group_rows;
  a.K = K;
  a.w_tiled = tiled_w;
  SliceInfo si{1, 0, 0, 0};
  float *part = static_cast<float *>(h->partial.p);
  long long stride = (long long)M * a.N;
  Timed t(h, cls, c.st);
  const bool fp8_sk = w8 && scales && M <= 128 && K % 256 == 0 && act == ACT_F16;
  if (use_stream_k(h, M, a.N, K, decode, tiled_w) && (!scales || fp8_sk)) {
    if (fp8_sk) {
      a.w_fp8 = 1;
      for (int g = 0; g < n_groups; ++g) a.w[g] = w8[g];
    }
    a.split = 1;
    a.epi = epi;
    // the projections' element-wise epilogues (QKV, fc1) take the stream-K +
    // data-parallel split when every run has a whole tile
    a.sk_hybrid = epi.kind == EPI_QKV || epi.kind == EPI_RELU;
    // element-wise epilogues finish inside the kernel (last run of each tile)
    const bool fix = sk_fixup_ok(a);
    const int P = sk_ctas(a, h->num_sms, fix);
    const long long U = sk_units(a), T = (a.N + 127) / 128;
    if (fix) stride = (long long)M * T * 128;  // tile-contiguous slices
    si = SliceInfo{0, U, (int)(U / T), P};
    c.check(launch_gemm_sk(a, P, part, stride, fix ? static_cast<int *>(h->tilecnt.p) : nullptr,
                           static_cast<int *>(h->err.p), c.st),
            1);
    // P == tiles: every tile is one run and was stored by the GEMM itself
    if (epi.kind != EPI_PARTIAL && !fix && P != T)
      c.check(launch_sk_reduce_epi(a.dtype, a.act, part, si, stride, a.N, M, a.N, epi, c.st), 1);
    return si;
  }
  int split = decode ? gemm_pick_split(a, h->num_sms) : 1;
  if (split > kMaxGemmSplit) split = kMaxGemmSplit;
  split = effective_split(K, split);
  a.split = split;
  si.split = split;
  if (epi.kind == EPI_PARTIAL || split > 1) {
    Epi pe = epi;
    pe.kind = EPI_PARTIAL;
    pe.partial = part;
    pe.ldp = a.N;
    pe.split_stride = stride;
    a.epi = pe;
  } else {
    a.epi = epi;
  }
  c.check(launch_gemm(a, static_cast<int *>(h->err.p), c.st), 1);
  if (epi.kind != EPI_PARTIAL && split > 1)
    c.check(launch_reduce_epi(a.dtype, a.act, part, split, stride, a.N, M, a.N, epi, c.st), 1);
  return si;
}

Epi qkv_epi(he_engine *h, int layer, int tok_per_seq, int pos0) {
  const he_config &c = h->cfg;
  const he_layer_weights &lw = h->layers[layer];
  Epi e{};
  e.kind = EPI_QKV;
  e.bias[0] = lw.b[HE_PROJ_Q];
  e.bias[1] = lw.b[HE_PROJ_K];
  e.bias[2] = lw.b[HE_PROJ_V];
  e.out = h->q.p;
  e.ldo = c.d_model;
  const size_t lay = (size_t)layer * h->kv_layer_elems() * h->elem;
  e.kc = at(h->kc.p, lay);
  e.vc = at(h->vc.p, lay);
  e.d_model = c.d_model;
  e.n_heads = c.n_heads;
  e.head_dim = c.d_model / c.n_heads;
  e.max_seq = c.max_seq;
  e.tok_per_seq = tok_per_seq;
  e.pos0 = pos0;
  e.q_scale = 1.0f / sqrtf((float)e.head_dim);
  return e;
}

// One decoder layer over M tokens (prefill: M = B*Lp, tok_per_seq = Lp, pos0 = 0;
// decode: M = B, tok_per_seq = 1, pos0 = t).  Input h = LN1(x); output h = LN1 of
// the next layer (or the final LN after the last layer).
void layer_forward(Ctx &c, int l, int B, int M, int tok_per_seq, int pos0, bool prefill) {
  he_engine *h = c.h;
  const he_config &cf = h->cfg;
  const he_layer_weights &lw = h->layers[l];
  const int d = cf.d_model, hd = d / cf.n_heads;
  const int cls_g = prefill ? HE_KCLASS_PREFILL_GEMM : HE_KCLASS_GEMM;
  const bool dec = !prefill;
  const int R = act_rows(h, B, dec);  // decode: h, ctx, mid are row-tiled with R rows
  const bool tw = h->tiled;
  const int act = h->act;
  // the last layer's final LayerNorm feeds the LM head, whose weight is the caller's
  // embedding table: that output is written in the parameter type
  const int out_act = l == cf.n_layers - 1 ? cf.dtype : act;
  // LN1 + QKV (+ KV append at the tokens' positions)
  // projections as generation reads them: the fused copies while fused on BF16
  auto W = [&](int p) { return tw ? h->fused_w[(size_t)l * HE_N_PROJ + p] : lw.w[p]; };
  // fp8 weights: codes and row scales next to the fp16 codes
  const bool f8 = tw && h->wfmt == HE_WEIGHTS_FP8;
  auto W8 = [&](int p) { return f8 ? h->fused_w8[(size_t)l * HE_N_PROJ + p] : nullptr; };
  auto SC = [&](int p) { return f8 ? h->fused_scale[(size_t)l * HE_N_PROJ + p] : nullptr; };
  const void *wqkv[3] = {W(HE_PROJ_Q), W(HE_PROJ_K), W(HE_PROJ_V)};
  const void *w8qkv[3] = {W8(HE_PROJ_Q), W8(HE_PROJ_K), W8(HE_PROJ_V)};
  const float *sqkv[3] = {SC(HE_PROJ_Q), SC(HE_PROJ_K), SC(HE_PROJ_V)};
  gemm(c, cls_g, h->h.p, d, wqkv, 3, d, M, d, qkv_epi(h, l, tok_per_seq, pos0), dec, tw, act,
       f8 ? w8qkv : nullptr, f8 ? sqkv : nullptr);
  Epi ep{};
  ep.kind = EPI_PARTIAL;
  // attention
  const size_t lay = (size_t)l * h->kv_layer_elems() * h->elem;
  if (prefill) {
    Timed t(h, HE_KCLASS_PREFILL_ATTN, c.st);
    c.check(launch_attn_prefill(act, h->q.p, at(h->kc.p, lay), at(h->vc.p, lay), h->ctx.p, B,
                                tok_per_seq, cf.n_heads, hd, cf.max_seq,
                                static_cast<int *>(h->err.p), c.st),
            1);
  } else {
    const int n_keys = pos0 + 1;
    // few (b, h) pairs: several key slices each, merged in-kernel by the last to finish
    int split = attn_decode_pick_split(B, cf.n_heads, n_keys, h->num_sms);
    if (split > kMaxAttnSplit) split = kMaxAttnSplit;
    Timed t(h, HE_KCLASS_ATTN_DECODE, c.st);
    c.check(launch_attn_decode(act, h->q.p, at(h->kc.p, lay), at(h->vc.p, lay), h->ctx.p, R,
                               B, cf.n_heads, hd, cf.max_seq, n_keys, split,
                               static_cast<float *>(h->attn_part.p), c.st,
                               static_cast<int *>(h->attncnt.p)),
            1);
  }
  // out projection -> partials; + bo + residual; LN2
  const void *wo[1] = {W(HE_PROJ_O)};
  const void *w8o[1] = {W8(HE_PROJ_O)};
  const float *so[1] = {SC(HE_PROJ_O)};
  SliceInfo si = gemm(c, cls_g, h->ctx.p, d, wo, 1, d, M, d, ep, dec, tw, act,
                      f8 ? w8o : nullptr, f8 ? so : nullptr);
  {
    Timed t(h, HE_KCLASS_NORM, c.st);
    c.check(launch_resid_ln(cf.dtype, act, static_cast<float *>(h->partial.p), si, (long long)M * d, d,
                            lw.b[HE_PROJ_O], static_cast<float *>(h->x.p), lw.ln2_g, lw.ln2_b,
                            cf.ln_eps, h->h.p, R, M, d, c.st, static_cast<int *>(h->err.p)),
            1);
  }
  // fc1 + b1 + ReLU
  Epi er{};
  er.kind = EPI_RELU;
  er.bias[0] = lw.b[HE_PROJ_FC1];
  er.out = h->mid.p;
  er.ldo = cf.ffn;
  er.out_rows = R;
  const void *w1[1] = {W(HE_PROJ_FC1)};
  const void *w81[1] = {W8(HE_PROJ_FC1)};
  const float *s1[1] = {SC(HE_PROJ_FC1)};
  gemm(c, cls_g, h->h.p, d, w1, 1, cf.ffn, M, d, er, dec, tw, act, f8 ? w81 : nullptr,
       f8 ? s1 : nullptr);
  // fc2 -> partials; + b2 + residual; next LN
  const void *w2[1] = {W(HE_PROJ_FC2)};
  const void *w82[1] = {W8(HE_PROJ_FC2)};
  const float *s2[1] = {SC(HE_PROJ_FC2)};
  si = gemm(c, cls_g, h->mid.p, cf.ffn, w2, 1, d, M, cf.ffn, ep, dec, tw, act, f8 ? w82 : nullptr,
            f8 ? s2 : nullptr);
  const bool last = l == cf.n_layers - 1;
  const void *g = last ? h->lnf_g : h->layers[l + 1].ln1_g;
  const void *bb = last ? h->lnf_b : h->layers[l + 1].ln1_b;
  Timed t(h, HE_KCLASS_NORM, c.st);
  c.check(launch_resid_ln(cf.dtype, out_act, static_cast<float *>(h->partial.p), si, (long long)M * d, d,
                          lw.b[HE_PROJ_FC2], static_cast<float *>(h->x.p), g, bb, cf.ln_eps,
                          h->h.p, R, M, d, c.st, static_cast<int *>(h->err.p)),
          1);
}

// Logits [B][vocab] (fp32, h->logits) of B row-major rows of the last LayerNorm's
// output (row stride ldh, the parameter type) against the tied embedding table.
void head_rows_gemm(Ctx &c, const void *hrows, int ldh, int B) {
  he_engine *h = c.h;
  const he_config &cf = h->cfg;
  Timed t(h, HE_KCLASS_HEAD, c.st);
  Epi el{};
  el.kind = EPI_STORE_F32;
  el.partial = static_cast<float *>(h->logits.p);
  el.ldp = cf.vocab;
  GemmArgs a{};
  a.dtype = cf.dtype;
  a.act = cf.dtype;  // the head reads the caller's embedding table
  a.x = hrows;
  a.ldx = ldh;
  a.w[0] = h->tok_emb;
  a.n_groups = 1;
  a.group_rows = cf.vocab;
  a.M = B;
  a.N = cf.vocab;
  a.K = cf.d_model;
  a.split = 1;
  a.epi = el;
  c.check(launch_gemm(a, static_cast<int *>(h->err.p), c.st), 1);
}

// LM head over B rows of h + greedy select for step k.  Step 0 (after the prefill)
// reads row-major h rows b*Lp + Lp-1 (row stride ldh); decode steps read the
// row-tiled h through the stream-K kernel.  The chosen token is embedded and
// normalised into the row-tiled decode h for the next step.
void head(Ctx &c, const void *hrows, int ldh, int B, int step, int Lp, int Lgen,
          const int32_t *force, int32_t *out_ids, float *out_lp, const int32_t *log_map,
          float *logits_out) {
  he_engine *h = c.h;
  const he_config &cf = h->cfg;
  const bool dec = step > 0;
  const int R = act_rows(h, B, true);
  Epi el{};
  el.kind = EPI_STORE_F32;
  el.partial = static_cast<float *>(h->logits.p);
  el.ldp = cf.vocab;
  // Greedy decode steps without teacher forcing or logit capture fuse the choice into
  // the LM head: its epilogue leaves per-tile {max, exp-sum, argmax} statistics
  // (in the logits buffer) instead of the logits, and a small kernel merges them.
  const int n_tiles = (cf.vocab + 127) / 128;
  bool fused_head = false;
  if (dec && use_stream_k(h, B, cf.vocab, cf.d_model, true, false)) {
    const void *we[1] = {h->tok_emb};
    if (h->temperature == 0.f && !force && !log_map) {
      Epi ea{};
      ea.kind = EPI_ARGMAX;
      ea.partial = static_cast<float *>(h->logits.p);
      ea.ldp = B;
      GemmArgs probe{};
      probe.act = cf.dtype;
      probe.x = hrows;
      probe.w[0] = h->tok_emb;
      probe.n_groups = 1;
      probe.group_rows = cf.vocab;
      probe.M = B;
      probe.N = cf.vocab;
      probe.K = cf.d_model;
      probe.split = 1;
      probe.epi = ea;
      fused_head = sk_argmax_ok(probe, sk_ctas(probe, h->num_sms, true));
      if (fused_head)
        gemm(c, HE_KCLASS_HEAD, hrows, ldh, we, 1, cf.vocab, B, cf.d_model, ea, true, false,
             cf.dtype);
    }
    if (!fused_head)
      gemm(c, HE_KCLASS_HEAD, hrows, ldh, we, 1, cf.vocab, B, cf.d_model, el, true, false,
           cf.dtype);
  } else {
    head_rows_gemm(c, hrows, ldh, B);
  }
  if (!dec && R > 0) {
    // from here on h, ctx and mid hold row-tiled decode tiles whose padding rows
    // (B..R-1) must read as zero
    const size_t e = h->elem;
    c.check(launch_zero(h->h.p, (size_t)R * cf.d_model * e, c.st), 1);
    c.check(launch_zero(h->ctx.p, (size_t)R * cf.d_model * e, c.st), 1);
    c.check(launch_zero(h->mid.p, (size_t)R * cf.ffn * e, c.st), 1);
  }
  Timed t(h, HE_KCLASS_HEAD, c.st);
  HeadArgs ha{};
  ha.logits = static_cast<float *>(h->logits.p);
  ha.ldl = cf.vocab;
  ha.vocab = cf.vocab;
  ha.B = B;
  ha.step = step;
  ha.gen_len = Lgen;
  ha.force_ids = force;
  ha.out_ids = out_ids;
  ha.out_lp = out_lp;
  ha.log_map = log_map;
  ha.logits_out = logits_out;
  ha.embed_next = step + 1 < Lgen;
  ha.pos = Lp + step;  // position of the token emitted at this step
  ha.tok_emb = h->tok_emb;
  ha.pos_emb = h->pos_emb;
  ha.pos_offset = cf.pos_offset;
  ha.g = h->layers[0].ln1_g;
  ha.b = h->layers[0].ln1_b;
  ha.eps = cf.ln_eps;
  ha.x = static_cast<float *>(h->x.p);
  ha.h = h->h.p;
  ha.d = cf.d_model;
  ha.h_rows = R;
  ha.temperature = h->temperature;
  ha.top_p = h->top_p;
  ha.seed = h->seed;
  if (fused_head) {
    ha.stats = static_cast<const float4 *>(h->logits.p);
    ha.n_tiles = n_tiles;
  }
  c.check(launch_head_select(cf.dtype, h->act, ha, c.st), 1);
}

// Total bytes of the six projections of every layer in the config's dtype.
size_t all_proj_bytes(const he_engine *h) {
  const he_config &c = h->cfg;
  return (size_t)c.n_layers * (4 * (size_t)c.d_model * c.d_model + 2 * (size_t)c.d_model * c.ffn) *
         h->elem;
}
int proj_rows(const he_config &c, int p) { return p == HE_PROJ_FC1 ? c.ffn : c.d_model; }
int proj_cols(const he_config &c, int p) { return p == HE_PROJ_FC2 ? c.ffn : c.d_model; }

// The generation copy of the projections on a BF16 engine: the fp16 tiled weights
// (all of them), then, with fp8 weights, the fp8 tiled codes and the fp32 row
// scales.  proj_copy_bytes sizes it; assign_proj_copy points fused_w (and fused_w8,
// fused_scale) into it.
size_t proj_copy_bytes(const he_engine *h) {
  const size_t w16 = all_proj_bytes(h);
  if (h->wfmt != HE_WEIGHTS_FP8) return w16;
  const he_config &c = h->cfg;
  const size_t rows = (size_t)c.n_layers * (5 * (size_t)c.d_model + c.ffn);
  return w16 + w16 / 2 + rows * sizeof(float);
}

void assign_proj_copy(he_engine *h, void *buf) {
  const he_config &c = h->cfg;
  const size_t n = (size_t)c.n_layers * HE_N_PROJ;
  const bool fp8 = h->wfmt == HE_WEIGHTS_FP8;
  h->fused_w.assign(n, nullptr);
  h->fused_w8.assign(fp8 ? n : 0, nullptr);
  h->fused_scale.assign(fp8 ? n : 0, nullptr);
  const size_t w16 = all_proj_bytes(h);
  size_t o16 = 0, o8 = w16, os = w16 + w16 / 2;
  for (int l = 0; l < c.n_layers; ++l)
    for (int p = 0; p < HE_N_PROJ; ++p) {
      const size_t i = (size_t)l * HE_N_PROJ + p, rc = (size_t)proj_rows(c, p) * proj_cols(c, p);
      h->fused_w[i] = at(buf, o16);
      o16 += rc * 2;
      if (fp8) {
        h->fused_w8[i] = at(buf, o8);
        h->fused_scale[i] = reinterpret_cast<const float *>(at(buf, os));
        o8 += rc;
        os += (size_t)proj_rows(c, p) * sizeof(float);
      }
    }
}

// Writes projection (l, p) of the generation copy from the caller's bf16 weight,
// merged with its LoRA pair when `lora`: fp16 tiled, or fp8 codes + scales.
cudaError_t convert_proj(he_engine *h, int l, int p, bool lora, cudaStream_t st) {
  const he_config &c = h->cfg;
  const he_layer_weights &lw = h->layers[l];
  const size_t i = (size_t)l * HE_N_PROJ + p;
  const float scale = lora ? c.lora_alpha / (float)c.lora_r : 0.f;
  const void *a = lora ? lw.lora_a[p] : nullptr, *b = lora ? lw.lora_b[p] : nullptr;
  if (h->wfmt == HE_WEIGHTS_FP8)
    return launch_fuse_fp8(const_cast<void *>(h->fused_w8[i]), const_cast<void *>(h->fused_w[i]),
                           const_cast<float *>(h->fused_scale[i]), lw.w[p], a, b, proj_rows(c, p),
                           proj_cols(c, p), c.lora_r, scale, st);
  return launch_fuse_tiled(const_cast<void *>(h->fused_w[i]), ACT_F16, lw.w[p], a, b,
                           proj_rows(c, p), proj_cols(c, p), c.lora_r, scale, st,
                           static_cast<int *>(h->err.p));
}

// BF16 engines always generate in fp16 from tiled projections.  While LoRA is fused
// those are he_fuse_lora's merged copies; otherwise every generation first converts
// the caller's bf16 weights into h->base (bf16 activations lose accuracy with depth;
// the weights may have changed since the last call).  prepare_base takes the
// buffer, outside any stream capture; retile_base enqueues the conversion.
he_status prepare_base(he_engine *h, cudaStream_t st) {
  const he_config &c = h->cfg;
  if (c.dtype != HE_DTYPE_BF16 || h->fused) return HE_OK;
  if (!h->base.p && !get(h, h->base, proj_copy_bytes(h), st))
    return fail(HE_ERR_OOM, "copy of the projections (%zu bytes) failed", proj_copy_bytes(h));
  assign_proj_copy(h, h->base.p);
  h->tiled = true;
  return HE_OK;
}

void retile_base(Ctx &c) {
  he_engine *h = c.h;
  const he_config &cf = h->cfg;
  if (cf.dtype != HE_DTYPE_BF16 || h->fused) return;
  for (int l = 0; l < cf.n_layers; ++l)
    for (int p = 0; p < HE_N_PROJ; ++p)
      c.check(convert_proj(h, l, p, false, c.st), h->wfmt == HE_WEIGHTS_FP8 ? 3 : 1);
}

// Activation type of a generation: fp32 engines fp32, bf16 engines fp16.
int gen_act(const he_engine *h) { return h->cfg.dtype == HE_DTYPE_F32 ? ACT_F32 : ACT_F16; }

// Phase events: recorded as graph nodes while a generation is being captured.
void record_phase(he_engine *h, int i, cudaStream_t st) {
  if (h->capturing)
    cudaEventRecordWithFlags(h->ph[i], st, cudaEventRecordExternal);
  else
    cudaEventRecord(h->ph[i], st);
}

he_status generate_impl(he_engine *h, const int32_t *prompt, int B, int Lp, int Lgen,
                        int32_t *out_ids, float *out_lp, const int32_t *force,
                        const int32_t *log_map, float *logits_out, cudaStream_t st) {
  const he_config &cf = h->cfg;
  const int d = cf.d_model;
  Ctx c{h, st};
  if (cf.dtype == HE_DTYPE_BF16 && !h->tiled) return fail(HE_ERR_STATE, "projections not prepared");
  h->act = gen_act(h);
  for (int k = 0; k < kClasses; ++k) h->prof_used[k] = 0;
  ensure_phase_events(h);
  retile_base(c);  // unfused bf16: this call's fp16 copy of the caller's weights
  record_phase(h, 0, st);
  // the GEMMs leave the tile counters at zero; clearing them here also recovers
  // from a call whose GEMM gave up on a wait part-way
  c.check(cudaMemsetAsync(h->tilecnt.p, 0, tilecnt_bytes(cf), st), 0);
  c.check(cudaMemsetAsync(h->attncnt.p, 0, attncnt_bytes(cf), st), 0);
  // ---- prefill: all prompt tokens of all sequences in one pass ----
  const int M = B * Lp;
  {
    Timed t(h, HE_KCLASS_OTHER, st);
    c.check(launch_embed_ln(cf.dtype, h->act, prompt, M, Lp, 0, h->tok_emb, h->pos_emb, cf.pos_offset,
                            cf.vocab, h->layers[0].ln1_g, h->layers[0].ln1_b, cf.ln_eps,
                            static_cast<float *>(h->x.p), h->h.p, d,
                            static_cast<int *>(h->err.p), st),
            1);
  }
  for (int l = 0; l < cf.n_layers; ++l) layer_forward(c, l, B, M, Lp, 0, true);
  // head on the last prompt position of every sequence (rows b*Lp + Lp-1)
  head(c, at(h->h.p, (size_t)(Lp - 1) * d * h->elem), Lp * d, B, 0, Lp, Lgen, force, out_ids,
       out_lp, log_map, logits_out);
  record_phase(h, 1, st);
  // ---- decode: token k is fed at position Lp + k - 1 ----
  for (int k = 1; k < Lgen; ++k) {
    const int t = Lp + k - 1;
    for (int l = 0; l < cf.n_layers; ++l) layer_forward(c, l, B, B, 1, t, false);
    head(c, h->h.p, d, B, k, Lp, Lgen, force, out_ids, out_lp, log_map, logits_out);
  }
  record_phase(h, 2, st);
  h->stats.generate_calls++;
  h->stats_pending = true;
  if (c.e != cudaSuccess) return cuda_fail(c.e, "he_generate launch");
  return HE_OK;
}

he_status check_generate_args(he_engine *h, const void *prompt, int B, int Lp, int Lgen,
                              const void *ids, const void *lp) {
  if (!h) return fail(HE_ERR_ARG, "engine is NULL");
  if (!prompt || !ids || !lp) return fail(HE_ERR_ARG, "NULL buffer");
  const he_config &c = h->cfg;
  if (B < 1 || B > c.max_batch) return fail(HE_ERR_ARG, "B=%d outside [1, max_batch=%d]", B, c.max_batch);
  if (Lp < 1 || Lgen < 1) return fail(HE_ERR_ARG, "Lp=%d and Lgen=%d must be >= 1", Lp, Lgen);
  if ((long long)Lp + Lgen > c.max_seq)
    return fail(HE_ERR_ARG, "Lp + Lgen = %lld exceeds max_seq=%d", (long long)Lp + Lgen, c.max_seq);
  if ((long long)Lp + Lgen - 1 > c.max_pos)
    return fail(HE_ERR_ARG, "positions up to %lld exceed max_pos=%d", (long long)Lp + Lgen - 2,
                c.max_pos);
  if (!h->taken) return fail(HE_ERR_STATE, "workspace is released; call he_retake_workspace");
  return HE_OK;
}

uint32_t float_bits(float f) {
  uint32_t u;
  std::memcpy(&u, &f, sizeof u);
  return u;
}

void drop_graph(he_engine *h) {
  if (h->gexec) cudaGraphExecDestroy(h->gexec);
  h->gexec = nullptr;
  h->gkey.clear();
}

// A generation from h->ids_in into h->ids_out / h->lp_out: launched directly, or,
// with he_set_cuda_graph on and profiling off, as the replay of a captured graph
// of the whole generation (re-captured when the shape, the activation type or any
// buffer address differs from the captured one).
he_status generate_internal(he_engine *h, int B, int Lp, int Lgen, cudaStream_t st) {
  int32_t *ids_in = static_cast<int32_t *>(h->ids_in.p);
  int32_t *ids_out = static_cast<int32_t *>(h->ids_out.p);
  float *lp_out = static_cast<float *>(h->lp_out.p);
  if (!h->graph_on || h->prof_mask)
    return generate_impl(h, ids_in, B, Lp, Lgen, ids_out, lp_out, nullptr, nullptr, nullptr, st);
  const int act = gen_act(h);
  std::vector<const void *> key = {
      reinterpret_cast<const void *>((uintptr_t)B), reinterpret_cast<const void *>((uintptr_t)Lp),
      reinterpret_cast<const void *>((uintptr_t)Lgen), reinterpret_cast<const void *>((uintptr_t)act),
      h->kc.p, h->vc.p, h->x.p, h->h.p, h->q.p, h->ctx.p, h->mid.p, h->partial.p, h->logits.p,
      h->attn_part.p, h->ids_in.p, h->ids_out.p, h->lp_out.p, h->err.p, h->tilecnt.p,
      h->restore.p, h->base.p, reinterpret_cast<const void *>((uintptr_t)h->fused),
      reinterpret_cast<const void *>((uintptr_t)h->wfmt),
      reinterpret_cast<const void *>((uintptr_t)float_bits(h->temperature)),
      reinterpret_cast<const void *>((uintptr_t)float_bits(h->top_p)),
      reinterpret_cast<const void *>((uintptr_t)h->seed)};
  if (!h->gexec || key != h->gkey) {
    if (!h->cap_stream &&
        cudaStreamCreateWithFlags(&h->cap_stream, cudaStreamNonBlocking) != cudaSuccess)
      return fail(HE_ERR_CUDA, "capture stream creation failed");
    ensure_phase_events(h);
    const unsigned long long l0 = h->stats.launches;
    const unsigned long long calls0 = h->stats.generate_calls;
    cudaError_t e = cudaStreamBeginCapture(h->cap_stream, cudaStreamCaptureModeRelaxed);
    if (e != cudaSuccess) return cuda_fail(e, "graph capture begin");
    h->capturing = true;
    he_status s = generate_impl(h, ids_in, B, Lp, Lgen, ids_out, lp_out, nullptr, nullptr,
                                nullptr, h->cap_stream);
    h->capturing = false;
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(h->cap_stream, &g);
    h->stats.generate_calls = calls0;  // counted at each replay below
    if (s != HE_OK || e != cudaSuccess || !g) {
      if (g) cudaGraphDestroy(g);
      drop_graph(h);
      return s != HE_OK ? s : cuda_fail(e != cudaSuccess ? e : cudaErrorUnknown, "graph capture");
    }
    h->glaunches = h->stats.launches - l0;
    h->stats.launches = l0;
    bool updated = false;
    if (h->gexec && h->gkey.size() >= 4 &&
        std::equal(key.begin(), key.begin() + 4, h->gkey.begin())) {
      cudaGraphExecUpdateResultInfo info;
      updated = cudaGraphExecUpdate(h->gexec, g, &info) == cudaSuccess;
      if (!updated) cudaGetLastError();
    }
    if (!updated) {
      drop_graph(h);
      e = cudaGraphInstantiate(&h->gexec, g, 0);
      if (e != cudaSuccess) {
        h->gexec = nullptr;
        cudaGraphDestroy(g);
        return cuda_fail(e, "graph instantiation");
      }
    }
    cudaGraphDestroy(g);
    h->gkey = key;
  }
  cudaError_t e = cudaGraphLaunch(h->gexec, st);
  if (e != cudaSuccess) return cuda_fail(e, "graph launch");
  h->stats.launches += h->glaunches;
  h->stats.generate_calls++;
  h->stats_pending = true;
  return HE_OK;
}

}  // namespace

// ============================================================================
// C ABI
// ============================================================================
extern "C" {

const char *he_last_error(void) { return g_err.c_str(); }

const char *he_version(void) { return "libhe 0.1 (sm_103a; tcgen05 bf16 GEMM, fp32 CUDA-core path)"; }

he_status he_create(const he_config *cfg, const he_weights *w, const he_allocator *alloc,
                    int device, he_engine **out) {
  g_err.clear();
  if (!out) return fail(HE_ERR_ARG, "out is NULL");
  *out = nullptr;
  if (!cfg || !w) return fail(HE_ERR_ARG, "cfg or weights is NULL");
  const he_config c = *cfg;
  if (c.n_layers < 1 || c.d_model < 1 || c.n_heads < 1 || c.ffn < 1 || c.vocab < 1 ||
      c.max_pos < 1 || c.pos_offset < 0 || c.max_batch < 1 || c.max_seq < 2)
    return fail(HE_ERR_ARG, "non-positive size in config");
  if (c.d_model % c.n_heads) return fail(HE_ERR_ARG, "d_model %% n_heads != 0");
  const int hd = c.d_model / c.n_heads;
  if (hd != 32 && hd != 64 && hd != 128)
    return fail(HE_ERR_UNSUPPORTED, "head_dim %d not in {32, 64, 128}", hd);
  if (c.dtype != HE_DTYPE_F32 && c.dtype != HE_DTYPE_BF16) return fail(HE_ERR_ARG, "bad dtype");
  if (!(c.ln_eps > 0.f)) return fail(HE_ERR_ARG, "ln_eps must be > 0");
  if (c.d_model % 8 || c.ffn % 8) return fail(HE_ERR_UNSUPPORTED, "d_model and ffn must be multiples of 8");
  if (c.dtype == HE_DTYPE_BF16 && (c.d_model % 128 || c.ffn % 128))
    return fail(HE_ERR_UNSUPPORTED, "bf16 path needs d_model and ffn multiples of 128");
  if (c.lora_targets & ~0x3Fu) return fail(HE_ERR_ARG, "unknown bits in lora_targets");
  if (c.lora_targets && (c.lora_r < 1 || c.lora_r > 64))
    return fail(HE_ERR_ARG, "lora_r %d outside [1, 64]", c.lora_r);
  if ((long long)c.max_batch * c.max_seq > (1LL << 30) ||
      (long long)c.max_batch * c.max_seq * (c.ffn > c.vocab ? c.ffn : c.vocab) > (1LL << 40))
    return fail(HE_ERR_UNSUPPORTED, "max_batch * max_seq too large");
  if (!w->tok_emb || !w->pos_emb || !w->lnf_g || !w->lnf_b || !w->layers)
    return fail(HE_ERR_ARG, "NULL global weight pointer");
  const size_t align = c.dtype == HE_DTYPE_BF16 ? 16 : 4;
  auto misaligned = [&](const void *p) { return ((uintptr_t)p) % align != 0; };
  if (misaligned(w->tok_emb)) return fail(HE_ERR_ARG, "tok_emb not %zu-byte aligned", align);
  for (int l = 0; l < c.n_layers; ++l) {
    const he_layer_weights &lw = w->layers[l];
    for (int p = 0; p < HE_N_PROJ; ++p) {
      if (!lw.w[p] || !lw.b[p]) return fail(HE_ERR_ARG, "layer %d projection %d: NULL", l, p);
      if (misaligned(lw.w[p])) return fail(HE_ERR_ARG, "layer %d projection %d: not %zu-byte aligned", l, p, align);
      if ((c.lora_targets >> p) & 1u)
        if (!lw.lora_a[p] || !lw.lora_b[p])
          return fail(HE_ERR_ARG, "layer %d projection %d: NULL LoRA factor", l, p);
    }
    if (!lw.ln1_g || !lw.ln1_b || !lw.ln2_g || !lw.ln2_b)
      return fail(HE_ERR_ARG, "layer %d: NULL LayerNorm parameter", l);
  }
  if (cudaSetDevice(device) != cudaSuccess) return fail(HE_ERR_CUDA, "cudaSetDevice(%d) failed", device);
  int sms = 0;
  cudaError_t ce = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
  if (ce != cudaSuccess) return cuda_fail(ce, "device query");
  if (c.dtype == HE_DTYPE_BF16) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device);
    if (major != 10 || minor != 3)
      return fail(HE_ERR_UNSUPPORTED, "bf16 kernels are built for sm_103a; device is sm_%d%d", major, minor);
  }
  he_engine *h = new he_engine();
  h->cfg = c;
  h->device = device;
  h->num_sms = sms;
  h->elem = c.dtype == HE_DTYPE_BF16 ? 2 : 4;
  h->tok_emb = w->tok_emb;
  h->pos_emb = w->pos_emb;
  h->lnf_g = w->lnf_g;
  h->lnf_b = w->lnf_b;
  h->layers.assign(w->layers, w->layers + c.n_layers);
  if (alloc && alloc->alloc && alloc->free)
    h->alloc = *alloc;
  else
    h->alloc = he_allocator{default_alloc, default_free, nullptr};
  if (!get(h, h->err, 256, nullptr)) {
    delete h;
    return fail(HE_ERR_OOM, "error-flag allocation failed");
  }
  if (!get(h, h->tilecnt, tilecnt_bytes(c), nullptr) ||
      !get(h, h->attncnt, attncnt_bytes(c), nullptr)) {
    put(h, h->tilecnt, nullptr);
    put(h, h->err, nullptr);
    delete h;
    return fail(HE_ERR_OOM, "counter allocation failed");
  }
  ce = cudaMemset(h->err.p, 0, 256);
  if (ce == cudaSuccess) ce = cudaMemset(h->tilecnt.p, 0, tilecnt_bytes(c));
  if (ce == cudaSuccess) ce = cudaMemset(h->attncnt.p, 0, attncnt_bytes(c));
  if (ce != cudaSuccess) {
    put(h, h->attncnt, nullptr);
    put(h, h->tilecnt, nullptr);
    put(h, h->err, nullptr);
    delete h;
    return cuda_fail(ce, "memset");
  }
  he_status s = take_workspace(h, nullptr);
  if (s != HE_OK) {
    put(h, h->attncnt, nullptr);
    put(h, h->tilecnt, nullptr);
    put(h, h->err, nullptr);
    delete h;
    return s;
  }
  *out = h;
  return HE_OK;
}

he_status he_destroy(he_engine *h) {
  if (!h) return HE_OK;
  cudaSetDevice(h->device);
  cudaDeviceSynchronize();
  free_workspace(h, nullptr);
  put(h, h->restore, nullptr);
  put(h, h->tilecnt, nullptr);
  put(h, h->attncnt, nullptr);
  put(h, h->err, nullptr);
  drop_graph(h);
  if (h->cap_stream) cudaStreamDestroy(h->cap_stream);
  for (auto &e : h->ph)
    if (e) cudaEventDestroy(e);
  for (auto &pool : h->prof_pool)
    for (auto &p : pool) {
      cudaEventDestroy(p.a);
      cudaEventDestroy(p.b);
    }
  delete h;
  return HE_OK;
}

// Which projections the fuse saves and rewrites: bf16 rewrites all six (merged
// where LoRA-targeted) into the tiled streaming layout; fp32 merges the targeted
// ones in place.
static bool fuse_touches(const he_engine *h, int p) {
  return h->cfg.dtype == HE_DTYPE_BF16 || ((h->cfg.lora_targets >> p) & 1u);
}

he_status he_fuse_lora(he_engine *h, void *stream) {
  g_err.clear();
  if (!h) return fail(HE_ERR_ARG, "engine is NULL");
  if (h->fused) return fail(HE_ERR_STATE, "LoRA is already fused");
  cudaSetDevice(h->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const he_config &c = h->cfg;
  const bool bf = c.dtype == HE_DTYPE_BF16;
  size_t total = 0;
  if (bf) {
    total = proj_copy_bytes(h);
  } else {
    for (int l = 0; l < c.n_layers; ++l)
      for (int p = 0; p < HE_N_PROJ; ++p)
        if (fuse_touches(h, p)) total += (size_t)proj_rows(c, p) * proj_cols(c, p) * h->elem;
  }
  put(h, h->base, st);  // the unfused generations' copy: the fused one replaces it
  h->fused_w.clear();
  h->fused_w8.clear();
  h->fused_scale.clear();
  h->tiled = false;
  if (!get(h, h->restore, total, st))
    return fail(HE_ERR_OOM, "LoRA fuse buffer of %zu bytes failed", total);
  ensure_phase_events(h);
  cudaEventRecord(h->ph[3], st);
  const float scale = c.lora_targets ? c.lora_alpha / (float)c.lora_r : 0.f;
  cudaError_t err = cudaSuccess;
  auto chk = [&](cudaError_t e, int n) {
    if (e != cudaSuccess && err == cudaSuccess) err = e;
    h->stats.launches += n;
  };
  if (bf) {
    // the merged weights (all six projections, tiled; fp8 codes and scales with fp8
    // weights) into the engine's buffer; w[] stays as it is
    assign_proj_copy(h, h->restore.p);
    for (int l = 0; l < c.n_layers; ++l)
      for (int p = 0; p < HE_N_PROJ; ++p)
        chk(convert_proj(h, l, p, (c.lora_targets >> p) & 1u, st),
            h->wfmt == HE_WEIGHTS_FP8 ? 3 : 1);
  } else {
    size_t off = 0;
    for (int l = 0; l < c.n_layers; ++l) {
      const he_layer_weights &lw = h->layers[l];
      for (int p = 0; p < HE_N_PROJ; ++p) {
        if (!fuse_touches(h, p)) continue;
        chk(launch_lora_fuse(c.dtype, lw.w[p], lw.lora_a[p], lw.lora_b[p], at(h->restore.p, off),
                             proj_rows(c, p), proj_cols(c, p), c.lora_r, scale, st),
            1);
        off += (size_t)proj_rows(c, p) * proj_cols(c, p) * h->elem;
      }
    }
  }
  cudaEventRecord(h->ph[4], st);
  h->fuse_pending = true;
  h->fused = true;
  h->tiled = bf;
  h->stats.restore_bytes = total;
  if (err != cudaSuccess) return cuda_fail(err, "LoRA fuse launch");
  return HE_OK;
}

he_status he_set_weight_format(he_engine *h, int format) {
  g_err.clear();
  if (!h) return fail(HE_ERR_ARG, "engine is NULL");
  if (format != HE_WEIGHTS_F16 && format != HE_WEIGHTS_FP8) return fail(HE_ERR_ARG, "bad format");
  if (h->cfg.dtype != HE_DTYPE_BF16 && format != HE_WEIGHTS_F16)
    return fail(HE_ERR_UNSUPPORTED, "fp8 weights need a BF16 engine");
  if (h->fused) return fail(HE_ERR_STATE, "unfuse LoRA before changing the weight format");
  if (format == h->wfmt) return HE_OK;
  cudaSetDevice(h->device);
  put(h, h->base, nullptr);  // its layout depends on the format
  h->fused_w.clear();
  h->fused_w8.clear();
  h->fused_scale.clear();
  h->tiled = false;
  h->wfmt = format;
  return HE_OK;
}

he_status he_read_fused_fp8(he_engine *h, int layer, int proj, void *codes, size_t code_bytes,
                            float *scales, void *stream) {
  g_err.clear();
  if (!h || !codes || !scales) return fail(HE_ERR_ARG, "NULL argument");
  if (!h->fused || h->wfmt != HE_WEIGHTS_FP8)
    return fail(HE_ERR_STATE, "LoRA is not fused with fp8 weights");
  const he_config &c = h->cfg;
  if (layer < 0 || layer >= c.n_layers || proj < 0 || proj >= HE_N_PROJ)
    return fail(HE_ERR_ARG, "bad layer or projection");
  const size_t rows = proj_rows(c, proj), cols = proj_cols(c, proj);
  if (code_bytes != rows * cols) return fail(HE_ERR_ARG, "code_bytes must be %zu", rows * cols);
  cudaSetDevice(h->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t i = (size_t)layer * HE_N_PROJ + proj;
  cudaError_t e = cudaMemcpyAsync(codes, h->fused_w8[i], rows * cols, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(scales, h->fused_scale[i], rows * sizeof(float), cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "he_read_fused_fp8");
  return HE_OK;
}

he_status he_read_fused_weight(he_engine *h, int layer, int proj, void *dst, size_t bytes,
                               void *stream) {
  g_err.clear();
  if (!h || !dst) return fail(HE_ERR_ARG, "NULL argument");
  if (!h->fused) return fail(HE_ERR_STATE, "LoRA is not fused");
  const he_config &c = h->cfg;
  if (layer < 0 || layer >= c.n_layers || proj < 0 || proj >= HE_N_PROJ)
    return fail(HE_ERR_ARG, "bad layer or projection");
  const size_t rows = proj == HE_PROJ_FC1 ? c.ffn : c.d_model;
  const size_t cols = proj == HE_PROJ_FC2 ? c.ffn : c.d_model;
  if (bytes != rows * cols * h->elem) return fail(HE_ERR_ARG, "bytes must be %zu", rows * cols * h->elem);
  cudaSetDevice(h->device);
  const void *src = h->tiled ? h->fused_w[(size_t)layer * HE_N_PROJ + proj] : h->layers[layer].w[proj];
  cudaError_t e = cudaMemcpyAsync(dst, src, bytes, cudaMemcpyDeviceToDevice,
                                  static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "he_read_fused_weight");
  return HE_OK;
}

he_status he_unfuse_lora(he_engine *h, void *stream) {
  g_err.clear();
  if (!h) return fail(HE_ERR_ARG, "engine is NULL");
  if (!h->fused) return fail(HE_ERR_STATE, "LoRA is not fused");
  cudaSetDevice(h->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const he_config &c = h->cfg;
  auto rows_of = [&](int p) { return p == HE_PROJ_FC1 ? c.ffn : c.d_model; };
  auto cols_of = [&](int p) { return p == HE_PROJ_FC2 ? c.ffn : c.d_model; };
  ensure_phase_events(h);
  cudaEventRecord(h->ph[5], st);
  size_t off = 0;
  cudaError_t err = cudaSuccess;
  if (c.dtype != HE_DTYPE_BF16) {  // BF16 never wrote w[]: releasing the buffer is all
    for (int l = 0; l < c.n_layers; ++l)
      for (int p = 0; p < HE_N_PROJ; ++p) {
        if (!fuse_touches(h, p)) continue;
        const size_t bytes = (size_t)rows_of(p) * cols_of(p) * h->elem;
        cudaError_t e = launch_copy(h->layers[l].w[p], at(h->restore.p, off), bytes, st);
        if (e != cudaSuccess && err == cudaSuccess) err = e;
        h->stats.launches += (bytes % 16 ? 2 : 1);
        off += bytes;
      }
  }
  cudaEventRecord(h->ph[6], st);
  h->unfuse_pending = true;
  put(h, h->restore, st);
  h->fused_w.clear();
  h->fused_w8.clear();
  h->fused_scale.clear();
  h->fused = false;
  h->tiled = false;
  h->stats.restore_bytes = 0;
  if (err != cudaSuccess) return cuda_fail(err, "LoRA restore launch");
  return HE_OK;
}

he_status he_generate(he_engine *h, const int32_t *prompt_ids, int B, int Lp, int Lgen,
                      int32_t *out_ids, float *out_logprob, void *stream) {
  if (!h || !h->graph_on)
    return he_generate_ex(h, prompt_ids, B, Lp, Lgen, out_ids, out_logprob, nullptr, nullptr, 0,
                          nullptr, stream);
  // graph mode: the captured generation reads and writes the engine's own buffers
  g_err.clear();
  he_status s = check_generate_args(h, prompt_ids, B, Lp, Lgen, out_ids, out_logprob);
  if (s != HE_OK) return s;
  cudaSetDevice(h->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = prepare_base(h, st);
  if (s != HE_OK) return s;
  cudaError_t e = cudaMemcpyAsync(h->ids_in.p, prompt_ids, (size_t)B * Lp * 4,
                                  cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "prompt copy");
  s = generate_internal(h, B, Lp, Lgen, st);
  if (s != HE_OK) return s;
  e = cudaMemcpyAsync(out_ids, h->ids_out.p, (size_t)B * Lgen * 4, cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(out_logprob, h->lp_out.p, (size_t)B * Lgen * 4, cudaMemcpyDeviceToDevice,
                        st);
  if (e != cudaSuccess) return cuda_fail(e, "result copy");
  return HE_OK;
}

he_status he_set_sampling(he_engine *h, float temperature, float top_p,
                          unsigned long long seed) {
  g_err.clear();
  if (!h) return fail(HE_ERR_ARG, "engine is NULL");
  if (!(temperature >= 0.f) || !std::isfinite(temperature))
    return fail(HE_ERR_ARG, "temperature must be finite and >= 0");
  if (!(top_p > 0.f && top_p <= 1.f)) return fail(HE_ERR_ARG, "top_p must be in (0, 1]");
  h->temperature = temperature;
  h->top_p = top_p;
  h->seed = seed;
  return HE_OK;
}

he_status he_set_cuda_graph(he_engine *h, int enable) {
  g_err.clear();
  if (!h) return fail(HE_ERR_ARG, "engine is NULL");
  cudaSetDevice(h->device);
  h->graph_on = enable != 0;
  if (!h->graph_on) drop_graph(h);
  return HE_OK;
}

he_status he_generate_ex(he_engine *h, const int32_t *prompt_ids, int B, int Lp, int Lgen,
                         int32_t *out_ids, float *out_logprob, const int32_t *force_ids,
                         const int32_t *log_rows, int n_rows, float *logits_out, void *stream) {
  g_err.clear();
  he_status s = check_generate_args(h, prompt_ids, B, Lp, Lgen, out_ids, out_logprob);
  if (s != HE_OK) return s;
  if (n_rows < 0 || (n_rows > 0 && (!log_rows || !logits_out)))
    return fail(HE_ERR_ARG, "n_rows > 0 needs log_rows and logits_out");
  cudaSetDevice(h->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = prepare_base(h, st);
  if (s != HE_OK) return s;
  const int32_t *log_map = nullptr;
  if (n_rows > 0) {
    std::vector<int32_t> map((size_t)Lgen * B, -1);
    for (int i = 0; i < n_rows; ++i) {
      const int b = log_rows[2 * i], k = log_rows[2 * i + 1];
      if (b < 0 || b >= B || k < 0 || k >= Lgen)
        return fail(HE_ERR_ARG, "log_rows[%d] = (%d, %d) out of range", i, b, k);
      map[(size_t)k * B + b] = i;
    }
    cudaError_t e = cudaMemcpyAsync(h->logmap.p, map.data(), map.size() * 4,
                                    cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return cuda_fail(e, "log map upload");
    // the host vector dies here: make the copy complete before returning
    e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "log map upload");
    log_map = static_cast<const int32_t *>(h->logmap.p);
  }
  return generate_impl(h, prompt_ids, B, Lp, Lgen, out_ids, out_logprob, force_ids, log_map,
                       logits_out, st);
}

he_status he_check(he_engine *h, void *stream) {
  g_err.clear();
  if (!h) return fail(HE_ERR_ARG, "engine is NULL");
  cudaSetDevice(h->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int flags = 0;
  cudaError_t e = cudaMemcpyAsync(&flags, h->err.p, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return cuda_fail(e, "he_check");
  if (flags) {
    cudaMemsetAsync(h->err.p, 0, sizeof(int), st);
    cudaStreamSynchronize(st);
    if (flags & DEVERR_WAIT_TIMEOUT)
      return fail(HE_ERR_DEVICE_CHECK, "a GEMM pipeline wait timed out (flags 0x%x)", flags);
    return fail(HE_ERR_DEVICE_CHECK, "token id outside [0, vocab) replaced by 0 (flags 0x%x)", flags);
  }
  return HE_OK;
}

he_status he_score(he_engine *h, const int32_t *ids, int B, int L, int Lp, float *out_logprob,
                   void *stream) {
  g_err.clear();
  if (!h) return fail(HE_ERR_ARG, "engine is NULL");
  if (!ids || !out_logprob) return fail(HE_ERR_ARG, "NULL buffer");
  const he_config &cf = h->cfg;
  if (B < 1 || B > cf.max_batch) return fail(HE_ERR_ARG, "B=%d outside [1, max_batch=%d]", B, cf.max_batch);
  if (Lp < 1 || L <= Lp) return fail(HE_ERR_ARG, "need 1 <= Lp < L (Lp=%d, L=%d)", Lp, L);
  if (L > cf.max_seq) return fail(HE_ERR_ARG, "L=%d exceeds max_seq=%d", L, cf.max_seq);
  if (L - 1 > cf.max_pos) return fail(HE_ERR_ARG, "positions up to %d exceed max_pos=%d", L - 2, cf.max_pos);
  if (!h->taken) return fail(HE_ERR_STATE, "workspace is released; call he_retake_workspace");
  cudaSetDevice(h->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int Lgen = L - Lp, T = L - 1, M = B * T, d = cf.d_model;
  int32_t *toks = static_cast<int32_t *>(h->ids_in.p);      // [B][T]: the tokens fed
  int32_t *targets = static_cast<int32_t *>(h->ids_out.p);  // [B][Lgen]: the tokens scored
  int32_t *echo = static_cast<int32_t *>(h->logmap.p);      // [B][Lgen]: ids the head emits
  cudaError_t e = cudaMemcpy2DAsync(toks, (size_t)T * 4, ids, (size_t)L * 4, (size_t)T * 4, B,
                                    cudaMemcpyDeviceToDevice, st);
  if (e == cudaSuccess)
    e = cudaMemcpy2DAsync(targets, (size_t)Lgen * 4, ids + Lp, (size_t)L * 4, (size_t)Lgen * 4, B,
                          cudaMemcpyDeviceToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "token copy");
  he_status ps = prepare_base(h, st);
  if (ps != HE_OK) return ps;
  Ctx c{h, st};
  h->act = gen_act(h);
  for (int k = 0; k < kClasses; ++k) h->prof_used[k] = 0;
  retile_base(c);
  c.check(cudaMemsetAsync(h->tilecnt.p, 0, tilecnt_bytes(cf), st), 0);
  // one pass over tokens 0 .. L-2 of every sequence (the prefill kernels)
  {
    Timed t(h, HE_KCLASS_OTHER, st);
    c.check(launch_embed_ln(cf.dtype, h->act, toks, M, T, 0, h->tok_emb, h->pos_emb, cf.pos_offset,
                            cf.vocab, h->layers[0].ln1_g, h->layers[0].ln1_b, cf.ln_eps,
                            static_cast<float *>(h->x.p), h->h.p, d,
                            static_cast<int *>(h->err.p), st),
            1);
  }
  for (int l = 0; l < cf.n_layers; ++l) layer_forward(c, l, B, M, T, 0, true);
  // the distribution at position Lp-1+k scores token Lp+k
  for (int k = 0; k < Lgen; ++k) {
    head_rows_gemm(c, at(h->h.p, (size_t)(Lp - 1 + k) * d * h->elem), T * d, B);
    Timed t(h, HE_KCLASS_HEAD, st);
    HeadArgs ha{};
    ha.logits = static_cast<float *>(h->logits.p);
    ha.ldl = cf.vocab;
    ha.vocab = cf.vocab;
    ha.B = B;
    ha.step = k;
    ha.gen_len = Lgen;
    ha.force_ids = targets;
    ha.out_ids = echo;
    ha.out_lp = out_logprob;
    ha.embed_next = 0;
    ha.temperature = h->temperature;  // log-probs under the sampling temperature
    ha.top_p = 1.f;
    c.check(launch_head_select(cf.dtype, h->act, ha, st), 1);
  }
  h->stats_pending = false;
  if (c.e != cudaSuccess) return cuda_fail(c.e, "he_score launch");
  return HE_OK;
}

he_status he_generate_host(he_engine *h, const int32_t *prompt_ids, int B, int Lp, int Lgen,
                           int32_t *out_ids, float *out_logprob, void *stream) {
  g_err.clear();
  he_status s = check_generate_args(h, prompt_ids, B, Lp, Lgen, out_ids, out_logprob);
  if (s != HE_OK) return s;
  cudaSetDevice(h->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  s = prepare_base(h, st);
  if (s != HE_OK) return s;
  cudaError_t e = cudaMemcpyAsync(h->ids_in.p, prompt_ids, (size_t)B * Lp * 4,
                                  cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return cuda_fail(e, "prompt upload");
  s = generate_internal(h, B, Lp, Lgen, st);
  if (s != HE_OK) return s;
  e = cudaMemcpyAsync(out_ids, h->ids_out.p, (size_t)B * Lgen * 4, cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(out_logprob, h->lp_out.p, (size_t)B * Lgen * 4, cudaMemcpyDeviceToHost, st);
  if (e != cudaSuccess) return cuda_fail(e, "result download");
  return he_check(h, stream);
}

he_status he_release_workspace(he_engine *h, void *stream) {
  g_err.clear();
  if (!h) return fail(HE_ERR_ARG, "engine is NULL");
  if (!h->taken) return fail(HE_ERR_STATE, "workspace already released");
  cudaSetDevice(h->device);
  free_workspace(h, static_cast<cudaStream_t>(stream));
  return HE_OK;
}

he_status he_retake_workspace(he_engine *h, void *stream) {
  g_err.clear();
  if (!h) return fail(HE_ERR_ARG, "engine is NULL");
  if (h->taken) return fail(HE_ERR_STATE, "workspace is already held");
  cudaSetDevice(h->device);
  return take_workspace(h, static_cast<cudaStream_t>(stream));
}

he_status he_set_profiling(he_engine *h, unsigned class_mask) {
  g_err.clear();
  if (!h) return fail(HE_ERR_ARG, "engine is NULL");
  h->prof_mask = class_mask & ((1u << kClasses) - 1);
  return HE_OK;
}

he_status he_get_stats(he_engine *h, he_stats *s) {
  g_err.clear();
  if (!h || !s) return fail(HE_ERR_ARG, "NULL argument");
  cudaSetDevice(h->device);
  float ms = 0.f;
  if (h->stats_pending) {
    if (cudaEventSynchronize(h->ph[2]) != cudaSuccess) return fail(HE_ERR_CUDA, "event sync");
    cudaEventElapsedTime(&ms, h->ph[0], h->ph[1]);
    h->stats.prefill_ms = ms;
    cudaEventElapsedTime(&ms, h->ph[1], h->ph[2]);
    h->stats.decode_ms = ms;
    for (int k = 0; k < kClasses; ++k) {
      double tot = 0.0;
      for (size_t i = 0; i < h->prof_used[k]; ++i) {
        float t = 0.f;
        cudaEventSynchronize(h->prof_pool[k][i].b);
        cudaEventElapsedTime(&t, h->prof_pool[k][i].a, h->prof_pool[k][i].b);
        tot += t;
      }
      h->stats.kclass_ms[k] = tot;
      h->stats.kclass_launches[k] = (long long)h->prof_used[k];
    }
    h->stats_pending = false;
  }
  if (h->fuse_pending) {
    cudaEventSynchronize(h->ph[4]);
    cudaEventElapsedTime(&ms, h->ph[3], h->ph[4]);
    h->stats.fuse_ms = ms;
    h->fuse_pending = false;
  }
  if (h->unfuse_pending) {
    cudaEventSynchronize(h->ph[6]);
    cudaEventElapsedTime(&ms, h->ph[5], h->ph[6]);
    h->stats.unfuse_ms = ms;
    h->unfuse_pending = false;
  }
  *s = h->stats;
  return HE_OK;
}

// ---------------------------------------------------------------------------
// Kernel-level entry (he_ops.h)
// ---------------------------------------------------------------------------
he_status he_op_attn_decode(int dtype, const void *q, const void *kc, const void *vc, void *ctx,
                            int B, int H, int hd, int max_seq, int n_keys, int split, float *part,
                            void *stream) {
  g_err.clear();
  if (!q || !kc || !vc || !ctx) return fail(HE_ERR_ARG, "NULL buffer");
  if (dtype != HE_DTYPE_F32 && dtype != HE_DTYPE_BF16 && dtype != HE_DTYPE_F16)
    return fail(HE_ERR_ARG, "bad dtype");
  if (B < 1 || H < 1 || n_keys < 1 || n_keys > max_seq || split < 1 || split > n_keys)
    return fail(HE_ERR_ARG, "bad sizes");
  if (hd != 32 && hd != 64 && hd != 128) return fail(HE_ERR_UNSUPPORTED, "head_dim %d", hd);
  if (split > 1 && !part) return fail(HE_ERR_ARG, "split > 1 needs part");
  cudaError_t r = launch_attn_decode(dtype, q, kc, vc, ctx, 0, B, H, hd, max_seq, n_keys, split,
                                     part, static_cast<cudaStream_t>(stream));
  if (r != cudaSuccess) return cuda_fail(r, "he_op_attn_decode");
  return HE_OK;
}

he_status he_op_attn_prefill(int dtype, const void *q, const void *kc, const void *vc, void *ctx,
                             int B, int Lp, int H, int hd, int max_seq, int flags, int *dev_flags,
                             void *stream) {
  g_err.clear();
  if (!q || !kc || !vc || !ctx) return fail(HE_ERR_ARG, "NULL buffer");
  if (dtype != HE_DTYPE_F32 && dtype != HE_DTYPE_BF16 && dtype != HE_DTYPE_F16)
    return fail(HE_ERR_ARG, "bad dtype");
  if (B < 1 || H < 1 || Lp < 1 || Lp > max_seq) return fail(HE_ERR_ARG, "bad sizes");
  if (hd != 32 && hd != 64 && hd != 128) return fail(HE_ERR_UNSUPPORTED, "head_dim %d", hd);
  if (flags & ~HE_ATTN_PREFILL_MMA_SYNC) return fail(HE_ERR_ARG, "unknown flags 0x%x", flags);
  if ((uintptr_t)q % 16 || (uintptr_t)kc % 16 || (uintptr_t)vc % 16 || (uintptr_t)ctx % 16)
    return fail(HE_ERR_ARG, "buffers not 16-byte aligned");
  cudaError_t r = launch_attn_prefill(dtype, q, kc, vc, ctx, B, Lp, H, hd, max_seq, dev_flags,
                                      static_cast<cudaStream_t>(stream),
                                      (flags & HE_ATTN_PREFILL_MMA_SYNC) != 0);
  if (r != cudaSuccess) return cuda_fail(r, "he_op_attn_prefill");
  return HE_OK;
}

he_status he_op_fuse_tiled(const void *w, const void *lora_a, const void *lora_b, int r, float scale,
                           void *out, int N, int K, void *stream) {
  g_err.clear();
  if (!w || !out || (r > 0 && (!lora_a || !lora_b))) return fail(HE_ERR_ARG, "NULL buffer");
  if (N < 128 || K < 64 || N % 128 || K % 64)
    return fail(HE_ERR_UNSUPPORTED, "tiled layout needs N %% 128 == 0 and K %% 64 == 0");
  if (r < 0 || r > 64) return fail(HE_ERR_ARG, "r %d outside [0, 64]", r);
  if ((uintptr_t)w % 16 || (uintptr_t)out % 16 || (r > 0 && (uintptr_t)lora_a % 16))
    return fail(HE_ERR_ARG, "buffers not 16-byte aligned");
  cudaError_t e = launch_fuse_tiled(out, ACT_F16, w, r > 0 ? lora_a : nullptr,
                                    r > 0 ? lora_b : nullptr, N, K, r, scale,
                                    static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "he_op_fuse_tiled");
  return HE_OK;
}

he_status he_op_tile_weight(const void *w, void *out, int N, int K, void *stream) {
  g_err.clear();
  if (!w || !out) return fail(HE_ERR_ARG, "NULL buffer");
  if (N < 128 || K < 64 || N % 128 || K % 64)
    return fail(HE_ERR_UNSUPPORTED, "tiled layout needs N %% 128 == 0 and K %% 64 == 0");
  if ((uintptr_t)w % 16 || (uintptr_t)out % 16) return fail(HE_ERR_ARG, "buffers not 16-byte aligned");
  cudaError_t r = launch_fuse_tiled(out, ACT_BF16, w, nullptr, nullptr, N, K, 0, 0.f,
                                    static_cast<cudaStream_t>(stream));
  if (r != cudaSuccess) return cuda_fail(r, "he_op_tile_weight");
  return HE_OK;
}

he_status he_op_head_greedy(int dtype, const void *x, int ldx, const void *w, int M, int N, int K,
                            int32_t *out_ids, float *out_lp, float *scratch, void *stream) {
  g_err.clear();
  if (!x || !w || !out_ids || !out_lp || !scratch) return fail(HE_ERR_ARG, "NULL buffer");
  if (dtype != HE_DTYPE_BF16 && dtype != HE_DTYPE_F16) return fail(HE_ERR_ARG, "dtype must be BF16 or F16");
  if (M < 1 || M > 256 || N < 1 || K < 64 || K % 64 || ldx < K || ldx % 8 || N % 4)
    return fail(HE_ERR_ARG, "need 1 <= M <= 256, K %% 64 == 0, ldx >= K, ldx %% 8 == 0, N %% 4 == 0");
  if ((uintptr_t)x % 16 || (uintptr_t)w % 16 || (uintptr_t)scratch % 16)
    return fail(HE_ERR_ARG, "buffers not 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long T = (N + 127) / 128;
  const int R = sk_token_tile(M);
  // scratch: slices [16][T][M][128] | row-tiled x | tile counters | statistics [T][M]
  const long long sstride = (long long)M * T * 128;
  void *xt = scratch + (size_t)16 * sstride;
  int *cnt = reinterpret_cast<int *>(((uintptr_t)xt + (size_t)R * K * 2 + 15) & ~(uintptr_t)15);
  float4 *stats = reinterpret_cast<float4 *>(((uintptr_t)(cnt + T) + 15) & ~(uintptr_t)15);
  GemmArgs a{};
  a.dtype = HE_DTYPE_BF16;
  a.act = dtype;
  a.x = xt;
  a.ldx = K;
  a.w[0] = w;
  a.n_groups = 1;
  a.group_rows = N;
  a.M = M;
  a.N = N;
  a.K = K;
  a.split = 1;
  Epi e{};
  e.kind = EPI_ARGMAX;
  e.partial = reinterpret_cast<float *>(stats);
  e.ldp = M;
  a.epi = e;
  const int P = sk_ctas(a, sms, true);
  if (!sk_argmax_ok(a, P)) return fail(HE_ERR_UNSUPPORTED, "tile statistics need the staged owner path");
  cudaError_t r = launch_tile_act(x, M, K, ldx, R, xt, st);
  if (r == cudaSuccess) r = cudaMemsetAsync(cnt, 0, (size_t)T * sizeof(int), st);
  if (r == cudaSuccess) r = launch_gemm_sk(a, P, scratch, sstride, cnt, nullptr, st);
  if (r == cudaSuccess) {
    HeadArgs ha{};
    ha.vocab = N;
    ha.B = M;
    ha.step = 0;
    ha.gen_len = 1;
    ha.out_ids = out_ids;
    ha.out_lp = out_lp;
    ha.stats = stats;
    ha.n_tiles = (int)T;
    ha.d = K;
    r = launch_head_select(HE_DTYPE_BF16, dtype, ha, st);
  }
  if (r != cudaSuccess) return cuda_fail(r, "he_op_head_greedy");
  return HE_OK;
}

he_status he_op_linear_fp8(const void *x, int ldx, const void *w8, const float *scale, float *y,
                           int M, int N, int K, int split, float *scratch, void *stream) {
  g_err.clear();
  if (!x || !w8 || !scale || !y || !scratch) return fail(HE_ERR_ARG, "NULL buffer");
  if (M < 1 || M > 128 || N < 128 || N % 128 || K < 256 || K % 256 || ldx < K || ldx % 8)
    return fail(HE_ERR_UNSUPPORTED, "fp8 GEMM needs 1 <= M <= 128, N %% 128 == 0, K %% 256 == 0, "
                                    "ldx >= K, ldx %% 8 == 0");
  if ((uintptr_t)x % 16 || (uintptr_t)w8 % 16 || (uintptr_t)y % 16 || (uintptr_t)scratch % 16)
    return fail(HE_ERR_ARG, "buffers not 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  GemmArgs a{};
  a.dtype = HE_DTYPE_BF16;
  a.act = ACT_F16;
  a.ldx = K;
  a.w[0] = w8;
  a.w_scale[0] = scale;
  a.w_fp8 = 1;
  a.w_tiled = 1;
  a.n_groups = 1;
  a.group_rows = N;
  a.M = M;
  a.N = N;
  a.K = K;
  a.split = 1;
  Epi e{};
  e.kind = EPI_STORE_F32;
  e.partial = y;
  e.ldp = N;
  a.epi = e;
  const long long T = N / 128, U = sk_units(a);
  int P = sk_ctas(a, sms, true);
  if (split < 0) {
    if (-split > U || -split > 15 * T)
      return fail(HE_ERR_ARG, "stream-K CTA count %d above min(units, 15 * tiles)", -split);
    P = -split;
  }
  const int R = sk_token_tile(M);
  const long long sstride = (long long)M * N;
  void *xt = scratch + (size_t)16 * sstride;
  int *cnt = reinterpret_cast<int *>(((uintptr_t)xt + (size_t)R * K * 2 + 15) & ~(uintptr_t)15);
  a.x = xt;
  cudaError_t r = launch_tile_act(x, M, K, ldx, R, xt, st);
  if (r == cudaSuccess) r = cudaMemsetAsync(cnt, 0, (size_t)T * sizeof(int), st);
  if (r == cudaSuccess) r = launch_gemm_sk(a, P, scratch, sstride, cnt, nullptr, st);
  if (r != cudaSuccess) return cuda_fail(r, "he_op_linear_fp8");
  return HE_OK;
}

he_status he_op_linear(int dtype, const void *x, int ldx, const void *w, int w_layout, float *y,
                       int M, int N, int K, int split, float *scratch, void *stream) {
  g_err.clear();
  if (w_layout != 0 && w_layout != 1) return fail(HE_ERR_ARG, "w_layout must be 0 or 1");
  if (w_layout == 1 && (dtype == HE_DTYPE_F32 || N % 128 || K % 64))
    return fail(HE_ERR_UNSUPPORTED, "tiled weights need a 16-bit type, N %% 128 == 0, K %% 64 == 0");
  if (!x || !w || !y) return fail(HE_ERR_ARG, "NULL buffer");
  if (M < 1 || N < 1 || K < 1 || ldx < K) return fail(HE_ERR_ARG, "bad sizes");
  if (dtype != HE_DTYPE_F32 && dtype != HE_DTYPE_BF16 && dtype != HE_DTYPE_F16)
    return fail(HE_ERR_ARG, "bad dtype");
  if (dtype != HE_DTYPE_F32 && (K % 8 || ldx % 8))
    return fail(HE_ERR_UNSUPPORTED, "16-bit types need K and ldx multiples of 8");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (split <= 0) {
    // stream-K: the persistent kernel of the decode projections
    if (dtype == HE_DTYPE_F32 || M > 256 || K % 64 || (w_layout == 1 && N % 128))
      return fail(HE_ERR_UNSUPPORTED, "stream-K needs a 16-bit type, M <= 256, K %% 64 == 0 (and N %% 128 == 0 for tiled weights)");
    if (!scratch) return fail(HE_ERR_ARG, "stream-K needs scratch");
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    GemmArgs a{};
    a.dtype = HE_DTYPE_BF16;
    a.act = dtype;
    a.x = x;
    a.ldx = ldx;
    a.w[0] = w;
    a.n_groups = 1;
    a.group_rows = N;
    a.M = M;
    a.N = N;
    a.K = K;
    a.split = 1;
    a.w_tiled = w_layout;
    Epi e{};
    e.kind = EPI_STORE_F32;
    e.partial = y;
    e.ldp = N;
    a.epi = e;
    const bool fix = sk_fixup_ok(a);
    int P = sk_ctas(a, sms, fix);
    const long long T = (N + 127) / 128, U = sk_units(a);
    if (split < 0) {
      if (-split > U || -split > 15 * T)
        return fail(HE_ERR_ARG, "stream-K CTA count %d above min(units, 15 * tiles)", -split);
      P = -split;
    }
    // the stream-K kernel reads row-tiled activations: tile x behind the slices
    // (16 per tile, tile-contiguous over whole 128-wide tiles), then the tile counters
    const int R = sk_token_tile(M);
    const long long sstride = (long long)M * T * 128;
    void *xt = scratch + (size_t)16 * sstride;
    int *cnt = reinterpret_cast<int *>(
        ((uintptr_t)xt + (size_t)R * K * 2 + 15) & ~(uintptr_t)15);
    a.x = xt;
    cudaError_t r = launch_tile_act(x, M, K, ldx, R, xt, st);
    const SliceInfo si{0, U, (int)(U / T), P};
    if (r == cudaSuccess && fix) r = cudaMemsetAsync(cnt, 0, (size_t)T * sizeof(int), st);
    if (r == cudaSuccess)
      r = launch_gemm_sk(a, P, scratch, fix ? sstride : (long long)M * N, fix ? cnt : nullptr,
                         nullptr, st);
    if (r == cudaSuccess && !fix)
      r = launch_sk_reduce_epi(HE_DTYPE_BF16, dtype, scratch, si, (long long)M * N, N, M, N, e, st);
    if (r != cudaSuccess) return cuda_fail(r, "he_op_linear (stream-K)");
    return HE_OK;
  }
  if (effective_split(K, split) != split)
    return fail(HE_ERR_ARG, "split %d leaves an empty K slice (K=%d)", split, K);
  if (split > 1 && !scratch) return fail(HE_ERR_ARG, "split > 1 needs scratch");
  GemmArgs a{};
  a.dtype = dtype == HE_DTYPE_F32 ? HE_DTYPE_F32 : HE_DTYPE_BF16;
  a.act = dtype;
  a.x = x;
  a.ldx = ldx;
  a.w[0] = w;
  a.n_groups = 1;
  a.group_rows = N;
  a.M = M;
  a.N = N;
  a.K = K;
  a.split = split;
  a.w_tiled = w_layout;
  Epi e{};
  e.kind = EPI_STORE_F32;
  e.partial = y;
  e.ldp = N;
  if (split > 1) {
    Epi pe{};
    pe.kind = EPI_PARTIAL;
    pe.partial = scratch;
    pe.ldp = N;
    pe.split_stride = (long long)M * N;
    a.epi = pe;
  } else {
    a.epi = e;
  }
  cudaError_t r = launch_gemm(a, nullptr, st);
  if (r == cudaSuccess && split > 1)
    r = launch_reduce_epi(dtype == HE_DTYPE_F32 ? HE_DTYPE_F32 : HE_DTYPE_BF16, dtype, scratch, split,
                          (long long)M * N, N, M, N, e, st);
  if (r != cudaSuccess) return cuda_fail(r, "he_op_linear");
  return HE_OK;
}

}  // extern "C"
