/*
 * he.h -- Hybrid-Engine experience generation for an OPT-style actor on one GPU.
 *
 * C ABI of libhe.so.  Plain pointers and sizes only.  All device pointers are
 * CUDA device addresses on the engine's device; every call that takes a
 * `stream` (a cudaStream_t passed as void*, NULL = legacy default stream)
 * enqueues its work on it and returns before the work finishes unless stated.
 *
 * The operations follow these passages:
 *  [DSC-gen]  "DeepSpeed-Chat: Easy, Fast and Affordable RLHF Training of
 *             ChatGPT-like Models at All Scales" (paper summary), §3.4, "Step 3:
 *             RLHF Training via PPO", item 1: the actor generates 256-token
 *             answers to 256-token prompts token by token; the phase is bound by
 *             memory bandwidth.
 *  [DSC-kv]   same page, §3.4 "Inference Mode: Generation Phase Optimizations",
 *             Optimization 2: keys and values of earlier tokens are cached,
 *             appended each step and reused; buffers are reused across steps.
 *  [DSC-lora] same page, §3.4 "Training Mode: ZeRO and LoRA Optimizations",
 *             Optimization 2: a weight W is used as W + B A (B: d x r, A: r x k).
 *  [DSC-he]   same page, §3.4 "The DeepSpeed Hybrid Engine: Architecture and
 *             Mode Switching": one model instance; at the inference/training
 *             switch the engine allocates or frees the KV-cache buffers.
 *  [HE-guide] "DeepSpeed-Chat 选型指南：Hybrid Engine 驱动的 RLHF 训练全解析",
 *             §三 (engine internals): generate() fuses LoRA into the inference
 *             model before generation and restores it after; the KV cache and
 *             intermediate results live in a workspace that is released after
 *             generation and retaken before the next; §四 (config fields):
 *             max_out_tokens, release_inference_cache, enable_cuda_graph.
 *  [RLHF-ch11] "Chapter 11 System Architecture & Infrastructure at Scale",
 *             "The Generation Bottleneck: Quantitative Analysis": generation
 *             returns the log-probabilities of the generated tokens.
 *
 * Model (OPT-style pre-LN decoder; the pages name the OPT family but not its
 * layer details, which are taken as OPT defines them): x = E_tok[id] +
 * E_pos[t + pos_offset]; per layer h = LN1(x); q = (h Wq^T + bq) hd^-1/2,
 * k = h Wk^T + bk, v = h Wv^T + bv; causal softmax attention per head;
 * x += ctx Wo^T + bo; x += ReLU(LN2(x) W1^T + b1) W2^T + b2; logits =
 * LN_f(x) E_tok^T (tied head, no bias).  LayerNorm: biased variance, eps
 * inside the square root.  Greedy choice: argmax, lowest index on ties.
 *
 * Errors: every call returns an he_status.  Argument and state errors are
 * found on the host before anything is enqueued and leave the engine as it
 * was.  he_last_error() gives a message for the last failing call on the
 * calling thread.  Nothing throws across this ABI.
 */
#ifndef HE_H
#define HE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct he_engine he_engine; /* opaque, owned by the library */

typedef enum {
  HE_OK = 0,
  HE_ERR_ARG = -1,          /* bad argument (NULL, out of range, inconsistent size) */
  HE_ERR_STATE = -2,        /* call not allowed in the engine's current state */
  HE_ERR_OOM = -3,          /* the allocator returned NULL */
  HE_ERR_CUDA = -4,         /* a CUDA runtime/driver call or launch failed */
  HE_ERR_UNSUPPORTED = -5,  /* shape or dtype outside what the kernels handle */
  HE_ERR_DEVICE_CHECK = -6  /* a device-side input check failed (e.g. token id >= vocab) */
} he_status;

/* Element types.  he_config.dtype takes F32 or BF16; the kernel-level entries of
 * he_ops.h also take F16. */
enum { HE_DTYPE_F32 = 0, HE_DTYPE_BF16 = 1, HE_DTYPE_F16 = 2 };

/* Bit i of he_config.lora_targets: projection i carries a LoRA pair. */
enum {
  HE_PROJ_Q = 0, HE_PROJ_K = 1, HE_PROJ_V = 2, HE_PROJ_O = 3, HE_PROJ_FC1 = 4, HE_PROJ_FC2 = 5,
  HE_N_PROJ = 6
};

typedef struct {
  int n_layers, d_model, n_heads, ffn, vocab;
  int max_pos;      /* usable positions; E_pos has max_pos + pos_offset rows */
  int pos_offset;   /* 2 for OPT's learned positions */
  int dtype;        /* HE_DTYPE_F32 or HE_DTYPE_BF16: storage type of every parameter.
                       F32: fp32 CUDA-core kernels throughout.  BF16: tensor cores with
                       fp32 accumulation on fp16 operands: generation reads the
                       projections as fp16 (merged while LoRA is fused, see
                       he_fuse_lora; the caller's weights converted at the start of
                       each generation otherwise, see he_generate), and activations
                       and the KV cache are fp16.  The residual stream, LayerNorm,
                       softmax, logits and log-probs are fp32; the tied LM head reads
                       the bf16 embedding. */
  float ln_eps;     /* 1e-5 for OPT */
  int max_batch;    /* workspace sizing: every he_generate has B <= max_batch */
  int max_seq;      /* workspace sizing: Lp + Lgen <= max_seq (the KV cache length);
                       the role of the hybrid_engine max_out_tokens field */
  int lora_r;       /* LoRA rank r (1..64) */
  float lora_alpha; /* the fused delta is (lora_alpha / lora_r) * B A */
  unsigned lora_targets; /* bit mask over HE_PROJ_*; 0 = no LoRA */
} he_config;

/* One decoder layer.  Projections are [out][in] row-major (y = x W^T + b):
 * Wq, Wk, Wv, Wo: [d][d]; W1: [ffn][d]; W2: [d][ffn].  All tensors have the
 * config's dtype and are caller-owned device memory that must stay valid until
 * he_destroy.  F32 engines write w[] in place in he_fuse_lora / he_unfuse_lora;
 * BF16 engines never write it. */
typedef struct {
  void *w[HE_N_PROJ];            /* indexed by HE_PROJ_* */
  const void *b[HE_N_PROJ];      /* biases [out] */
  const void *ln1_g, *ln1_b, *ln2_g, *ln2_b; /* [d] */
  const void *lora_a[HE_N_PROJ]; /* A: [r][in]  (NULL where the target bit is clear) */
  const void *lora_b[HE_N_PROJ]; /* B: [out][r] */
} he_layer_weights;

typedef struct {
  const void *tok_emb;   /* [vocab][d]; also the tied LM head */
  const void *pos_emb;   /* [max_pos + pos_offset][d] */
  const void *lnf_g, *lnf_b; /* final LayerNorm [d] */
  const he_layer_weights *layers; /* host array of n_layers; copied by he_create */
} he_weights;

/* Device-memory allocator the engine uses for its workspace, its KV cache and
 * the LoRA restore copy, so that released memory goes back to the caller (for
 * example to a framework's caching allocator for the training phase).
 * alloc returns a device pointer aligned to >= 256 bytes or NULL; free gets the
 * same size.  `stream` is the stream the memory will be used on. */
typedef struct {
  void *(*alloc)(size_t bytes, void *stream, void *ctx);
  void (*free)(void *ptr, size_t bytes, void *stream, void *ctx);
  void *ctx;
} he_allocator;

typedef struct {
  double fuse_ms, prefill_ms, decode_ms, unfuse_ms; /* last call of each, device time */
  long long launches;            /* kernels launched by the library since he_create */
  long long generate_calls;
  size_t workspace_bytes;        /* KV cache + scratch currently held */
  size_t kv_bytes;               /* KV cache part of it */
  size_t restore_bytes;          /* held by he_fuse_lora (restore copy or fused buffer) */
  /* Per-kernel-class device time of the last he_generate, filled only while
   * profiling is on (he_set_profiling); index by HE_KCLASS_*. */
  double kclass_ms[8];
  long long kclass_launches[8];
} he_stats;

enum {
  HE_KCLASS_GEMM = 0,        /* decode projections (QKV, out, fc1, fc2) */
  HE_KCLASS_ATTN_DECODE = 1, /* decode single-query attention (+ its combine) */
  HE_KCLASS_NORM = 2,        /* residual + LayerNorm rows, split reductions */
  HE_KCLASS_HEAD = 3,        /* LM head GEMM + greedy select / log-prob / next embed */
  HE_KCLASS_PREFILL_GEMM = 4,
  HE_KCLASS_PREFILL_ATTN = 5,
  HE_KCLASS_OTHER = 6
};

/* Creates an engine on `device` (the CUDA ordinal; it becomes current for the
 * calling thread).  Checks the config (d_model % n_heads == 0, head_dim in
 * {32, 64, 128}; BF16 also needs d_model, ffn multiples of 128, vocab % 8 == 0),
 * records the weight pointers (no copy: one model instance, [DSC-he]) and takes
 * the workspace (KV cache [n_layers][max_batch][n_heads][max_seq][head_dim] for
 * K and for V, plus activations) through `alloc`.  alloc == NULL uses cudaMalloc /
 * cudaFree.  On failure *out is NULL and nothing is held. */
he_status he_create(const he_config *cfg, const he_weights *w, const he_allocator *alloc,
                    int device, he_engine **out);

/* Frees everything the engine holds (restoring fused weights first is the
 * caller's job: destroying a fused F32 engine leaves its weights fused).  NULL is
 * a no-op. */
he_status he_destroy(he_engine *h);

/* [DSC-lora], [HE-guide]: the merged weight W + (alpha/r) * B A (fp32
 * arithmetic) for generation.  F32: saves the bits of the targeted projections,
 * then writes the merged weight in place (round to nearest).  BF16: all six
 * projections of every layer, merged where LoRA-targeted, are written as fp16
 * (round to nearest even; the pages' hybrid-engine test config runs with
 * fp16.enabled) in the tiled streaming layout of he_ops.h into a buffer of the
 * same size as those projections, taken through the allocator; w[] is not
 * written, and generation reads that buffer while fused.  HE_ERR_STATE if
 * already fused; HE_ERR_OOM (from the allocator) leaves the engine unfused and
 * the weights untouched. */
he_status he_fuse_lora(he_engine *h, void *stream);

/* F32: restores the saved bits of every targeted projection (bit-exact).  Both
 * dtypes: frees the buffer he_fuse_lora took.  HE_ERR_STATE if not fused. */
he_status he_unfuse_lora(he_engine *h, void *stream);

/* Weight formats of he_set_weight_format. */
enum { HE_WEIGHTS_F16 = 0, HE_WEIGHTS_FP8 = 1 };

/* [RLHF-ch11] "The Generation Bottleneck: Quantitative Analysis" (the optimisation
 * stack: INT8/FP8 weights for generation halve the bandwidth the weights need):
 * the format generation reads the six projections in, from the next he_fuse_lora
 * (or the next unfused generation) on.  HE_WEIGHTS_F16 (the default): fp16, as
 * described at he_fuse_lora.  HE_WEIGHTS_FP8 (BF16 engines): each projection,
 * after the LoRA merge, is stored as OCP FP8 E4M3 codes with one fp32 scale per
 * output row, s_n = max_k |W[n][k]| / 448, codes = W / s_n rounded to the nearest
 * E4M3 value (ties to even, saturated at 448); generation computes with the
 * weights codes * s_n.  The decode projections stream the one-byte codes (half
 * the weight bytes), decoded exactly to fp16 on the chip, with fp16 activations
 * and fp32 accumulation; the prefill GEMMs read the same codes as fp16 values.  The
 * tied LM head, the KV cache and the activations are unchanged.  The copy takes
 * 3 bytes per projection weight plus 4 per row (the fp16 copy: 2).  HE_ERR_STATE
 * while fused; HE_ERR_UNSUPPORTED for FP8 on an F32 engine. */
he_status he_set_weight_format(he_engine *h, int format);

/* With HE_WEIGHTS_FP8 fused: copies projection `proj` of `layer`'s E4M3 codes (device
 * `codes`, rows * cols bytes in the fp8 tiled layout of he_ops.h) and its fp32 row
 * scales (device `scales`, rows floats).  For tests and inspection.  HE_ERR_STATE if
 * not fused with fp8 weights.  Asynchronous on `stream`. */
he_status he_read_fused_fp8(he_engine *h, int layer, int proj, void *codes, size_t code_bytes,
                            float *scales, void *stream);

/* Copies projection `proj` of `layer` as generation reads it while fused into
 * dst (device, `bytes` = rows * cols * element size of the config's dtype): the
 * merged weight in place for F32, the fp16 tiled copy for BF16 (element layout
 * of he_op_tile_weight, 2-byte elements).  For tests and inspection.
 * HE_ERR_STATE if not fused, HE_ERR_ARG for a bad layer, projection or size.
 * Asynchronous on `stream`. */
he_status he_read_fused_weight(he_engine *h, int layer, int proj, void *dst, size_t bytes,
                               void *stream);

/* [DSC-gen], [DSC-kv], [RLHF-ch11]: greedy generation of Lgen tokens for B
 * prompts of Lp tokens.  prompt_ids: device int32 [B][Lp], every id in
 * [0, vocab).  out_ids: device int32 [B][Lgen]; out_logprob: device fp32
 * [B][Lgen], natural-log softmax of the chosen token.  One prefill pass over the
 * prompts, then Lgen - 1 single-token passes over the KV cache; the last token
 * is not fed back.  Requires 1 <= B <= max_batch, Lp >= 1, Lgen >= 1,
 * Lp + Lgen <= max_seq, Lp + Lgen - 1 <= max_pos, and a taken workspace
 * (HE_ERR_STATE after he_release_workspace).  Runs fused or unfused.  Unfused
 * on a BF16 engine, every generation first converts the caller's bf16
 * projections to fp16 in the tiled layout (one pass over the weights, in the
 * same stream), into a buffer of that size taken through the allocator on the
 * first unfused call and held with the workspace (he_release_workspace and
 * he_fuse_lora give it back); HE_ERR_OOM if it cannot be taken.  The weights may
 * change between calls.  An id out of range is replaced by 0 on the device and
 * reported by he_check. */
he_status he_generate(he_engine *h, const int32_t *prompt_ids, int B, int Lp, int Lgen,
                      int32_t *out_ids, float *out_logprob, void *stream);

/* he_generate with teacher forcing and logit capture (parity checks):
 * force_ids: device int32 [B][Lgen] or NULL; where force_ids[b][k] >= 0 step k
 * emits and feeds back that id (its log-prob is reported) instead of the argmax.
 * log_rows: HOST int32 pairs (b, k), n_rows of them; the fp32 logits of sequence
 * b at step k are written to logits_out[i][0..vocab) (device, [n_rows][vocab]).
 * n_rows may be 0 (then log_rows and logits_out may be NULL). */
he_status he_generate_ex(he_engine *h, const int32_t *prompt_ids, int B, int Lp, int Lgen,
                         int32_t *out_ids, float *out_logprob, const int32_t *force_ids,
                         const int32_t *log_rows, int n_rows, float *logits_out,
                         void *stream);

/* he_generate on HOST buffers: copies prompt_ids [B][Lp] in, generates, copies
 * out_ids / out_logprob [B][Lgen] back and synchronises `stream` before it
 * returns.  Also returns HE_ERR_DEVICE_CHECK if a prompt id was out of range. */
he_status he_generate_host(he_engine *h, const int32_t *prompt_ids, int B, int Lp, int Lgen,
                           int32_t *out_ids, float *out_logprob, void *stream);

/* Synchronises `stream` and reports (then clears) the device-side input check:
 * HE_ERR_DEVICE_CHECK if an id was out of range since the last check. */
he_status he_check(he_engine *h, void *stream);

/* [HE-guide] release_inference_cache: hands the KV cache and activation
 * workspace (and an unfused BF16 engine's fp16 copy of the projections) back to
 * the allocator (stream-ordered on `stream`).  The LoRA restore copy is kept
 * while fused.  HE_ERR_STATE if already released. */
he_status he_release_workspace(he_engine *h, void *stream);

/* Takes the workspace again before the next generation.  HE_ERR_STATE if held;
 * HE_ERR_OOM leaves the engine released and usable (retry later). */
he_status he_retake_workspace(he_engine *h, void *stream);

/* [DSC-gen] item 2 (the training phase consumes the log-probabilities of the
 * generated responses under the reference model) and [RLHF-ch11] (log-probs of
 * every generated token are needed for PPO): the log-probability of each answer
 * token under this model, computed in one forward pass over prompt + answer
 * rather than token by token.  ids: device
 * int32 [B][L], a prompt of Lp tokens followed by L - Lp answer tokens, every id
 * in [0, vocab).  out_logprob: device fp32 [B][L - Lp]; element (b, k) is the
 * natural-log softmax at position Lp - 1 + k of token ids[b][Lp + k], i.e. what
 * he_generate_ex reports when teacher-forced on the same answer.  One pass of the
 * prefill kernels over tokens 0 .. L-2 (filling the KV cache), then the head on
 * rows Lp - 1 .. L - 2.  Requires 1 <= B <= max_batch, 1 <= Lp < L <= max_seq,
 * L - 1 <= max_pos and a taken workspace.  Runs fused or unfused; an id out of
 * range is replaced by 0 on the device and reported by he_check. */
he_status he_score(he_engine *h, const int32_t *ids, int B, int L, int Lp, float *out_logprob,
                   void *stream);

/* [RLHF-ch11] (the production generation setup there samples with a temperature
 * and a nucleus cut-off and returns the log-probs PPO needs): sampled instead of
 * greedy generation for the following he_generate* calls.  temperature 0 (the
 * default) is greedy.  Otherwise, per sequence b and step k, with q_i =
 * exp((l_i - max l) / temperature): the nucleus is every token with q_i >= tau,
 * tau the largest value for which those tokens hold at least top_p of the sum of
 * q (so ties at the boundary are in); the token is the argmax over the nucleus of
 * (l_i - max l) / temperature - log(-log u_i), lowest index on ties, u_i in (0, 1)
 * from SplitMix64 output number c + 1 started at `seed`, c = (b * 2^20 + k) * 2^20
 * + i, u = (2 (z >> 41) + 1) / 2^24.  The reported log-prob (and he_score's) is
 * log softmax(l / temperature) of the emitted token over the whole vocabulary.
 * temperature >= 0 and finite, 0 < top_p <= 1, else HE_ERR_ARG. */
he_status he_set_sampling(he_engine *h, float temperature, float top_p,
                          unsigned long long seed);

/* [HE-guide] enable_cuda_graph (§三 and the §四 field table: a CUDA-graph cache
 * for generation to cut launch overhead; off by default there and here).  With
 * enable != 0, he_generate and he_generate_host run the generation as one CUDA
 * graph, captured on first use and replayed afterwards; it is re-captured when
 * B, Lp, Lgen, fused / unfused, or the address of a workspace buffer changes
 * (e.g. after he_release_workspace / he_retake_workspace).  The kernels and their
 * order are those of the direct launch, so the results are identical.
 * he_generate_ex with teacher forcing or logit capture, and any generation with
 * profiling on, launch directly.  enable == 0 frees the cached graph. */
he_status he_set_cuda_graph(he_engine *h, int enable);

/* Per-kernel-class event timing of he_generate: class_mask has bit c set for
 * every HE_KCLASS_c to time (0 = off, the default).  Costs two events per
 * timed launch; the totals of the last he_generate appear in he_stats. */
he_status he_set_profiling(he_engine *h, unsigned class_mask);

/* Fills *s.  Synchronises the engine's events from the last calls first. */
he_status he_get_stats(he_engine *h, he_stats *s);

/* Message of the last failing call on this thread ("" if none). */
const char *he_last_error(void);

/* Library build identifier (static string). */
const char *he_version(void);

#ifdef __cplusplus
}
#endif

#endif /* HE_H */
