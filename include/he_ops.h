/*
 * he_ops.h -- kernel-level entry points of libhe, for testing the kernels that
 * he_generate runs on shapes of the caller's choosing.
 */
#ifndef HE_OPS_H
#define HE_OPS_H

#include "he.h"

#ifdef __cplusplus
extern "C" {
#endif

/* y[M][N] (fp32, row-major) = x[M][K] w[N][K]^T: the projection y = x W^T of
 * every linear layer of the model ("DeepSpeed-Chat: Easy, Fast and Affordable
 * RLHF Training of ChatGPT-like Models at All Scales", §3.4 "Inference Mode:
 * Generation Phase Optimizations", Optimization 1: each generation step
 * multiplies the current tokens' activations with every weight matrix).
 * dtype HE_DTYPE_BF16 runs the tcgen05 tensor-core kernel (K and ldx multiples
 * of 8, x and w 16-byte aligned); HE_DTYPE_F32 runs the fp32 CUDA-core kernel.
 * x has row stride ldx >= K; w is dense [N][K] (w_layout 0) or in the tiled
 * streaming layout below (w_layout 1, bf16 only).  split >= 1 splits K into
 * slices of whole 64-wide blocks (no empty slice allowed) whose fp32 partial
 * sums go to scratch [split][M][N] and are then added in slice order.
 * split <= 0 runs the persistent stream-K kernel of the decode projections
 * (bf16, M <= 256, K % 64 == 0, N % 128 == 0 with tiled weights): the
 * (128-row tile, k-block) units are cut into P equal runs, P = -split if
 * split < 0 (at most min(units, 15 * tiles)), else the engine's choice (one per
 * SM).  A tile split over several runs is finished inside the kernel by the run
 * holding its first k-blocks, which adds the others' fp32 slices in slot order
 * and stores y (N % 4 == 0 and y 16-byte aligned; otherwise a second kernel adds
 * the slices).  scratch needs 16 * M * Np floats (Np = N rounded up to a
 * multiple of 128) for the slices, then R * K bf16 (R = M rounded up to 16, 32,
 * 64, 128 or 256) for the row-tiled copy of x that the kernel reads, then, from
 * the next 16-byte boundary, Np / 128 ints of per-tile counters that the op
 * clears itself before the kernel.
 * All pointers are device memory; asynchronous on `stream`. */
he_status he_op_linear(int dtype, const void *x, int ldx, const void *w, int w_layout, float *y,
                       int M, int N, int K, int split, float *scratch, void *stream);

/* Greedy choice fused into the LM-head GEMM, as the decode steps run it when they
 * neither sample, force tokens nor capture logits ("DeepSpeed-Chat: Easy, Fast and
 * Affordable RLHF Training of ChatGPT-like Models at All Scales", §3.4 "Inference
 * Mode: Generation Phase Optimizations", Optimization 1: fused kernels cut the
 * intermediate reads and writes; "Chapter 11 System Architecture & Infrastructure
 * at Scale", "The Generation Bottleneck": generation returns the log-probabilities
 * of the chosen tokens).  For the logits l = x w^T (x [M][K] with row stride ldx,
 * w [N][K] dense, both dtype BF16 or F16, fp32 accumulation): out_ids[m] = the
 * lowest n with l[m][n] = max_n l[m][n], and out_lp[m] = log softmax of that
 * logit, computed without storing the logits: the stream-K kernel's epilogue
 * reduces each 128-row tile of w to {max, sum of exp(l - max), argmax} per row of
 * x, and a second kernel merges the tiles.  Needs 1 <= M <= 256, K % 64 == 0,
 * ldx >= K, ldx % 8 == 0, N % 4 == 0, 16-byte aligned buffers.  scratch: 16 * M *
 * Np floats (Np = N rounded up to 128) for split-tile slices, then R * K 16-bit
 * values (R = M rounded up to 16, 32, 64, 128 or 256) for the row-tiled copy of x,
 * then from the next 16-byte boundary Np / 128 ints of tile counters, then from
 * the next 16-byte boundary Np / 128 * M float4 of tile statistics.  Device
 * pointers; asynchronous on `stream`. */
he_status he_op_head_greedy(int dtype, const void *x, int ldx, const void *w, int M, int N, int K,
                            int32_t *out_ids, float *out_lp, float *scratch, void *stream);

/* The streaming layout he_fuse_lora writes the bf16 projections in while LoRA
 * is fused ("DeepSpeed-Chat: Easy, Fast and Affordable RLHF Training of
 * ChatGPT-like Models at All Scales", §3.4 "Inference Mode: Generation Phase
 * Optimizations", Optimization 1: the inference kernels lay weights out for
 * bandwidth).  w_layout 1 in he_op_linear means w holds this layout.  For a
 * bf16 W [N][K] with N % 128 == 0 and K % 64 == 0, element (n, k) sits at index
 *   ((n / 128) * (K / 64) + k / 64) * 8192 + (n % 128) * 64
 *     + (((k % 64) / 8) ^ (n % 8)) * 8 + k % 8,
 * i.e. 128 x 64 tiles stored contiguously, k-tiles of a tile row consecutive,
 * each tile in the 128-byte-swizzled order the tensor cores read, so one bulk
 * copy moves a whole tile.  he_op_tile_weight writes out (N*K elements, no
 * overlap with w) from the row-major w; asynchronous on `stream`. */
he_status he_op_tile_weight(const void *w, void *out, int N, int K, void *stream);

/* One projection of he_fuse_lora on a BF16 engine ("DeepSpeed-Chat 选型指南", §三:
 * the LoRA weights are fused into the inference model before generation; "DeepSpeed-
 * Chat: Easy, Fast and Affordable RLHF Training of ChatGPT-like Models at All
 * Scales", §3.4 "Training Mode: ZeRO and LoRA Optimizations", Optimization 2):
 * out = W + scale * B A (fp32 arithmetic, one rounding to fp16) in the tiled
 * streaming layout above (fp16 elements).  w: bf16 [N][K] (N % 128 == 0, K % 64 ==
 * 0); lora_a: bf16 [r][K], lora_b: bf16 [N][r] (r = 0: no delta, w converted to
 * fp16; 0 <= r <= 64).  For r = 8 or 16 with 16-byte-aligned factors the product B A
 * runs on the tensor cores (exact products, fp32 sums), otherwise as fp32 fused
 * multiply-adds in j order.  For tests and profiling.  Asynchronous on `stream`. */
he_status he_op_fuse_tiled(const void *w, const void *lora_a, const void *lora_b, int r, float scale,
                           void *out, int N, int K, void *stream);

/* The fp8 tiled layout (he_set_weight_format HE_WEIGHTS_FP8): for W [N][K] with
 * N % 128 == 0 and K % 128 == 0, the one-byte code of element (n, k) sits at
 *   ((n / 128) * (K / 128) + k / 128) * 16384 + (n % 128) * 128
 *     + (((k % 128) / 16) ^ (n % 8)) * 16 + k % 16,
 * 128 x 128 tiles of 16 KB, each a single bulk copy of a decode GEMM stage.
 * y[M][N] (fp32) = (x[M][K] codes^T) * scale[n]: the stream-K decode GEMM on fp8
 * weights (codes in that layout, fp32 scales per row) and fp16 activations x
 * (row stride ldx; 1 <= M <= 128, K % 256 == 0, ldx >= K, ldx % 8 == 0,
 * 16-byte aligned).
 * split < 0 runs on -split CTAs (at most min(units, 15 * tiles)), otherwise one
 * per SM.  scratch: as he_op_linear's stream-K scratch (16 * M * N floats of
 * slices, then R * K fp16 of row-tiled x, then N / 128 counters).  Asynchronous
 * on `stream`. */
he_status he_op_linear_fp8(const void *x, int ldx, const void *w8, const float *scale, float *y,
                           int M, int N, int K, int split, float *scratch, void *stream);

/* Causal attention of the prompt pass: every prompt token attends to the prompt's
 * tokens up to itself ("DeepSpeed-Chat: Easy, Fast and Affordable RLHF Training
 * of ChatGPT-like Models at All Scales", §3.4 "Step 3: RLHF Training via PPO",
 * item 1: the actor first reads the whole 256-token prompt, then generates; the
 * prompt pass fills the key/value cache of §3.4 "Inference Mode", Optimization 2).
 * q: [B][Lp][H*hd] (already scaled by hd^-1/2); kc, vc: [B][H][max_seq][hd], the
 * prompt's keys and values at positions 0..Lp-1 (later positions are not read);
 * ctx: [B][Lp][H*hd] out.  dtype F32, BF16 or F16; hd in {32, 64, 128}; fp32
 * softmax and accumulation.  BF16 / F16 with hd 64 or 128 run on the tcgen05
 * tensor cores (the probabilities rounded to dtype for the P V product), unless
 * flags has HE_ATTN_PREFILL_MMA_SYNC, which selects the mma.sync kernel (also used
 * for hd 32).  All four pointers 16-byte aligned, Lp <= max_seq, else HE_ERR_ARG.
 * dev_flags: device int that receives DEVERR bits (a bounded pipeline wait that
 * ran out: the output is then not valid), or NULL.  Asynchronous on `stream`. */
enum { HE_ATTN_PREFILL_MMA_SYNC = 1 };
he_status he_op_attn_prefill(int dtype, const void *q, const void *kc, const void *vc, void *ctx,
                             int B, int Lp, int H, int hd, int max_seq, int flags, int *dev_flags,
                             void *stream);

/* Single-query attention of one decode step over the KV cache
 * ("DeepSpeed-Chat: Easy, Fast and Affordable RLHF Training of ChatGPT-like
 * Models at All Scales", §3.4 "Inference Mode: Generation Phase Optimizations",
 * Optimizations 1 and 2: attention specialised for one new query against a
 * long cached context, keys and values read from the cache).
 * q: [B][H*hd] (already scaled by hd^-1/2); kc, vc: [B][H][max_seq][hd];
 * ctx: [B][H*hd] row-major out; keys/values 0..n_keys-1 are used.  split >= 1
 * cuts the keys of each (b, h) into that many slices merged afterwards (part:
 * B*H*split*(hd+2) floats when split > 1).  dtype F32, BF16 or F16 (fp32 softmax
 * and accumulation in every case); hd in {32, 64, 128}.  Asynchronous on
 * `stream`. */
he_status he_op_attn_decode(int dtype, const void *q, const void *kc, const void *vc, void *ctx,
                            int B, int H, int hd, int max_seq, int n_keys, int split, float *part,
                            void *stream);

/* he_op_attn_decode for callers that cannot allocate device memory.  The pages
 * have no counterpart: this is a convenience of this library.  Runtimes whose
 * device memory belongs to a pooling allocator or a fixed budget cannot hand out
 * an extra buffer on demand, plugins hosted by another framework may have no
 * allocator of their own, and latency-bound loops avoid cudaMalloc because it may
 * synchronise the device; such callers pass only inputs and outputs here.  Same
 * arguments and results as he_op_attn_decode (dtype F32, BF16 or F16), except
 * that the split-over-keys partial results live in a 16 MiB array built into the
 * library (4194304 floats, held on every GPU that loads it until the process
 * exits): B * H * split * (hd + 2) must not exceed 4194304 when split > 1, else
 * HE_ERR_ARG.  It calls no allocator.  The first call on a device (and the first
 * after that device's context changes, e.g. after cudaDeviceReset) looks up the
 * array's device address with that device current (host-side set-up); make that
 * first call before any stream capture.  Every call shares the one array, so
 * calls whose work overlaps on the GPU (other streams, other threads) race and
 * must be ordered by the caller; a call writes every partial it reads before
 * reading it, so nothing needs to start at zero. */
he_status he_op_attn_decode_noalloc(int dtype, const void *q, const void *kc, const void *vc,
                                    void *ctx, int B, int H, int hd, int max_seq, int n_keys,
                                    int split, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* HE_OPS_H */
