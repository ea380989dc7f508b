// Internal launcher interface between the engine (engine.cu) and the kernels.
// Host-side declarations only; no torch types, no exceptions.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

namespace he {

// Activation / operand types (values 0 and 1 double as the parameter dtype).
enum ActType : int { ACT_F32 = 0, ACT_BF16 = 1, ACT_F16 = 2 };

// Host dispatch over the (parameter type PT, activation type CT) pairs the
// library runs: (float, float), (bf16, bf16) and (bf16, fp16).
#define HE_DISPATCH_PT_CT(pt, ct, ...)                        \
  do {                                                        \
    if ((pt) == 0 && (ct) == ACT_F32) {                       \
      using PT = float;                                       \
      using CT = float;                                       \
      __VA_ARGS__                                             \
    } else if ((pt) == 1 && (ct) == ACT_BF16) {               \
      using PT = __nv_bfloat16;                               \
      using CT = __nv_bfloat16;                               \
      __VA_ARGS__                                             \
    } else if ((pt) == 1 && (ct) == ACT_F16) {                \
      using PT = __nv_bfloat16;                               \
      using CT = __half;                                      \
      __VA_ARGS__                                             \
    } else {                                                  \
      return cudaErrorInvalidValue;                           \
    }                                                         \
  } while (0)

// Launch with programmatic stream serialisation (see pdl_wait in common.cuh) when
// `pdl` is set; every kernel launched this way waits before its dependent reads
// and writes.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t st, bool pdl, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (pdl) {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// launch_k for clusters of two CTAs along x (grid.x even).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_k_cluster2(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t st, bool pdl, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  int n = 1;
  if (pdl) {
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Raises Kernel's dynamic shared-memory limit to `bytes` on the current device, once
// per (kernel, device): the attribute is per device, so an engine on a second GPU
// of the process sets it again.  Concurrent first calls may both set it (harmless).
template <auto Kernel>
inline cudaError_t ensure_smem_limit(int bytes) {
  static std::atomic<unsigned long long> done{0};  // bit d: device d is set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

// Whether decode-path kernels are launched with programmatic dependent launch.
extern bool g_pdl;

// Error flags written by kernels (the host reads them in he_check).
enum : int {
  DEVERR_BAD_TOKEN = 1,    // a token id outside [0, vocab) was replaced by 0
  DEVERR_WAIT_TIMEOUT = 2  // an mbarrier wait ran out of iterations (kernel bailed out)
};

// What a GEMM (or the split-K reduction after it) does with each output
// element C[tok][n] = sum_k X[tok][k] * W[n][k].
enum EpiKind : int {
  EPI_PARTIAL = 0,  // fp32 partial[split][tok][n] (bias/residual applied later, per row)
  EPI_QKV = 1,      // n < d: q (+bq, * hd^-1/2) -> q_out[tok][n]; else k / v (+bias) -> cache
  EPI_RELU = 2,     // out[tok][n] = relu(C + bias[n]) in the storage type
  EPI_STORE_F32 = 3, // fp32 out[tok][n] = C (LM-head logits, kernel tests)
  EPI_ARGMAX = 4     // per 128-row tile t and token: {max_n C, sum_n exp(C - max), lowest n
                     // reaching the max (int bits), 0} as a float4 at partial[t * ldp + tok]
};

struct Epi {
  int kind;
  float *partial;        // EPI_PARTIAL / EPI_STORE_F32 destination
  long long split_stride;// elements between splits of `partial`
  int ldp;               // row stride of `partial`
  const void *bias[3];   // QKV: bq, bk, bv; RELU: bias[0]
  void *out;             // RELU output / QKV q output (storage type)
  int ldo;
  int out_rows;          // RELU output row-tiled with this R (0 = row-major, stride ldo)
  void *kc, *vc;         // QKV: this layer's K / V cache [B][H][max_seq][hd]
  int d_model, n_heads, head_dim, max_seq;
  int tok_per_seq;       // tokens of one sequence in this launch (Lp prefill, 1 decode)
  int pos0;              // position of a sequence's first token in this launch
  float q_scale;
};

// Tiled weight layout used while LoRA is fused (bf16 only): W [N][K] with
// N % 128 == 0 and K % 64 == 0 is stored as (N/128) x (K/64) tiles of 128 x 64,
// tile (mt, kt) contiguous at element (mt * K/64 + kt) * 8192; inside a tile, row r
// occupies 128 bytes whose 16-byte chunk c sits at slot c ^ (r % 8) -- the image
// the tensor cores read with 128-byte swizzling, so one bulk copy fills a stage.
__host__ __device__ inline long long tiled_index(long long n, long long k, long long K) {
  return ((n / 128) * (K / 64) + k / 64) * 8192 + (n % 128) * 64 +
         ((((k % 64) / 8) ^ (n % 8)) * 8) + (k % 8);
}

// Decode activations that feed the stream-K GEMM are stored row-tiled: for a
// buffer of R rows (R = the GEMM's token tile, sk_token_tile(M)) and K columns,
// element (r, k) sits at ((k / 64) * R + r) * 64 + (((k % 64) / 8) ^ (r % 8)) * 8
// + k % 8, so the KPS k-blocks of a pipeline stage are one contiguous, already
// swizzled block.  R == 0 means row-major with row stride K.
__host__ __device__ inline long long act_index(int r, int k, int K, int R) {
  if (R == 0) return (long long)r * K + k;
  return ((long long)(k >> 6) * R + r) * 64 + ((((k & 63) >> 3) ^ (r & 7)) << 3) + (k & 7);
}
inline int sk_token_tile(int M) { return M <= 16 ? 16 : M <= 32 ? 32 : M <= 64 ? 64 : M <= 128 ? 128 : 256; }

struct GemmArgs {
  int dtype;             // parameter type (bias reads): HE_DTYPE_F32 / HE_DTYPE_BF16
  int act;               // operand type of W and X and of the epilogue outputs (ActType)
  const void *x;         // [M][ldx] activations (tokens x K), storage type
  int ldx;
  const void *w[3];      // up to three row groups of `group_rows` rows, each [rows][K]
  int n_groups, group_rows;
  int M, N, K;           // tokens, output features (= n_groups * group_rows), reduction
  int split;             // split-K factor (EPI_PARTIAL writes split slices)
  int w_tiled;           // bf16 only: w[] hold the tiled layout above
  // fp8 weights (stream-K only): w[] hold E4M3 codes in the fp8 tiled layout below and
  // w_scale[] the fp32 scale of every row of each group; output = scale * (codes . x)
  int w_fp8;
  const float *w_scale[3];
  // stream-K with the in-kernel fix-up and at least one whole tile per run: each run
  // takes its share of the leftover tiles first and whole tiles after (no run ends in
  // an owner's fix-up).  Results match plain stream-K up to the order of the fp32 sums.
  int sk_hybrid;
  Epi epi;
};

// FP8 tiled weight layout: W [N][K] with N % 128 == 0 and K % 128 == 0 as (N/128) x
// (K/128) tiles of 128 x 128 one-byte E4M3 codes, tile (mt, kt) contiguous at byte
// (mt * K/128 + kt) * 16384; inside a tile row r occupies 128 bytes whose 16-byte
// chunk c (k = 16 c .. 16 c + 15) sits at slot c ^ (r % 8).
__host__ __device__ inline long long tiled8_index(long long n, long long k, long long K) {
  return ((n / 128) * (K / 128) + k / 128) * 16384 + (n % 128) * 128 +
         ((((k % 128) / 16) ^ (n % 8)) * 16) + (k % 16);
}

// Split-K works in blocks of 64 along K; a split covers split_kblocks(K, S)
// consecutive blocks.  effective_split(K, S) is the number of non-empty slices,
// which callers must pass as GemmArgs::split (the launchers reject other values).
inline int split_kblocks(int K, int split) {
  const int kb = (K + 63) / 64;
  return (kb + split - 1) / split;
}
inline int effective_split(int K, int split) {
  const int kb = (K + 63) / 64;
  if (split < 1) split = 1;
  if (split > kb) split = kb;
  const int per = (kb + split - 1) / split;
  return (kb + per - 1) / per;
}

// Stream-K bookkeeping.  The U = T * KB units (tile, 64-wide k-block) of a GEMM are
// cut into P contiguous runs, run c = [floor(c U / P), floor((c+1) U / P)), so unit x
// belongs to run floor(((x + 1) P - 1) / U).  Tile t is covered by runs c_first..c_last;
// run c writes its part of tile t to slice c - c_first, and S = c_last - c_first + 1
// slices make up the tile.
__host__ __device__ inline void sk_segments(int t, int KB, int P, long long U, int *c_first,
                                            int *S) {
  const long long x0 = (long long)t * KB, x1 = x0 + KB - 1;
  int cf, cl;
  if (U * P < (1LL << 32)) {
    // the same quotients in 32-bit arithmetic ((x + 1) P <= U P fits): a 64-bit
    // division is a long software routine on the GPU, and row kernels ask per thread
    const unsigned u = (unsigned)U, p = (unsigned)P;
    cf = (int)(((unsigned)(x0 + 1) * p - 1u) / u);
    cl = (int)(((unsigned)(x1 + 1) * p - 1u) / u);
  } else {
    cf = (int)(((x0 + 1) * P - 1) / U);
    cl = (int)(((x1 + 1) * P - 1) / U);
  }
  *c_first = cf;
  *S = cl - cf + 1;
}

// How the fp32 slices of a GEMM's output are organised for its consumer: a uniform
// split-K (sk_U == 0: `split` slices everywhere) or stream-K (per 128-column tile).
struct SliceInfo {
  int split;       // uniform slice count (sk_U == 0)
  long long sk_U;  // stream-K units, 0 if not stream-K
  int sk_KB, sk_P;
  __host__ __device__ int slices(int col) const {
    if (sk_U == 0) return split;
    int cf, S;
    sk_segments(col / 128, sk_KB, sk_P, sk_U, &cf, &S);
    return S;
  }
};

// Result codes of the launchers (cudaError_t values pass through).
cudaError_t launch_gemm(const GemmArgs &a, int *dev_err, cudaStream_t st);

// Persistent stream-K tcgen05 GEMM (bf16, M <= 256 tokens, K % 64 == 0; a.x row-tiled
// with R = sk_token_tile(M); N % 128 == 0 for tiled weights, any N for row-major
// weights) on P CTAs; writes fp32 slices [slot][M][N] (slot stride slice_stride)
// except for tiles covered by one run under an element-wise a.epi, stored directly.
// A unit is sk_kps(a) 64-wide k-blocks (2 when K % 128 == 0); sk_units = tiles x
// units per tile.
int sk_kps(const GemmArgs &a);
long long sk_units(const GemmArgs &a);
int sk_ctas(const GemmArgs &a, int num_sms, bool fixup);
// Whether a.epi can be completed inside the kernel (tile_cnt != null): an
// element-wise kind, N % 4 == 0 and vector-aligned outputs.
bool sk_fixup_ok(const GemmArgs &a);
// EPI_ARGMAX needs every split tile finished by its owner's staged reduction
// (shared memory for the slices of the tile with the most runs, on P CTAs).
bool sk_argmax_ok(const GemmArgs &a, int P);
// tile_cnt: null, or ceil(N / 128) ints that are zero at the launch (and are left
// zero): the other runs of a split tile count their finished slices there and the
// tile's owner applies a.epi to the sum, so no reduction kernel follows; the
// slices are then tile-contiguous, [slot][tile][M][128], slice_stride >= M *
// 128 * ceil(N / 128).
cudaError_t launch_gemm_sk(const GemmArgs &a, int P, float *slices, long long slice_stride,
                           int *tile_cnt, int *dev_err, cudaStream_t st);
int gemm_pick_split(const GemmArgs &a, int num_sms);  // heuristic for decode shapes

cudaError_t launch_reduce_epi(int dtype, int act, const float *partial, int split,
                              long long split_stride, int ldp, int M, int N, const Epi &epi,
                              cudaStream_t st);
// Element-wise epilogue over stream-K slices (tiles with one slice were stored already).
cudaError_t launch_sk_reduce_epi(int dtype, int act, const float *partial, const SliceInfo &si,
                                 long long split_stride, int ldp, int M, int N, const Epi &epi,
                                 cudaStream_t st);

// x[row] += sum_s partial[s][row] + bias; h[row] = LN(x[row]; g, b) (storage type,
// row-tiled with h_rows rows when h_rows > 0).
// dev_err (may be null): DEVERR_WAIT_TIMEOUT from the bounded waits of the streaming
// many-rows variant (one slice of 16-bit-model output, d a multiple of 1024).
cudaError_t launch_resid_ln(int dtype, int out_act, const float *partial, const SliceInfo &si,
                            long long split_stride, int ldp, const void *bias, float *x,
                            const void *g, const void *b, float eps, void *h, int h_rows,
                            int rows, int d, cudaStream_t st, int *dev_err = nullptr);
// out (row-tiled, R rows) <- x rows 0..M-1 (row stride ldx), rows M..R-1 zero.
// 16-bit elements (bf16 or fp16 bits).
cudaError_t launch_tile_act(const void *x, int M, int K, int ldx, int R, void *out,
                            cudaStream_t st);
cudaError_t launch_zero(void *p, size_t bytes, cudaStream_t st);

// x[tok] = E[id] + P[pos + off]; h[tok] = LN(x[tok]).  Token tok of a launch is
// sequence tok / tok_per_seq at position pos0 + tok % tok_per_seq.
cudaError_t launch_embed_ln(int dtype, int act, const int32_t *ids, int n_tok, int tok_per_seq, int pos0,
                            const void *tok_emb, const void *pos_emb, int pos_offset, int vocab,
                            const void *g, const void *b, float eps, float *x, void *h, int d,
                            int *dev_err, cudaStream_t st);

struct HeadArgs {
  const float *logits; int ldl; int vocab; int B;
  int step, gen_len;
  const int32_t *force_ids;          // [B][gen_len] or null
  int32_t *out_ids; float *out_lp;   // [B][gen_len]
  const int32_t *log_map;            // [gen_len][B] -> logits_out row or -1 (null = none)
  float *logits_out;
  int embed_next; int pos;           // embed the chosen token at position `pos` for the next pass
  const void *tok_emb, *pos_emb; int pos_offset;
  const void *g, *b; float eps;      // first layer's LN1
  float *x; void *h; int d;
  int h_rows;                        // h row-tiled with this R (0 = row-major)
  // sampling (temperature > 0): softmax(logits / T) cut to its top_p nucleus, drawn by
  // Gumbel-max with SplitMix64 uniforms keyed by (seed, b, step, token); 0 = greedy
  float temperature, top_p;
  unsigned long long seed;
  // greedy from per-tile statistics (EPI_ARGMAX of the LM head) instead of logits:
  // stats[t * B + b] for the n_tiles 128-row vocabulary tiles (logits unused)
  const float4 *stats;
  int n_tiles;
};
// h is written in `act`.
cudaError_t launch_head_select(int dtype, int act, const HeadArgs &a, cudaStream_t st);

// Decode attention: one query per (b, h) over keys 0..n_keys-1 of the cache.
// part: scratch of B*H*split*(hd+2) floats when split > 1; the slices are merged by a
// second kernel, or, with cnt (B*H ints, zero at the launch and left zero), by the
// last CTA of each (b, h) to finish.
// act: type of q, K/V and ctx.  ctx is row-tiled with ctx_rows rows when ctx_rows > 0.
cudaError_t launch_attn_decode(int act, const void *q, const void *kc, const void *vc,
                               void *ctx, int ctx_rows, int B, int H, int hd, int max_seq,
                               int n_keys, int split, float *part, cudaStream_t st,
                               int *cnt = nullptr);
int attn_decode_pick_split(int B, int H, int n_keys, int num_sms);

// Prefill attention: causal within each prompt of Lp tokens (positions 0..Lp-1).
// dev_err: error flags (a bounded wait of the tcgen05 kernel ran out), may be null;
// legacy_mma: use the mma.sync kernel even where the tcgen05 one applies.
cudaError_t launch_attn_prefill(int act, const void *q, const void *kc, const void *vc,
                                void *ctx, int B, int Lp, int H, int hd, int max_seq,
                                int *dev_err, cudaStream_t st, bool legacy_mma = false);
bool attn_prefill_tc_supported(int act, int hd);
cudaError_t launch_attn_prefill_tc(int act, const void *q, const void *kc, const void *vc,
                                   void *ctx, int B, int Lp, int H, int hd, int max_seq,
                                   int *dev_err, cudaStream_t st);

// W <- round(W + scale * B A) after saving W's bits to `save`.
cudaError_t launch_lora_fuse(int dtype, void *w, const void *a, const void *bm, void *save,
                             int rows, int cols, int r, float scale, cudaStream_t st);
// out (tiled layout, type out_act: ACT_BF16 or ACT_F16) <- round(src + scale * B A),
// src, A, B bf16, src row-major [rows][cols]; A / B may be null (then a plain
// re-tiling, bit-exact for ACT_BF16).  out and src must not overlap.  For ACT_F16 with
// r = 8 or 16 (16-byte aligned factors) the delta runs on the tensor cores
// (k_fuse_tc), otherwise on the SIMT pipes (k_fuse_tiled).  dev_err (may be null)
// receives DEVERR_WAIT_TIMEOUT if a bounded wait of the tensor-core kernel ran out.
cudaError_t launch_fuse_tiled(void *out, int out_act, const void *src, const void *a,
                              const void *bm, int rows, int cols, int r, float scale,
                              cudaStream_t st, int *dev_err = nullptr);
bool fuse_tc_supported(int r, const void *a, const void *bm);
cudaError_t launch_fuse_tc(void *out, const void *src, const void *a, const void *bm, int rows,
                           int cols, int r, float scale, int num_sms, int *dev_err,
                           cudaStream_t st);
cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t st);
// FP8 weights of a projection W [rows][cols] (bf16, rows and cols multiples of 128):
// the merged weight W + scale B A (A / B may be null) gets the row scales
// rscale[n] = max_k |W'[n][k]| / 448 (1 for a zero row), its E4M3 codes (nearest,
// ties to even, saturated) in the fp8 tiled layout (out8, rows * cols bytes) and the
// same codes as exact fp16 values in the 16-bit tiled layout (out16).  3 launches
// and a memset of rscale.
cudaError_t launch_fuse_fp8(void *out8, void *out16, float *rscale, const void *src, const void *a,
                            const void *bm, int rows, int cols, int r, float scale,
                            cudaStream_t st);

}  // namespace he
