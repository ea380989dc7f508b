// Row kernels of the generation path: embedding + LayerNorm, split-K reduction
// with bias + residual + LayerNorm, the element-wise split-K epilogue, the
// greedy head (argmax, log-softmax, next-token embedding), the LoRA fuse and the
// restore copy.
#include <type_traits>

#include "../../include/he.h"
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "rowops.cuh"

namespace he {

namespace {

// LayerNorm of the fp32 row held in shared memory `row[0..d)`: two passes
// (mean, then the biased variance of the centred values), eps inside the root.
template <typename PT, typename OT>
__device__ void ln_store(const float *row, int d, const PT *g, const PT *b, float eps, OT *h, int r,
                         int R, float *red) {
  float s = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) s += row[i];
  const float mean = block_sum(s, red) / (float)d;
  float v = 0.f;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float c = row[i] - mean;
    v += c * c;
  }
  const float var = block_sum(v, red) / (float)d;
  const float rstd = 1.0f / sqrtf(var + eps);
  for (int i = threadIdx.x; i < d; i += blockDim.x)
    h[act_index(r, i, d, R)] = from_f<OT>((row[i] - mean) * rstd * to_f<PT>(g[i]) + to_f<PT>(b[i]));
}

template <typename PT>
__device__ void embed_row(int id, int pos, const PT *tok_emb, const PT *pos_emb, int d, float *row,
                          float *xout) {
  const PT *e = tok_emb + (long long)id * d;
  const PT *p = pos_emb + (long long)pos * d;
  for (int i = threadIdx.x; i < d; i += blockDim.x) {
    const float v = to_f<PT>(e[i]) + to_f<PT>(p[i]);
    row[i] = v;
    xout[i] = v;
  }
  __syncthreads();
}

template <typename PT, typename CT>
__global__ void k_embed_ln(const int32_t *ids, int tok_per_seq, int pos0, const PT *tok_emb,
                           const PT *pos_emb, int pos_offset, int vocab, const PT *g, const PT *b,
                           float eps, float *x, CT *h, int d, int *dev_err) {
  extern __shared__ float row[];
  __shared__ float red[33];
  pdl_wait();
  pdl_trigger();
  const int tok = blockIdx.x;
  int id = ids[tok];
  if (id < 0 || id >= vocab) {
    if (threadIdx.x == 0) set_dev_error(dev_err, DEVERR_BAD_TOKEN);
    id = 0;
  }
  const int pos = pos0 + tok % tok_per_seq + pos_offset;
  embed_row<PT>(id, pos, tok_emb, pos_emb, d, row, x + (long long)tok * d);
  ln_store<PT, CT>(row, d, g, b, eps, h, tok, 0, red);
}


// One block per row (d % 4 == 0, ldp % 4 == 0): x += sum of slices + bias, then LN.
template <typename PT, typename OT>
__global__ void k_resid_ln(const float *partial, const SliceInfo si, long long split_stride,
                           int ldp, const PT *bias, float *x, const PT *g, const PT *b, float eps,
                           OT *h, int h_rows, int d) {
  extern __shared__ float row[];
  __shared__ float red[33];
  pdl_wait();
  pdl_trigger();
  const long long r = blockIdx.x;
  float4 *xr = reinterpret_cast<float4 *>(x + r * d);
  const float *pr = partial + r * ldp;
  for (int i = threadIdx.x; i < d / 4; i += blockDim.x) {
    const float4 acc = sum_slices(pr + 4 * i, si.slices(4 * i), split_stride);
    float4 v = xr[i];
    v.x += acc.x + to_f<PT>(bias[4 * i]);
    v.y += acc.y + to_f<PT>(bias[4 * i + 1]);
    v.z += acc.z + to_f<PT>(bias[4 * i + 2]);
    v.w += acc.w + to_f<PT>(bias[4 * i + 3]);
    xr[i] = v;
    reinterpret_cast<float4 *>(row)[i] = v;
  }
  __syncthreads();
  ln_store<PT, OT>(row, d, g, b, eps, h, (int)r, h_rows, red);
}


// k_resid_ln with the row held in registers: d / 8 threads (a multiple of 32),
// thread t owns elements 8t .. 8t + 7, so the LN output leaves as one 16-byte
// store into either layout of act_index (eight consecutive elements of a row stay
// contiguous there).  Same arithmetic as k_resid_ln: slices summed in slot order,
// then bias; mean, then the biased variance of the centred values.
template <typename PT, typename OT, int MAXT>
__global__ void __launch_bounds__(MAXT)
    k_resid_ln8(const float *partial, const SliceInfo si, long long split_stride,
                            int ldp, const PT *bias, float *x, const PT *g, const PT *b, float eps,
                            OT *h, int h_rows, int d) {
  __shared__ float red[33];
  const int c = 8 * threadIdx.x;
  float bs[8];
  load8<PT>(bias + c, bs);  // parameters do not depend on the kernel before this one
  // gamma and beta stay packed (4 registers each for 16-bit parameters) until the end
  constexpr int PW = sizeof(PT) / 2;  // 16-byte words per 8 parameters
  uint4 graw[PW], braw[PW];
#pragma unroll
  for (int k = 0; k < PW; ++k) {
    graw[k] = __ldg(reinterpret_cast<const uint4 *>(g + c) + k);
    braw[k] = __ldg(reinterpret_cast<const uint4 *>(b + c) + k);
  }
  pdl_wait();
  pdl_trigger();
  const long long r = blockIdx.x;
  float4 *xr = reinterpret_cast<float4 *>(x + r * d + c);
  const float *pr = partial + r * ldp + c;
  const int S = si.slices(c);
  float4 x0 = xr[0], x1 = xr[1];
  float4 a0, a1;
  sum_slices8<4>(pr, S, split_stride, a0, a1);
  x0.x += a0.x + bs[0];
  x0.y += a0.y + bs[1];
  x0.z += a0.z + bs[2];
  x0.w += a0.w + bs[3];
  x1.x += a1.x + bs[4];
  x1.y += a1.y + bs[5];
  x1.z += a1.z + bs[6];
  x1.w += a1.w + bs[7];
  xr[0] = x0;
  xr[1] = x1;
  float v[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
  float s = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) s += v[i];
  const float mean = block_sum(s, red) / (float)d;
  float q = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    v[i] -= mean;
    q += v[i] * v[i];
  }
  const float var = block_sum(q, red) / (float)d;
  const float rstd = 1.0f / sqrtf(var + eps);
  const PT *gp = reinterpret_cast<const PT *>(graw), *bp = reinterpret_cast<const PT *>(braw);
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = v[i] * rstd * to_f<PT>(gp[i]) + to_f<PT>(bp[i]);
  store8<OT>(h + act_index((int)r, c, d, h_rows), v);
}

// k_resid_ln8 for many rows (prefill): 128 threads per row, so that 16 rows are in
// flight per SM; thread t owns the 8-element groups 8t + 1024 j (d % 1024 == 0).
template <typename PT, typename OT, int NG>
__global__ void __launch_bounds__(128)
    k_resid_ln_rows(const float *partial, const SliceInfo si, long long split_stride, int ldp,
                    const PT *bias, float *x, const PT *g, const PT *b, float eps, OT *h,
                    int h_rows, int d) {
  __shared__ float red[33];
  pdl_wait();
  pdl_trigger();
  const long long r = blockIdx.x;
  float v[NG][8];
  float s = 0.f;
#pragma unroll
  for (int j = 0; j < NG; ++j) {
    const int c = 8 * threadIdx.x + 1024 * j;
    float bs[8];
    load8<PT>(bias + c, bs);
    float4 *xr = reinterpret_cast<float4 *>(x + r * d + c);
    const float *pr = partial + r * ldp + c;
    const int S = si.slices(c);
    const float4 a0 = sum_slices(pr, S, split_stride);
    const float4 a1 = sum_slices(pr + 4, S, split_stride);
    float4 x0 = xr[0], x1 = xr[1];
    x0.x += a0.x + bs[0];
    x0.y += a0.y + bs[1];
    x0.z += a0.z + bs[2];
    x0.w += a0.w + bs[3];
    x1.x += a1.x + bs[4];
    x1.y += a1.y + bs[5];
    x1.z += a1.z + bs[6];
    x1.w += a1.w + bs[7];
    xr[0] = x0;
    xr[1] = x1;
    v[j][0] = x0.x; v[j][1] = x0.y; v[j][2] = x0.z; v[j][3] = x0.w;
    v[j][4] = x1.x; v[j][5] = x1.y; v[j][6] = x1.z; v[j][7] = x1.w;
#pragma unroll
    for (int i = 0; i < 8; ++i) s += v[j][i];
  }
  const float mean = block_sum(s, red) / (float)d;
  float q = 0.f;
#pragma unroll
  for (int j = 0; j < NG; ++j)
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[j][i] -= mean;
      q += v[j][i] * v[j][i];
    }
  const float var = block_sum(q, red) / (float)d;
  const float rstd = 1.0f / sqrtf(var + eps);
#pragma unroll
  for (int j = 0; j < NG; ++j) {
    const int c = 8 * threadIdx.x + 1024 * j;
    float gs[8], bt[8];
    load8<PT>(g + c, gs);
    load8<PT>(b + c, bt);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[j][i] = v[j][i] * rstd * gs[i] + bt[i];
    store8<OT>(h + act_index((int)r, c, d, h_rows), v[j]);
  }
}

// Element-wise epilogue after a split-K GEMM: four consecutive outputs per thread.
template <typename PT, typename CT>
__global__ void k_reduce_epi4(const float *partial, int split, long long split_stride, int ldp,
                              int M, int N, const __grid_constant__ Epi epi) {
  pdl_wait();
  pdl_trigger();
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int n4 = N / 4;
  if (e >= (long long)M * n4) return;
  const int tok = (int)(e / n4), n = (int)(e % n4) * 4;
  const float4 acc = sum_slices(partial + (long long)tok * ldp + n, split, split_stride);
  epi_store<PT, CT>(epi, 0, tok, n, acc.x);
  epi_store<PT, CT>(epi, 0, tok, n + 1, acc.y);
  epi_store<PT, CT>(epi, 0, tok, n + 2, acc.z);
  epi_store<PT, CT>(epi, 0, tok, n + 3, acc.w);
}

// Stream-K slices: tiles with a single slice were stored by the GEMM itself.
template <typename PT, typename CT>
__global__ void k_sk_reduce_epi4(const float *partial, const SliceInfo si, long long split_stride,
                                 int ldp, int M, int N, const __grid_constant__ Epi epi) {
  pdl_wait();
  pdl_trigger();
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int n4 = N / 4;
  if (e >= (long long)M * n4) return;
  const int tok = (int)(e / n4), n = (int)(e % n4) * 4;
  const int S = si.slices(n);
  if (S == 1) return;
  const float4 acc = sum_slices(partial + (long long)tok * ldp + n, S, split_stride);
  epi_store<PT, CT>(epi, 0, tok, n, acc.x);
  epi_store<PT, CT>(epi, 0, tok, n + 1, acc.y);
  epi_store<PT, CT>(epi, 0, tok, n + 2, acc.z);
  epi_store<PT, CT>(epi, 0, tok, n + 3, acc.w);
}

template <typename PT, typename CT>
__global__ void k_reduce_epi(const float *partial, int split, long long split_stride, int ldp,
                             int M, int N, const __grid_constant__ Epi epi) {
  pdl_wait();
  pdl_trigger();
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)M * N) return;
  const int tok = (int)(e / N), n = (int)(e % N);
  float acc = 0.f;
  for (int s = 0; s < split; ++s) acc += partial[s * split_stride + (long long)tok * ldp + n];
  epi_store<PT, CT>(epi, 0, tok, n, acc);
}

// Uniform in (0, 1) for (sequence b, step, token i): output number c + 1 of SplitMix64
// (Steele, Lea and Flood 2014: state += 0x9E3779B97F4A7C15, then the two
// xor-shift-multiply rounds) started from `seed`, c = (b * 2^20 + step) * 2^20 + i,
// as (2 (z >> 41) + 1) / 2^24, exactly representable in fp32.
__device__ __forceinline__ float sample_uniform(unsigned long long seed, int b, int step, int i) {
  const unsigned long long c = ((((unsigned long long)b << 20) + (unsigned long long)step) << 20) +
                               (unsigned long long)i;
  unsigned long long z = seed + (c + 1ull) * 0x9E3779B97F4A7C15ull;
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
  z ^= z >> 31;
  return (float)(2ull * (z >> 41) + 1ull) * (1.0f / 16777216.0f);
}

// Block-wide (value, index) maximum, lowest index on equal values; every thread
// gets the result.
__device__ __forceinline__ void block_argmax(float &best, int &bidx, float *s_val, int *s_idx) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
    if (ov > best || (ov == best && oi < bidx)) {
      best = ov;
      bidx = oi;
    }
  }
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  __syncthreads();
  if (lane == 0) {
    s_val[wid] = best;
    s_idx[wid] = bidx;
  }
  __syncthreads();
  if (wid == 0) {
    best = lane < nw ? s_val[lane] : -INFINITY;
    bidx = lane < nw ? s_idx[lane] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bidx, o);
      if (ov > best || (ov == best && oi < bidx)) {
        best = ov;
        bidx = oi;
      }
    }
    if (lane == 0) {
      s_val[0] = best;
      s_idx[0] = bidx;
    }
  }
  __syncthreads();
  best = s_val[0];
  bidx = s_idx[0];
}

// One block per sequence: greedy choice (lowest index among equal maxima),
// log-prob of the emitted token, optional logit capture, then the embedding of
// the emitted token at the next position followed by the first layer's LN1.
template <typename PT, typename CT>
__global__ void __launch_bounds__(1024) k_head_select(HeadArgs a) {
  extern __shared__ float row[];
  __shared__ float red[33];
  __shared__ float s_val[32];
  __shared__ int s_idx[32];
  __shared__ int s_tok;
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  const float *lg = a.logits + (long long)b * a.ldl;
  // One pass over the row: per thread the maximum with its lowest index (an ascending
  // scan keeps the first hit of a value) and sum exp(l - max), rescaled when the
  // maximum grows; 16-byte loads where the row allows.
  float best = -INFINITY, se = 0.f;
  int bidx = 0x7fffffff;
  auto take = [&](float v, int i) {
    if (v > best) {
      se = se * expf(best - v) + 1.f;  // (0 while best is -inf)
      best = v;
      bidx = i;
    } else {
      se += expf(v - best);
    }
  };
  int done = 0;
  if (a.ldl % 4 == 0 && (reinterpret_cast<uintptr_t>(a.logits) & 15) == 0) {
    const int n4 = a.vocab / 4;
    const float4 *l4 = reinterpret_cast<const float4 *>(lg);
    for (int i = threadIdx.x; i < n4; i += blockDim.x) {
      const float4 v = l4[i];
      take(v.x, 4 * i);
      take(v.y, 4 * i + 1);
      take(v.z, 4 * i + 2);
      take(v.w, 4 * i + 3);
    }
    done = 4 * n4;
  }
  // the scalar rest (indices above every vector one: the scan stays ascending)
  for (int i = done + threadIdx.x; i < a.vocab; i += blockDim.x) take(lg[i], i);
  const float tmax = best, tse = se;
  block_argmax(best, bidx, s_val, s_idx);
  const float m = best;
  const int amax = bidx == 0x7fffffff ? 0 : bidx;
  if (a.temperature > 0.f) {
    // ---- sampling: q_i = exp((l_i - m) / T), nucleus {q_i >= tau}, Gumbel-max ----
    const float inv_t = 1.f / a.temperature;
    float zs = 0.f;
    for (int i = threadIdx.x; i < a.vocab; i += blockDim.x) zs += expf((lg[i] - m) * inv_t);
    const float Z = block_sum(zs, red);
    // tau: the largest q whose "q_j >= tau" mass still reaches top_p * Z, built bit by
    // bit (q <= 1 = the maximum's, so bits 30 and 31 stay clear); every decision is
    // on a block sum, the same in all threads
    uint32_t tau_bits = 0;
    if (a.top_p < 1.f) {
      const float target = a.top_p * Z;
      for (int bit = 29; bit >= 0; --bit) {
        const uint32_t cand = tau_bits | (1u << bit);
        const float x = __uint_as_float(cand);
        float ms = 0.f;
        for (int i = threadIdx.x; i < a.vocab; i += blockDim.x) {
          const float q = expf((lg[i] - m) * inv_t);
          if (q >= x) ms += q;
        }
        if (block_sum(ms, red) >= target) tau_bits = cand;
      }
    }
    const float tau = __uint_as_float(tau_bits);
    float sb = -INFINITY;
    int si = 0x7fffffff;
    for (int i = threadIdx.x; i < a.vocab; i += blockDim.x) {
      const float zi = (lg[i] - m) * inv_t;
      if (expf(zi) >= tau) {
        const float g = -logf(-logf(sample_uniform(a.seed, b, a.step, i)));
        const float sc = zi + g;
        if (sc > sb) {  // ascending scan: the first of equal scores keeps the lowest index
          sb = sc;
          si = i;
        }
      }
    }
    block_argmax(sb, si, s_val, s_idx);
    if (threadIdx.x == 0) {
      int tok = si == 0x7fffffff ? amax : si;
      if (a.force_ids) {
        const int f = a.force_ids[(long long)b * a.gen_len + a.step];
        if (f >= 0 && f < a.vocab) tok = f;
      }
      a.out_ids[(long long)b * a.gen_len + a.step] = tok;
      a.out_lp[(long long)b * a.gen_len + a.step] = (lg[tok] - m) * inv_t - logf(Z);
      s_tok = tok;
    }
  } else {
    const float se = block_sum(tmax == -INFINITY ? 0.f : tse * expf(tmax - m), red);
    if (threadIdx.x == 0) {
      int tok = amax;
      if (a.force_ids) {
        const int f = a.force_ids[(long long)b * a.gen_len + a.step];
        if (f >= 0 && f < a.vocab) tok = f;
      }
      a.out_ids[(long long)b * a.gen_len + a.step] = tok;
      a.out_lp[(long long)b * a.gen_len + a.step] = lg[tok] - (m + logf(se));
      s_tok = tok;
    }
  }
  if (a.log_map) {
    const int r = a.log_map[(long long)a.step * a.B + b];
    if (r >= 0)
      for (int i = threadIdx.x; i < a.vocab; i += blockDim.x)
        a.logits_out[(long long)r * a.vocab + i] = lg[i];
  }
  __syncthreads();
  if (a.embed_next) {
    embed_row<PT>(s_tok, a.pos + a.pos_offset, static_cast<const PT *>(a.tok_emb),
                  static_cast<const PT *>(a.pos_emb), a.d, row, a.x + (long long)b * a.d);
    ln_store<PT, CT>(row, a.d, static_cast<const PT *>(a.g), static_cast<const PT *>(a.b), a.eps,
                     static_cast<CT *>(a.h), b, a.h_rows, red);
  }
}

// Greedy head from the LM head's per-tile statistics (EPI_ARGMAX): one CTA per
// sequence merges the n_tiles {max, exp-sum, lowest index} of its row -- each thread
// the tiles t, t + 1024, ... in order, then a butterfly over each warp and the warps
// in order -- so the token is the lowest index of the row's maximum and its
// log-prob is l_tok - (max + log sum exp(l - max)) = -log(merged sum).  Then, as in
// k_head_select and with its block size (so the LayerNorm sums, and the next step's
// input, are the same bits), the token is embedded and normalised for the next step.
template <typename PT, typename CT>
__global__ void __launch_bounds__(1024) k_head_stats(HeadArgs a) {
  extern __shared__ float row[];
  __shared__ float red[33];
  __shared__ ArgStat wpart[32];
  __shared__ int s_tok;
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.x;
  ArgStat st{-INFINITY, 0.f, 0};
  for (int t = threadIdx.x; t < a.n_tiles; t += blockDim.x) {
    const float4 v = a.stats[(long long)t * a.B + b];
    st = argstat_merge(st, ArgStat{v.x, v.y, __float_as_int(v.z)});
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) st = argstat_merge(st, argstat_shfl_xor(st, o));
  if ((threadIdx.x & 31) == 0) wpart[threadIdx.x >> 5] = st;
  __syncthreads();
  if (threadIdx.x == 0) {
    ArgStat m = wpart[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = argstat_merge(m, wpart[w]);
    a.out_ids[(long long)b * a.gen_len + a.step] = m.i;
    a.out_lp[(long long)b * a.gen_len + a.step] = -logf(m.s);
    s_tok = m.i;
  }
  __syncthreads();
  if (a.embed_next) {
    embed_row<PT>(s_tok, a.pos + a.pos_offset, static_cast<const PT *>(a.tok_emb),
                  static_cast<const PT *>(a.pos_emb), a.d, row, a.x + (long long)b * a.d);
    ln_store<PT, CT>(row, a.d, static_cast<const PT *>(a.g), static_cast<const PT *>(a.b), a.eps,
                     static_cast<CT *>(a.h), b, a.h_rows, red);
  }
}

// W <- round(W + scale * sum_j B[row][j] A[j][col]) for 8 consecutive columns
// per thread, after copying the original bits of W to `save`.
template <typename T>
__global__ void k_lora_fuse(T *w, const T *A, const T *Bm, T *save, int rows, int cols, int r,
                            float scale) {
  const long long gidx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const int gpr = cols / 8;
  if (gidx >= (long long)rows * gpr) return;
  const int row = (int)(gidx / gpr), c0 = (int)(gidx % gpr) * 8;
  T *wp = w + (long long)row * cols + c0;
  T *sp = save + (long long)row * cols + c0;
  T wv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) wv[e] = wp[e];
#pragma unroll
  for (int e = 0; e < 8; ++e) sp[e] = wv[e];
  float delta[8] = {};
  for (int j = 0; j < r; ++j) {
    const float bj = to_f<T>(Bm[(long long)row * r + j]);
    const T *ap = A + (long long)j * cols + c0;
#pragma unroll
    for (int e = 0; e < 8; ++e) delta[e] = fmaf(bj, to_f<T>(ap[e]), delta[e]);
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) wp[e] = from_f<T>(to_f<T>(wv[e]) + scale * delta[e]);
}

// Packed fp32 pairs (low word = first element) and the paired fused multiply-add
// (fma.rn.f32x2: two independent round-to-nearest fmaf in one instruction).
__device__ __forceinline__ uint64_t pack_f2(float lo, float hi) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}
__device__ __forceinline__ void unpack_f2(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// two bf16 (a 32-bit word) -> the packed fp32 pair (exact)
__device__ __forceinline__ uint64_t widen2(uint32_t u) {
  return pack_f2(__uint_as_float(u << 16), __uint_as_float(u & 0xFFFF0000u));
}

// k_resid_ln_rows for one slice of projection output (the prefill GEMMs), as a
// persistent pipeline: each CTA walks rows blockIdx.x, + gridDim.x, ..., and one thread
// keeps the next rows' projection output and residual (d fp32 each) coming into a ring
// of RS_STAGES stages by bulk copies while the CTA works on the current row, so the HBM
// stream does not stop between rows.  Thread t owns the same 8-element groups
// (8t + 1024 j) and does the same arithmetic in the same order as k_resid_ln_rows, so the
// results are bit-identical.  Every wait is bounded (DEVERR_WAIT_TIMEOUT on a timeout).
constexpr int RS_STAGES = 2;

template <typename PT, typename OT, int NG>
__global__ void __launch_bounds__(128)
    k_resid_ln_stream(const float *partial, int ldp, const PT *bias, float *x, const PT *g,
                      const PT *b, float eps, OT *h, int h_rows, int rows, int d, int *dev_err) {
  __shared__ float red[33];
  __shared__ uint64_t full[RS_STAGES];
  extern __shared__ __align__(16) float ring[];  // RS_STAGES x (projection row, residual row)
  const long long first = blockIdx.x, step = gridDim.x;
  const long long n_mine = first < rows ? (rows - first + step - 1) / step : 0;
  const uint32_t row_bytes = (uint32_t)d * 4u;
  if (threadIdx.x == 0) {
    for (int st = 0; st < RS_STAGES; ++st) mbar_init(&full[st], 1);
    fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();  // the projection output and the residual come from the kernels before
  pdl_trigger();
  auto issue = [&](long long i) {
    const int st = (int)(i % RS_STAGES);
    const long long r = first + i * step;
    float *dst = ring + (size_t)st * 2 * d;
    mbar_arrive_expect_tx(&full[st], 2 * row_bytes);
    bulk_load(dst, partial + r * ldp, row_bytes, &full[st]);
    bulk_load(dst + d, x + r * d, row_bytes, &full[st]);
  };
  if (threadIdx.x == 0)
    for (long long i = 0; i < n_mine && i < RS_STAGES; ++i) issue(i);
  long long done = 0;
  for (long long i = 0; i < n_mine; ++i) {
    const int st = (int)(i % RS_STAGES);
    const long long r = first + i * step;
    if (!mbar_wait_bounded(&full[st], (uint32_t)((i / RS_STAGES) & 1))) {
      set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
      break;
    }
    done = i + 1;
    const float *ps = ring + (size_t)st * 2 * d, *xs = ps + d;
    float v[NG][8];
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      const int c = 8 * threadIdx.x + 1024 * j;
      float bs[8];
      load8<PT>(bias + c, bs);
      const float4 p0 = *reinterpret_cast<const float4 *>(ps + c);
      const float4 p1 = *reinterpret_cast<const float4 *>(ps + c + 4);
      float4 x0 = *reinterpret_cast<const float4 *>(xs + c);
      float4 x1 = *reinterpret_cast<const float4 *>(xs + c + 4);
      // the one slice added to zero, as the slice sum does
      x0.x += (0.f + p0.x) + bs[0];
      x0.y += (0.f + p0.y) + bs[1];
      x0.z += (0.f + p0.z) + bs[2];
      x0.w += (0.f + p0.w) + bs[3];
      x1.x += (0.f + p1.x) + bs[4];
      x1.y += (0.f + p1.y) + bs[5];
      x1.z += (0.f + p1.z) + bs[6];
      x1.w += (0.f + p1.w) + bs[7];
      float4 *xr = reinterpret_cast<float4 *>(x + r * d + c);
      xr[0] = x0;
      xr[1] = x1;
      v[j][0] = x0.x; v[j][1] = x0.y; v[j][2] = x0.z; v[j][3] = x0.w;
      v[j][4] = x1.x; v[j][5] = x1.y; v[j][6] = x1.z; v[j][7] = x1.w;
#pragma unroll
      for (int e = 0; e < 8; ++e) sum += v[j][e];
    }
    // every thread has read this stage: refill it with the row after next
    const float mean = block_sum(sum, red) / (float)d;
    if (threadIdx.x == 0 && i + RS_STAGES < n_mine) issue(i + RS_STAGES);
    float q = 0.f;
#pragma unroll
    for (int j = 0; j < NG; ++j)
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        v[j][e] -= mean;
        q += v[j][e] * v[j][e];
      }
    const float var = block_sum(q, red) / (float)d;
    const float rstd = 1.0f / sqrtf(var + eps);
#pragma unroll
    for (int j = 0; j < NG; ++j) {
      const int c = 8 * threadIdx.x + 1024 * j;
      float gs[8], bt[8];
      load8<PT>(g + c, gs);
      load8<PT>(b + c, bt);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[j][e] = v[j][e] * rstd * gs[e] + bt[e];
      store8<OT>(h + act_index((int)r, c, d, h_rows), v[j]);
    }
  }
  // nothing may still be landing when the CTA exits (only after a timeout)
  if (threadIdx.x == 0) {
    const long long issued = n_mine < done + RS_STAGES ? n_mine : done + RS_STAGES;
    for (long long i = done; i < issued; ++i)
      if (!mbar_wait_bounded(&full[i % RS_STAGES], (uint32_t)((i / RS_STAGES) & 1))) break;
  }
}

// The tiled output in 16-byte chunks: chunk q of tile t holds row r = (q % 1024) / 8,
// logical 16-byte column chunk (q % 8) ^ (r % 8).
template <typename OT>
__global__ void __launch_bounds__(256, 4)
    k_fuse_tiled(uint4 *out, const bf16 *src, const bf16 *A, const bf16 *Bm, int rows, int cols,
                 int r, float scale) {
  // One CTA per 128 x 64 tile (1024 chunks).  Thread x takes chunks x + 256 i, i < 4:
  // rows rr + 32 i of the tile, all with the same column chunk c; the four weight
  // loads are in flight together.  The delta of two rows at a time: each 16-byte
  // chunk of a row of A is widened once for both, and a row's r factors of B are one
  // 16-byte load (r % 8 == 0).
  const long long t = blockIdx.x;
  const int KT = cols / 64;
  const int rr = threadIdx.x >> 3, slot = threadIdx.x & 7;
  const int c = slot ^ (rr & 7);
  const int n0 = (int)(t / KT) * 128 + rr, k0 = (int)(t % KT) * 64 + c * 8;
  uint4 raw[4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
    raw[i] = *reinterpret_cast<const uint4 *>(src + (long long)(n0 + 32 * i) * cols + k0);
  uint4 *o = out + t * 1024 + threadIdx.x;
  const bool lora = A != nullptr && r > 0;
  if constexpr (std::is_same<OT, bf16>::value) {
    if (!lora) {
#pragma unroll
      for (int i = 0; i < 4; ++i) o[256 * i] = raw[i];  // plain re-tiling keeps the bits
      return;
    }
  }
  auto widen = [](uint32_t u, float &lo, float &hi) {  // two bf16 -> fp32 (exact)
    lo = __uint_as_float(u << 16);
    hi = __uint_as_float(u & 0xFFFF0000u);
  };
#pragma unroll
  for (int pr = 0; pr < 2; ++pr) {  // rows 2 pr and 2 pr + 1 of this thread
    // delta[i][e] and delta[i][e + 1] as one packed pair: each fma.rn.f32x2 is two
    // independent fmaf, so the sums are those of the scalar loop, bit for bit
    uint64_t delta[2][4] = {};
    for (int j0 = 0; j0 < (lora ? r : 0); j0 += 8) {
      uint4 bu[2];
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const bf16 *bp = Bm + (long long)(n0 + 32 * (2 * pr + i)) * r + j0;
        if (r % 8 == 0) {
          bu[i] = *reinterpret_cast<const uint4 *>(bp);
        } else {
          uint16_t h[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) h[q] = j0 + q < r ? __bfloat16_as_ushort(bp[q]) : (uint16_t)0;
          bu[i] = make_uint4(h[0] | (uint32_t)h[1] << 16, h[2] | (uint32_t)h[3] << 16,
                             h[4] | (uint32_t)h[5] << 16, h[6] | (uint32_t)h[7] << 16);
        }
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        if (j0 + q >= r) break;
        const uint4 av = *reinterpret_cast<const uint4 *>(A + (long long)(j0 + q) * cols + k0);
        const uint64_t a2[4] = {widen2(av.x), widen2(av.y), widen2(av.z), widen2(av.w)};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint32_t word = q < 2 ? bu[i].x : q < 4 ? bu[i].y : q < 6 ? bu[i].z : bu[i].w;
          const float b = __uint_as_float(q & 1 ? (word & 0xFFFF0000u) : (word << 16));
          const uint64_t b2 = pack_f2(b, b);
#pragma unroll
          for (int e = 0; e < 4; ++e) delta[i][e] = fma_f32x2(b2, a2[e], delta[i][e]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const uint4 rw = raw[2 * pr + i];
      float w[8];
      widen(rw.x, w[0], w[1]);
      widen(rw.y, w[2], w[3]);
      widen(rw.z, w[4], w[5]);
      widen(rw.w, w[6], w[7]);
      uint4 res;
      OT *rp = reinterpret_cast<OT *>(&res);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float d0, d1;
        unpack_f2(delta[i][e], d0, d1);
        rp[2 * e] = from_f<OT>(w[2 * e] + scale * d0);
        rp[2 * e + 1] = from_f<OT>(w[2 * e + 1] + scale * d1);
      }
      o[256 * (2 * pr + i)] = res;
    }
  }
}

// FP8 weights, pass 1: per row of the merged weight W + scale B A (bf16 W, A, B),
// the largest |value| as float bits (atomicMax on non-negative bits is the float
// maximum, whatever the order of the tiles) into amax_bits[row], zero on entry.
// One CTA per 128 x 64 tile, the thread layout of k_fuse_tiled.
__global__ void __launch_bounds__(256, 4)
    k_fuse_amax(unsigned *amax_bits, const bf16 *src, const bf16 *A, const bf16 *Bm, int rows,
                int cols, int r, float scale) {
  const long long t = blockIdx.x;
  const int KT = cols / 64;
  const int rr = threadIdx.x >> 3, c = threadIdx.x & 7;
  const int n0 = (int)(t / KT) * 128 + rr, k0 = (int)(t % KT) * 64 + c * 8;
  const bool lora = A != nullptr && r > 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int n = n0 + 32 * i;
    const uint4 raw = *reinterpret_cast<const uint4 *>(src + (long long)n * cols + k0);
    float delta[8] = {};
    for (int j = 0; j < (lora ? r : 0); ++j) {
      const uint4 av = *reinterpret_cast<const uint4 *>(A + (long long)j * cols + k0);
      const bf16 *ap = reinterpret_cast<const bf16 *>(&av);
      const float bj = __bfloat162float(Bm[(long long)n * r + j]);
#pragma unroll
      for (int e = 0; e < 8; ++e) delta[e] = fmaf(bj, __bfloat162float(ap[e]), delta[e]);
    }
    const bf16 *wv = reinterpret_cast<const bf16 *>(&raw);
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(__bfloat162float(wv[e]) + scale * delta[e]));
    // the eight threads of a row (lanes 8 rr' .. 8 rr' + 7 of the warp)
#pragma unroll
    for (int o = 1; o < 8; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (c == 0) atomicMax(&amax_bits[n], __float_as_uint(m));
  }
}

// amax bits -> the row's fp8 scale max|W| / 448 (1 for an all-zero row), in place.
__global__ void k_amax_to_scale(float *s, int rows) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= rows) return;
  const float m = __uint_as_float(reinterpret_cast<const unsigned *>(s)[n]);
  s[n] = m > 0.f ? m / 448.f : 1.f;
}

// FP8 weights, pass 2: the merged weight divided by its row scale, rounded to the
// nearest E4M3 value (ties to even, saturating at 448), into the fp8 tiled layout
// (out8), and the same codes as exact fp16 values into the 16-bit tiled layout
// (out16, read by the prefill GEMMs, which apply the scale in their epilogue).  One
// CTA per 128 x 128 fp8 tile; thread (rr, c) takes 16-byte chunk c of rows rr + 32 i.
__global__ void __launch_bounds__(256, 4)
    k_fuse_q8(uint8_t *out8, uint16_t *out16, const float *rscale, const bf16 *src, const bf16 *A,
              const bf16 *Bm, int rows, int cols, int r, float scale) {
  const long long t = blockIdx.x;
  const int KT8 = cols / 128;
  const int rr = threadIdx.x >> 3, c = threadIdx.x & 7;
  const int tr = (int)(t / KT8), kt = (int)(t % KT8);
  const int k0 = kt * 128 + c * 16;
  const bool lora = A != nullptr && r > 0;
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    const int n = tr * 128 + rr + 32 * i;
    const uint4 *sp = reinterpret_cast<const uint4 *>(src + (long long)n * cols + k0);
    const uint4 raw0 = sp[0], raw1 = sp[1];
    float v[16];
    const bf16 *w0 = reinterpret_cast<const bf16 *>(&raw0);
    const bf16 *w1 = reinterpret_cast<const bf16 *>(&raw1);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      v[e] = __bfloat162float(w0[e]);
      v[8 + e] = __bfloat162float(w1[e]);
    }
    if (lora) {
      float delta[16] = {};
      for (int j = 0; j < r; ++j) {
        const uint4 *ap = reinterpret_cast<const uint4 *>(A + (long long)j * cols + k0);
        const uint4 a0 = ap[0], a1 = ap[1];
        const bf16 *x0 = reinterpret_cast<const bf16 *>(&a0);
        const bf16 *x1 = reinterpret_cast<const bf16 *>(&a1);
        const float bj = __bfloat162float(Bm[(long long)n * r + j]);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          delta[e] = fmaf(bj, __bfloat162float(x0[e]), delta[e]);
          delta[8 + e] = fmaf(bj, __bfloat162float(x1[e]), delta[8 + e]);
        }
      }
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = v[e] + scale * delta[e];
    }
    const float s = rscale[n];
    uint32_t q[4];
    uint4 h16[2];
    uint32_t *hw = reinterpret_cast<uint32_t *>(h16);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const __nv_fp8x2_storage_t p2 =
          __nv_cvt_float2_to_fp8x2(make_float2(v[2 * e] / s, v[2 * e + 1] / s), __NV_SATFINITE,
                                   __NV_E4M3);
      if (e % 2 == 0)
        q[e / 2] = p2;
      else
        q[e / 2] |= (uint32_t)p2 << 16;
      const __half2_raw hp = __nv_cvt_fp8x2_to_halfraw2(p2, __NV_E4M3);
      hw[e] = (uint32_t)hp.x | ((uint32_t)hp.y << 16);
    }
    *reinterpret_cast<uint4 *>(out8 + tiled8_index(n, k0, cols)) = make_uint4(q[0], q[1], q[2], q[3]);
    // the 16 codes as fp16: two 8-element chunks of the 16-bit tiled layout
    *reinterpret_cast<uint4 *>(out16 + tiled_index(n, k0, cols)) = h16[0];
    *reinterpret_cast<uint4 *>(out16 + tiled_index(n, k0 + 8, cols)) = h16[1];
  }
}

__global__ void k_tile_act(const uint16_t *x, int M, int K, int ldx, int R, uint16_t *out) {
  const long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= (long long)R * K) return;
  const int r = (int)(e / K), k = (int)(e % K);
  out[act_index(r, k, K, R)] = r < M ? x[(long long)r * ldx + k] : (uint16_t)0;
}

__global__ void k_zero16(uint4 *p, long long n16) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (long long)gridDim.x * blockDim.x)
    p[i] = make_uint4(0, 0, 0, 0);
}

__global__ void k_copy16(uint4 *dst, const uint4 *src, long long n16) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

__global__ void k_copy1(uint8_t *dst, const uint8_t *src, long long n) {
  const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) dst[i] = src[i];
}

template <typename PT, typename OT, int N>
cudaError_t launch_resid_rows_n(const float *partial, const SliceInfo &si, long long split_stride,
                                int ldp, const PT *bias, float *x, const PT *g, const PT *b,
                                float eps, OT *h, int h_rows, int rows, int d, cudaStream_t st) {
  return launch_k(k_resid_ln_rows<PT, OT, N>, dim3(rows), dim3(128), 0, st, g_pdl, partial, si,
                  split_stride, ldp, bias, x, g, b, eps, h, h_rows, d);
}

template <typename PT, typename OT>
cudaError_t launch_resid_rows(int ng, const float *partial, const SliceInfo &si,
                              long long split_stride, int ldp, const PT *bias, float *x,
                              const PT *g, const PT *b, float eps, OT *h, int h_rows, int rows,
                              int d, cudaStream_t st) {
#define HE_RL(N)                                                                          \
  case N:                                                                                 \
    return launch_resid_rows_n<PT, OT, N>(partial, si, split_stride, ldp, bias, x, g, b, eps, \
                                          h, h_rows, rows, d, st);
  switch (ng) { HE_RL(1) HE_RL(2) HE_RL(3) HE_RL(4) HE_RL(5) HE_RL(6) HE_RL(7) HE_RL(8) }
#undef HE_RL
  return cudaErrorInvalidValue;
}

int row_threads(int d) { return d >= 2048 ? 512 : (d >= 512 ? 256 : 128); }

}  // namespace

cudaError_t launch_embed_ln(int dtype, int act, const int32_t *ids, int n_tok, int tok_per_seq,
                            int pos0, const void *tok_emb, const void *pos_emb, int pos_offset,
                            int vocab, const void *g, const void *b, float eps, float *x, void *h,
                            int d, int *dev_err, cudaStream_t st) {
  if (n_tok <= 0) return cudaSuccess;
  const size_t sm = (size_t)d * sizeof(float);
  HE_DISPATCH_PT_CT(dtype, act, {
    return launch_k(k_embed_ln<PT, CT>, dim3(n_tok), dim3(row_threads(d)), sm, st, g_pdl, ids,
                    tok_per_seq, pos0, (const PT *)tok_emb, (const PT *)pos_emb, pos_offset,
                    vocab, (const PT *)g, (const PT *)b, eps, x, (CT *)h, d, dev_err);
  });
  return cudaSuccess;
}

cudaError_t launch_sk_reduce_epi(int dtype, int act, const float *partial, const SliceInfo &si,
                                 long long split_stride, int ldp, int M, int N, const Epi &epi,
                                 cudaStream_t st) {
  if (N % 4 || ldp % 4 || split_stride % 4 || (uintptr_t)partial % 16) return cudaErrorInvalidValue;
  const long long work = (long long)M * N / 4;
  if (work <= 0) return cudaSuccess;
  const int blocks = (int)((work + 255) / 256);
  HE_DISPATCH_PT_CT(dtype, act, {
    return launch_k(k_sk_reduce_epi4<PT, CT>, dim3(blocks), dim3(256), 0, st, g_pdl, partial, si,
                    split_stride, ldp, M, N, epi);
  });
  return cudaSuccess;
}

template <typename PT, typename OT, int NG>
cudaError_t launch_resid_stream_n(const float *partial, int ldp, const PT *bias, float *x,
                                  const PT *g, const PT *b, float eps, OT *h, int h_rows, int rows,
                                  int d, int *dev_err, cudaStream_t st) {
  const int smem = RS_STAGES * 2 * d * 4;
  cudaError_t e = ensure_smem_limit<k_resid_ln_stream<PT, OT, NG>>(RS_STAGES * 2 * 8192 * 4);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  // as many CTAs as fit the SMs by shared memory (two at d = 5120)
  const int per_sm = std::max(1, std::min(8, (227 * 1024) / (smem + 1024)));
  const int grid = (int)std::min<long long>(rows, (long long)per_sm * sms);
  return launch_k(k_resid_ln_stream<PT, OT, NG>, dim3(grid), dim3(128), (size_t)smem, st, g_pdl,
                  partial, ldp, bias, x, g, b, eps, h, h_rows, rows, d, dev_err);
}

template <typename PT, typename OT>
cudaError_t launch_resid_stream(int ng, const float *partial, int ldp, const PT *bias, float *x,
                                const PT *g, const PT *b, float eps, OT *h, int h_rows, int rows,
                                int d, int *dev_err, cudaStream_t st) {
  switch (ng) {
#define HE_RS_CASE(N)                                                                            \
  case N:                                                                                        \
    return launch_resid_stream_n<PT, OT, N>(partial, ldp, bias, x, g, b, eps, h, h_rows, rows, d, \
                                            dev_err, st);
    HE_RS_CASE(1) HE_RS_CASE(2) HE_RS_CASE(3) HE_RS_CASE(4) HE_RS_CASE(5) HE_RS_CASE(6)
    HE_RS_CASE(7) HE_RS_CASE(8)
#undef HE_RS_CASE
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_resid_ln(int dtype, int out_act, const float *partial, const SliceInfo &si,
                            long long split_stride, int ldp, const void *bias, float *x,
                            const void *g, const void *b, float eps, void *h, int h_rows,
                            int rows, int d, cudaStream_t st, int *dev_err) {
  if (rows <= 0) return cudaSuccess;
  if (d % 4 || ldp % 4 || split_stride % 4 || (uintptr_t)partial % 16 || (uintptr_t)x % 16)
    return cudaErrorInvalidValue;
  const size_t sm = (size_t)d * sizeof(float);
  // 16-bit parameters: the register-resident variant (row of d / 8 threads).
  const bool reg8 = dtype == HE_DTYPE_BF16 && d % 256 == 0 && d / 8 <= 1024 &&
                    (uintptr_t)bias % 16 == 0 && (uintptr_t)g % 16 == 0 &&
                    (uintptr_t)b % 16 == 0 && (uintptr_t)h % 16 == 0;
  // many rows (prefill): four warps per row, up to 8 groups of 1024 elements
  const int ng = d / 1024;
  const bool rows4 = reg8 && rows >= 2048 && d % 1024 == 0 && ng >= 1 && ng <= 8;
  // one slice (the prefill GEMMs): rows streamed into shared memory by bulk copies
  const bool stream1 = rows4 && si.split == 1 && si.sk_U == 0 && ldp % 4 == 0;
  HE_DISPATCH_PT_CT(dtype, out_act, {
    if (stream1)
      return launch_resid_stream<PT, CT>(ng, partial, ldp, (const PT *)bias, x, (const PT *)g,
                                         (const PT *)b, eps, (CT *)h, h_rows, rows, d, dev_err,
                                         st);
    if (rows4)
      return launch_resid_rows<PT, CT>(ng, partial, si, split_stride, ldp, (const PT *)bias, x,
                                       (const PT *)g, (const PT *)b, eps, (CT *)h, h_rows, rows,
                                       d, st);
    if (reg8) {
      // register budget by row width (d / 8 threads)
      auto k = d / 8 <= 512   ? k_resid_ln8<PT, CT, 512>
               : d / 8 <= 640 ? k_resid_ln8<PT, CT, 640>
               : d / 8 <= 768 ? k_resid_ln8<PT, CT, 768>
                              : k_resid_ln8<PT, CT, 1024>;
      return launch_k(k, dim3(rows), dim3(d / 8), 0, st, g_pdl, partial, si, split_stride, ldp,
                      (const PT *)bias, x, (const PT *)g, (const PT *)b, eps, (CT *)h, h_rows, d);
    }
    return launch_k(k_resid_ln<PT, CT>, dim3(rows), dim3(row_threads(d)), sm, st, g_pdl, partial,
                    si, split_stride, ldp, (const PT *)bias, x, (const PT *)g, (const PT *)b, eps,
                    (CT *)h, h_rows, d);
  });
  return cudaSuccess;
}

cudaError_t launch_reduce_epi(int dtype, int act, const float *partial, int split,
                              long long split_stride, int ldp, int M, int N, const Epi &epi,
                              cudaStream_t st) {
  const long long n = (long long)M * N;
  if (n <= 0) return cudaSuccess;
  const bool vec = N % 4 == 0 && ldp % 4 == 0 && split_stride % 4 == 0 &&
                   (uintptr_t)partial % 16 == 0;
  const long long work = vec ? n / 4 : n;
  const int blocks = (int)((work + 255) / 256);
  HE_DISPATCH_PT_CT(dtype, act, {
    if (vec)
      return launch_k(k_reduce_epi4<PT, CT>, dim3(blocks), dim3(256), 0, st, g_pdl, partial,
                      split, split_stride, ldp, M, N, epi);
    return launch_k(k_reduce_epi<PT, CT>, dim3(blocks), dim3(256), 0, st, g_pdl, partial, split,
                    split_stride, ldp, M, N, epi);
  });
  return cudaSuccess;
}

cudaError_t launch_head_select(int dtype, int act, const HeadArgs &a, cudaStream_t st) {
  const size_t sm = (size_t)a.d * sizeof(float);
  if (a.stats && (a.temperature > 0.f || a.force_ids || a.log_map || a.n_tiles < 1))
    return cudaErrorInvalidValue;  // the statistics serve greedy choice only
  HE_DISPATCH_PT_CT(dtype, act, {
    if (a.stats) return launch_k(k_head_stats<PT, CT>, dim3(a.B), dim3(1024), sm, st, g_pdl, a);
    return launch_k(k_head_select<PT, CT>, dim3(a.B), dim3(1024), sm, st, g_pdl, a);
  });
  return cudaSuccess;
}

cudaError_t launch_lora_fuse(int dtype, void *w, const void *a, const void *bm, void *save,
                             int rows, int cols, int r, float scale, cudaStream_t st) {
  if (cols % 8) return cudaErrorInvalidValue;
  const long long groups = (long long)rows * (cols / 8);
  const int blocks = (int)((groups + 255) / 256);
  if (dtype == 1)
    k_lora_fuse<bf16><<<blocks, 256, 0, st>>>((bf16 *)w, (const bf16 *)a, (const bf16 *)bm,
                                              (bf16 *)save, rows, cols, r, scale);
  else
    k_lora_fuse<float><<<blocks, 256, 0, st>>>((float *)w, (const float *)a, (const float *)bm,
                                               (float *)save, rows, cols, r, scale);
  return cudaGetLastError();
}

cudaError_t launch_fuse_tiled(void *out, int out_act, const void *src, const void *a,
                              const void *bm, int rows, int cols, int r, float scale,
                              cudaStream_t st, int *dev_err) {
  if (rows % 128 || cols % 64) return cudaErrorInvalidValue;
  const long long tiles = (long long)(rows / 128) * (cols / 64);
  if (tiles > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int blocks = (int)tiles;
  if (out_act == ACT_F16 && fuse_tc_supported(r, a, bm)) {  // the delta on the tensor cores
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    return launch_fuse_tc(out, src, a, bm, rows, cols, r, scale, sms, dev_err, st);
  }
  if (out_act == ACT_F16)
    k_fuse_tiled<f16><<<blocks, 256, 0, st>>>((uint4 *)out, (const bf16 *)src, (const bf16 *)a,
                                              (const bf16 *)bm, rows, cols, r, scale);
  else if (out_act == ACT_BF16)
    k_fuse_tiled<bf16><<<blocks, 256, 0, st>>>((uint4 *)out, (const bf16 *)src, (const bf16 *)a,
                                               (const bf16 *)bm, rows, cols, r, scale);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

cudaError_t launch_fuse_fp8(void *out8, void *out16, float *rscale, const void *src, const void *a,
                            const void *bm, int rows, int cols, int r, float scale,
                            cudaStream_t st) {
  if (rows % 128 || cols % 128 || !out8 || !out16 || !rscale) return cudaErrorInvalidValue;
  const long long tiles64 = (long long)(rows / 128) * (cols / 64);
  if (tiles64 > 0x7fffffffLL) return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(rscale, 0, (size_t)rows * sizeof(float), st);
  if (e != cudaSuccess) return e;
  k_fuse_amax<<<(int)tiles64, 256, 0, st>>>(reinterpret_cast<unsigned *>(rscale),
                                            (const bf16 *)src, (const bf16 *)a, (const bf16 *)bm,
                                            rows, cols, r, scale);
  k_amax_to_scale<<<(rows + 255) / 256, 256, 0, st>>>(rscale, rows);
  k_fuse_q8<<<(int)(tiles64 / 2), 256, 0, st>>>((uint8_t *)out8, (uint16_t *)out16, rscale,
                                                (const bf16 *)src, (const bf16 *)a,
                                                (const bf16 *)bm, rows, cols, r, scale);
  return cudaGetLastError();
}

cudaError_t launch_tile_act(const void *x, int M, int K, int ldx, int R, void *out,
                            cudaStream_t st) {
  if (K % 64 || R < M) return cudaErrorInvalidValue;
  const long long n = (long long)R * K;
  k_tile_act<<<(int)((n + 255) / 256), 256, 0, st>>>((const uint16_t *)x, M, K, ldx, R,
                                                    (uint16_t *)out);
  return cudaGetLastError();
}

cudaError_t launch_zero(void *p, size_t bytes, cudaStream_t st) {
  if (bytes % 16 || (uintptr_t)p % 16) return cudaErrorInvalidValue;
  const long long n16 = (long long)(bytes / 16);
  if (n16 == 0) return cudaSuccess;
  const long long blocks = (n16 + 255) / 256;
  k_zero16<<<(int)(blocks < 4096 ? blocks : 4096), 256, 0, st>>>((uint4 *)p, n16);
  return cudaGetLastError();
}

cudaError_t launch_copy(void *dst, const void *src, size_t bytes, cudaStream_t st) {
  if (bytes == 0) return cudaSuccess;
  const bool aligned = ((uintptr_t)dst % 16 == 0) && ((uintptr_t)src % 16 == 0);
  const long long n16 = aligned ? (long long)(bytes / 16) : 0;
  if (n16 > 0) {
    const long long blocks = (n16 + 255) / 256;
    k_copy16<<<(int)(blocks < 4096 ? blocks : 4096), 256, 0, st>>>((uint4 *)dst, (const uint4 *)src,
                                                                   n16);
  }
  const long long done = n16 * 16, rest = (long long)bytes - done;
  if (rest > 0)
    k_copy1<<<(int)((rest + 255) / 256), 256, 0, st>>>((uint8_t *)dst + done,
                                                      (const uint8_t *)src + done, rest);
  return cudaGetLastError();
}

}  // namespace he
