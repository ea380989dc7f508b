// Attention over the KV cache.
//
// Decode: one query per (sequence, head) against keys 0..n-1.  The cache rows of
// one (b, h) are contiguous ([max_seq][hd]), so a group of hd*sizeof(T)/16 lanes
// reads one key (or value) row with 16-byte loads; the CTA's groups walk the keys
// in an interleaved order, several keys in flight per group, with an online
// (running max) softmax per group, and the groups are merged at the end.  Long
// contexts with few (b, h) pairs are split over the sequence; the slices are
// merged by a second small kernel (no inter-CTA waiting).
//
// Prefill: causal attention inside each prompt, 64 queries per CTA, key blocks
// of 64 staged in shared memory, online softmax across key blocks.  This file
// holds the fp32 CUDA-core version; the 16-bit types run on tensor cores
// (attn_prefill_mma.cu).
#include "common.cuh"
#include "kernels.h"

namespace he {

namespace {

template <typename T> struct Vec16;
template <> struct Vec16<bf16> {
  static constexpr int N = 8;
  __device__ static void load(const bf16 *p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};
template <> struct Vec16<f16> {
  static constexpr int N = 8;
  __device__ static void load(const f16 *p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const __half2 *h = reinterpret_cast<const __half2 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __half22float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  }
};
template <> struct Vec16<float> {
  static constexpr int N = 4;
  __device__ static void load(const float *p, float (&v)[4]) {
    const float4 u = __ldg(reinterpret_cast<const float4 *>(p));
    v[0] = u.x;
    v[1] = u.y;
    v[2] = u.z;
    v[3] = u.w;
  }
};

template <typename T, int HD, int UNROLL>
__global__ void __launch_bounds__(128, 7)  // 72 registers, seven CTAs (28 warps) per SM
    k_attn_decode(const T *__restrict__ q, const T *__restrict__ kc, const T *__restrict__ vc,
                  T *__restrict__ ctx, int ctx_rows, int H, int max_seq, int n_keys, int per_split,
                  float *__restrict__ part, int *__restrict__ cnt) {
  constexpr int VEC = Vec16<T>::N;
  constexpr int LPK = HD / VEC;       // lanes per key row
  constexpr int GROUPS = 128 / LPK;   // key groups per CTA
  static_assert(LPK <= 32 && (32 % LPK) == 0, "a key row must fit in a warp");
  __shared__ float s_m[GROUPS], s_l[GROUPS];
  __shared__ float s_o[GROUPS][HD];
  __shared__ int s_last;

  const int bh = blockIdx.x, sidx = blockIdx.y, nsplit = gridDim.y;
  const int b = bh / H, h = bh - b * H;
  const int j0 = sidx * per_split, j1 = min(n_keys, j0 + per_split);
  const int g = threadIdx.x / LPK, li = threadIdx.x % LPK;
  const long long row0 = ((long long)b * H + h) * max_seq;
  const T *kb = kc + row0 * HD + li * VEC;
  const T *vb = vc + row0 * HD + li * VEC;

  pdl_wait();
  // The next kernel (the out projection) may launch once every CTA of this grid has
  // started, i.e. during the last wave: its CTAs take SMs as these finish, set up and
  // prefetch weights, and wait for this grid to complete before reading its output.
  pdl_trigger();
  float qv[VEC];
  Vec16<T>::load(q + ((long long)b * H + h) * HD + li * VEC, qv);
  float m = -INFINITY, l = 0.f, o[VEC];
#pragma unroll
  for (int i = 0; i < VEC; ++i) o[i] = 0.f;

  for (int base = j0; base < j1; base += GROUPS * UNROLL) {
    float kv[UNROLL][VEC], vv[UNROLL][VEC], s[UNROLL];
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int j = base + u * GROUPS + g;
      if (j < j1) {
        Vec16<T>::load(kb + (long long)j * HD, kv[u]);
        Vec16<T>::load(vb + (long long)j * HD, vv[u]);
      } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) kv[u][i] = vv[u][i] = 0.f;
      }
    }
    float mb = m;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      float d = 0.f;
#pragma unroll
      for (int i = 0; i < VEC; ++i) d = fmaf(qv[i], kv[u][i], d);
#pragma unroll
      for (int o2 = LPK / 2; o2 > 0; o2 >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o2);
      const int j = base + u * GROUPS + g;
      s[u] = j < j1 ? d : -INFINITY;
      mb = fmaxf(mb, s[u]);
    }
    if (mb == -INFINITY) continue;  // no key of this group in this round
    const float corr = expf(m - mb);
    l *= corr;
#pragma unroll
    for (int i = 0; i < VEC; ++i) o[i] *= corr;
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const float p = expf(s[u] - mb);
      l += p;
#pragma unroll
      for (int i = 0; i < VEC; ++i) o[i] = fmaf(p, vv[u][i], o[i]);
    }
    m = mb;
  }
  if (li == 0) {
    s_m[g] = m;
    s_l[g] = l;
  }
#pragma unroll
  for (int i = 0; i < VEC; ++i) s_o[g][li * VEC + i] = o[i];
  __syncthreads();
  if (threadIdx.x < HD) {
    const int dd = threadIdx.x;
    float M = -INFINITY;
#pragma unroll
    for (int k = 0; k < GROUPS; ++k) M = fmaxf(M, s_m[k]);
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int k = 0; k < GROUPS; ++k) {
      const float w = s_m[k] == -INFINITY ? 0.f : expf(s_m[k] - M);
      L = fmaf(s_l[k], w, L);
      O = fmaf(s_o[k][dd], w, O);
    }
    if (nsplit == 1) {
      ctx[act_index(b, h * HD + dd, H * HD, ctx_rows)] = from_f<T>(O / L);
    } else {
      float *pp = part + ((long long)bh * nsplit + sidx) * (HD + 2);
      pp[dd] = O;
      if (dd == 0) {
        pp[HD] = M;
        pp[HD + 1] = L;
      }
    }
  }
  if (nsplit > 1 && cnt) {
    // The key slices of (b, h) are merged by whichever CTA finishes its slice last
    // (a counter per (b, h), no waiting), in slice order, so the result does not
    // depend on which one it is.
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(&cnt[bh], 1) == nsplit - 1;
    __syncthreads();
    if (s_last) {
      __threadfence();
      if (threadIdx.x < HD) {
        const int dd = threadIdx.x;
        const float *pp = part + (long long)bh * nsplit * (HD + 2);
        float M = -INFINITY;
        for (int s2 = 0; s2 < nsplit; ++s2) M = fmaxf(M, __ldcg(pp + s2 * (HD + 2) + HD));
        float L = 0.f, O = 0.f;
        for (int s2 = 0; s2 < nsplit; ++s2) {
          const float ms = __ldcg(pp + s2 * (HD + 2) + HD);
          const float w = ms == -INFINITY ? 0.f : expf(ms - M);
          L = fmaf(__ldcg(pp + s2 * (HD + 2) + HD + 1), w, L);
          O = fmaf(__ldcg(pp + s2 * (HD + 2) + dd), w, O);
        }
        ctx[act_index(b, h * HD + dd, H * HD, ctx_rows)] = from_f<T>(O / L);
      }
      if (threadIdx.x == 0) cnt[bh] = 0;  // every slice of (b, h) has arrived
    }
  }
}

template <typename T, int HD>
__global__ void k_attn_combine(const float *__restrict__ part, T *__restrict__ ctx, int ctx_rows,
                               int H, int nsplit) {
  pdl_wait();
  pdl_trigger();
  const int bh = blockIdx.x, dd = threadIdx.x;
  const float *pp = part + (long long)bh * nsplit * (HD + 2);
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, pp[s * (HD + 2) + HD]);
  float L = 0.f, O = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float ms = pp[s * (HD + 2) + HD];
    const float w = ms == -INFINITY ? 0.f : expf(ms - M);
    L = fmaf(pp[s * (HD + 2) + HD + 1], w, L);
    O = fmaf(pp[s * (HD + 2) + dd], w, O);
  }
  ctx[act_index(bh / H, (bh % H) * HD + dd, H * HD, ctx_rows)] = from_f<T>(O / L);
}

// ---------------------------------------------------------------------------
// Prefill (causal) attention.  Thread (query qi, part p) of 256: scores of keys
// p*16..p*16+15 of the current key block, output dims p*HD/4..(p+1)*HD/4.
// ---------------------------------------------------------------------------
template <typename T, int HD>
__global__ void __launch_bounds__(256)
    k_attn_prefill(const T *__restrict__ q, const T *__restrict__ kc, const T *__restrict__ vc,
                   T *__restrict__ ctx, int H, int Lp, int max_seq) {
  constexpr int QB = 64, KB = 64, LD = HD + 1, DP = HD / 4;
  extern __shared__ float sm[];
  float *qs = sm;               // [QB][LD]
  float *ks = qs + QB * LD;     // [KB][LD]
  float *vs = ks + KB * LD;     // [KB][LD]
  float *ps = vs + KB * LD;     // [QB][KB + 1]
  const int qb = blockIdx.x, bh = blockIdx.y;
  const int b = bh / H, h = bh - b * H;
  const int d = H * HD;
  const int qi = threadIdx.x >> 2, p = threadIdx.x & 3;
  const int t_q = qb * QB + qi;  // query position
  const long long row0 = ((long long)b * H + h) * max_seq;

  for (int e = threadIdx.x; e < QB * HD; e += 256) {
    const int r = e / HD, c = e - r * HD, t = qb * QB + r;
    qs[r * LD + c] = t < Lp ? to_f<T>(q[((long long)b * Lp + t) * d + h * HD + c]) : 0.f;
  }
  float m = -INFINITY, l = 0.f, o[DP];
#pragma unroll
  for (int i = 0; i < DP; ++i) o[i] = 0.f;

  for (int kb = 0; kb <= qb; ++kb) {
    __syncthreads();
    for (int e = threadIdx.x; e < KB * HD; e += 256) {
      const int r = e / HD, c = e - r * HD, t = kb * KB + r;
      const bool in = t < Lp;
      ks[r * LD + c] = in ? to_f<T>(kc[(row0 + t) * HD + c]) : 0.f;
      vs[r * LD + c] = in ? to_f<T>(vc[(row0 + t) * HD + c]) : 0.f;
    }
    __syncthreads();
    float s[16];
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) s[jj] = 0.f;
    for (int c = 0; c < HD; ++c) {
      const float qv = qs[qi * LD + c];
#pragma unroll
      for (int jj = 0; jj < 16; ++jj) s[jj] = fmaf(qv, ks[(p * 16 + jj) * LD + c], s[jj]);
    }
    float mb = -INFINITY;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const int t_k = kb * KB + p * 16 + jj;
      if (t_k > t_q) s[jj] = -INFINITY;
      mb = fmaxf(mb, s[jj]);
    }
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
    mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
    const float mn = fmaxf(m, mb);  // finite: key 0 <= every query position
    const float corr = expf(m - mn);
    float rs = 0.f;
#pragma unroll
    for (int jj = 0; jj < 16; ++jj) {
      const float pj = expf(s[jj] - mn);
      rs += pj;
      ps[qi * (KB + 1) + p * 16 + jj] = pj;
    }
    rs += __shfl_xor_sync(0xffffffffu, rs, 1);
    rs += __shfl_xor_sync(0xffffffffu, rs, 2);
    l = l * corr + rs;
    m = mn;
    __syncwarp();
#pragma unroll
    for (int i = 0; i < DP; ++i) o[i] *= corr;
    for (int j = 0; j < KB; ++j) {
      const float pj = ps[qi * (KB + 1) + j];
#pragma unroll
      for (int i = 0; i < DP; ++i) o[i] = fmaf(pj, vs[j * LD + p * DP + i], o[i]);
    }
  }
  if (t_q < Lp) {
    T *out = ctx + ((long long)b * Lp + t_q) * d + h * HD + p * DP;
#pragma unroll
    for (int i = 0; i < DP; ++i) out[i] = from_f<T>(o[i] / l);
  }
}

template <typename T, int HD>
cudaError_t decode_t(const void *q, const void *kc, const void *vc, void *ctx, int ctx_rows, int B,
                     int H, int max_seq, int n_keys, int split, float *part, int *cnt,
                     cudaStream_t st) {
  const int per = (n_keys + split - 1) / split;
  const int ns = (n_keys + per - 1) / per;
  if (ns > 1 && !part) return cudaErrorInvalidValue;
  dim3 grid(B * H, ns);
  cudaError_t e = launch_k(k_attn_decode<T, HD, 4>, grid, dim3(128), 0, st, g_pdl, (const T *)q,
                           (const T *)kc, (const T *)vc, (T *)ctx, ctx_rows, H, max_seq, n_keys,
                           per, part, cnt);
  if (e == cudaSuccess && ns > 1 && !cnt)
    e = launch_k(k_attn_combine<T, HD>, dim3(B * H), dim3(HD), 0, st, g_pdl, (const float *)part,
                 (T *)ctx, ctx_rows, H, ns);
  return e;
}

template <typename T, int HD>
cudaError_t prefill_t(const void *q, const void *kc, const void *vc, void *ctx, int B, int Lp,
                      int H, int max_seq, cudaStream_t st) {
  constexpr int LD = HD + 1;
  const size_t sm = (size_t)(64 * LD * 3 + 64 * 65) * sizeof(float);
  cudaError_t e = ensure_smem_limit<k_attn_prefill<T, HD>>((int)sm);
  if (e != cudaSuccess) return e;
  dim3 grid((Lp + 63) / 64, B * H);
  k_attn_prefill<T, HD><<<grid, 256, sm, st>>>((const T *)q, (const T *)kc, (const T *)vc,
                                               (T *)ctx, H, Lp, max_seq);
  return cudaGetLastError();
}

}  // namespace

int attn_decode_pick_split(int B, int H, int n_keys, int num_sms) {
  // Enough CTAs for several per SM; no slice shorter than 64 keys.
  const int pairs = B * H;
  int s = 1;
  while (pairs * s < 4 * num_sms && n_keys / (2 * s) >= 64 && s < 32) s *= 2;
  const int per = (n_keys + s - 1) / s;
  return (n_keys + per - 1) / per;
}

cudaError_t launch_attn_decode(int act, const void *q, const void *kc, const void *vc,
                               void *ctx, int ctx_rows, int B, int H, int hd, int max_seq,
                               int n_keys, int split, float *part, cudaStream_t st, int *cnt) {
  if (n_keys <= 0 || split < 1) return cudaErrorInvalidValue;
  auto run = [&](auto tag) -> cudaError_t {
    using T = decltype(tag);
    if (hd == 128)
      return decode_t<T, 128>(q, kc, vc, ctx, ctx_rows, B, H, max_seq, n_keys, split, part, cnt, st);
    if (hd == 64)
      return decode_t<T, 64>(q, kc, vc, ctx, ctx_rows, B, H, max_seq, n_keys, split, part, cnt, st);
    if (hd == 32)
      return decode_t<T, 32>(q, kc, vc, ctx, ctx_rows, B, H, max_seq, n_keys, split, part, cnt, st);
    return cudaErrorInvalidValue;
  };
  if (act == ACT_BF16) return run(bf16{});
  if (act == ACT_F16) return run(f16{});
  if (act == ACT_F32) return run(0.f);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_prefill_mma(int act, const void *q, const void *kc, const void *vc,
                                    void *ctx, int B, int Lp, int H, int hd, int max_seq,
                                    cudaStream_t st);

cudaError_t launch_attn_prefill(int act, const void *q, const void *kc, const void *vc,
                                void *ctx, int B, int Lp, int H, int hd, int max_seq,
                                int *dev_err, cudaStream_t st, bool legacy_mma) {
  // 16-bit types: tcgen05 (attn_prefill_tc.cu) for head sizes 64 and 128, else
  // mma.sync (attn_prefill_mma.cu)
  if (!legacy_mma && attn_prefill_tc_supported(act, hd))
    return launch_attn_prefill_tc(act, q, kc, vc, ctx, B, Lp, H, hd, max_seq, dev_err, st);
  if (act != ACT_F32)
    return launch_attn_prefill_mma(act, q, kc, vc, ctx, B, Lp, H, hd, max_seq, st);
  if (hd == 128) return prefill_t<float, 128>(q, kc, vc, ctx, B, Lp, H, max_seq, st);
  if (hd == 64) return prefill_t<float, 64>(q, kc, vc, ctx, B, Lp, H, max_seq, st);
  if (hd == 32) return prefill_t<float, 32>(q, kc, vc, ctx, B, Lp, H, max_seq, st);
  return cudaErrorInvalidValue;
}

}  // namespace he
