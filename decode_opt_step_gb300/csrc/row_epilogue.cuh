// Row-wise GEMM epilogue for the tensor-core kernels (bias bf16, outputs CT).
//
// In the tcgen05 kernels a thread owns one output feature n (a TMEM lane) and a
// run of consecutive tokens (TMEM columns).  Everything that depends only on n
// (bias, which of q/k/v, head and lane of the KV cache, destination base) is
// computed once; the token loop then does one add and one store per element,
// tracking (sequence, position) of the token incrementally instead of dividing.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace he {

template <typename CT>
struct RowEpi {
  int mode;          // 0 fp32 store (partial / logits / slices), 1 q, 2 k or v cache, 3 relu
  float bias, scale;
  float *f32;        // mode 0: element of token 0; token stride f32_stride
  long long f32_stride;
  CT *dst;           // modes 1-3
  long long tok_stride;  // modes 1, 2 (per sequence for 2)
  long long pos_stride;  // mode 2: per position inside a sequence
  int n, ldo, out_rows;  // mode 3 (row-tiled output when out_rows > 0)
  int tok_per_seq;
};

// Constants of output row n for tokens starting at `tok0`.  slices != null means
// "write fp32 slice `slot`" instead of the epilogue of `e`.
template <typename CT>
__device__ __forceinline__ RowEpi<CT> row_epi_prepare(const Epi &e, int n, float *slices,
                                                      long long slice_stride, int slot, int ldn) {
  RowEpi<CT> r{};
  r.n = n;
  if (slices) {
    r.mode = 0;
    r.f32 = slices + (long long)slot * slice_stride + n;
    r.f32_stride = ldn;
    return r;
  }
  switch (e.kind) {
    case EPI_PARTIAL:
      r.mode = 0;
      r.f32 = e.partial + n;
      r.f32_stride = e.ldp;
      break;
    case EPI_STORE_F32:
      r.mode = 0;
      r.f32 = e.partial + n;
      r.f32_stride = e.ldp;
      break;
    case EPI_RELU:
      r.mode = 3;
      r.bias = __bfloat162float(static_cast<const bf16 *>(e.bias[0])[n]);
      r.dst = static_cast<CT *>(e.out);
      r.ldo = e.ldo;
      r.out_rows = e.out_rows;
      break;
    case EPI_QKV: {
      const int which = n / e.d_model;
      const int c = n - which * e.d_model;
      r.bias = __bfloat162float(static_cast<const bf16 *>(e.bias[which])[c]);
      if (which == 0) {
        r.mode = 1;
        r.scale = e.q_scale;
        r.dst = static_cast<CT *>(e.out) + c;
        r.tok_stride = e.ldo;
      } else {
        r.mode = 2;
        const int hh = c / e.head_dim, dd = c - hh * e.head_dim;
        r.dst = static_cast<CT *>(which == 1 ? e.kc : e.vc) +
                ((long long)hh * e.max_seq + e.pos0) * e.head_dim + dd;
        r.tok_stride = (long long)e.n_heads * e.max_seq * e.head_dim;  // next sequence
        r.pos_stride = e.head_dim;                                      // next position
        r.tok_per_seq = e.tok_per_seq;
      }
      break;
    }
  }
  return r;
}

// Stores v[0..cnt) for tokens tok0 .. tok0 + cnt - 1 (all < M).
template <typename CT, int CNT>
__device__ __forceinline__ void row_epi_store(const RowEpi<CT> &r, int tok0, int cnt,
                                              const float (&v)[CNT]) {
  switch (r.mode) {
    case 0: {
      float *p = r.f32 + (long long)tok0 * r.f32_stride;
#pragma unroll
      for (int j = 0; j < CNT; ++j)
        if (j < cnt) p[(long long)j * r.f32_stride] = v[j];
      break;
    }
    case 1: {
      CT *p = r.dst + (long long)tok0 * r.tok_stride;
#pragma unroll
      for (int j = 0; j < CNT; ++j)
        if (j < cnt) p[(long long)j * r.tok_stride] = from_f<CT>((v[j] + r.bias) * r.scale);
      break;
    }
    case 2: {
      int b = tok0 / r.tok_per_seq, t = tok0 - b * r.tok_per_seq;
#pragma unroll
      for (int j = 0; j < CNT; ++j) {
        if (j < cnt)
          r.dst[(long long)b * r.tok_stride + (long long)t * r.pos_stride] =
              from_f<CT>(v[j] + r.bias);
        if (++t == r.tok_per_seq) {
          t = 0;
          ++b;
        }
      }
      break;
    }
    case 3: {
#pragma unroll
      for (int j = 0; j < CNT; ++j)
        if (j < cnt)
          r.dst[act_index(tok0 + j, r.n, r.ldo, r.out_rows)] =
              from_f<CT>(fmaxf(v[j] + r.bias, 0.f));
      break;
    }
  }
}

template <typename CT>
__device__ __forceinline__ void store4(CT *p, float a, float b, float c, float d) {
  union {
    uint2 u;
    CT e[4];
  } pk;
  pk.e[0] = from_f<CT>(a);
  pk.e[1] = from_f<CT>(b);
  pk.e[2] = from_f<CT>(c);
  pk.e[3] = from_f<CT>(d);
  *reinterpret_cast<uint2 *>(p) = pk.u;
}

// Final epilogue of one 128-feature output tile from its S fp32 slices
// (tile-contiguous: tslices + s * sstride + tok * 128 + feature in the tile,
// s = 0 .. S-1), summed in slot order.  Called by the NT threads et = 0..NT-1
// of one CTA: thread et owns features n0 .. n0 + 3 with n0 = 128 t + 4 (et % 32)
// and tokens et / 32, et / 32 + NT / 32, ...; a warp thus reads and writes 128
// consecutive features of one token (coalesced).
// Needs N % 4 == 0 and, per kind, 16-byte aligned fp32 rows (STORE_F32) or
// 8-byte aligned groups of four 16-bit outputs (QKV, RELU).
template <typename CT, int NT>
__device__ __forceinline__ void tile_fixup(const Epi &e, const float *tslices, long long sstride,
                                           int N, int M, int t, int S, int et) {
  const int n0 = t * 128 + 4 * (et & 31);
  if (n0 >= N || e.kind == EPI_ARGMAX) return;  // (EPI_ARGMAX tiles are always staged)
  float b4[4] = {0.f, 0.f, 0.f, 0.f};
  float scale = 1.f;
  int mode = 0;
  float *f32 = nullptr;
  CT *dst = nullptr;
  long long tok_stride = 0, pos_stride = 0;
  int tps = 1;
  auto bias4 = [&](const void *bp, int c) {
    const bf16 *bb = static_cast<const bf16 *>(bp) + c;
#pragma unroll
    for (int i = 0; i < 4; ++i) b4[i] = __bfloat162float(bb[i]);
  };
  switch (e.kind) {
    case EPI_STORE_F32:
    case EPI_PARTIAL:
      mode = 0;
      f32 = e.partial + n0;
      tok_stride = e.ldp;
      break;
    case EPI_RELU:
      mode = 3;
      bias4(e.bias[0], n0);
      dst = static_cast<CT *>(e.out);
      break;
    case EPI_QKV: {
      const int which = n0 / e.d_model;
      const int c = n0 - which * e.d_model;
      bias4(e.bias[which], c);
      if (which == 0) {
        mode = 1;
        scale = e.q_scale;
        dst = static_cast<CT *>(e.out) + c;
        tok_stride = e.ldo;
      } else {
        mode = 2;
        const int hh = c / e.head_dim, dd = c - hh * e.head_dim;
        dst = static_cast<CT *>(which == 1 ? e.kc : e.vc) +
              ((long long)hh * e.max_seq + e.pos0) * e.head_dim + dd;
        tok_stride = (long long)e.n_heads * e.max_seq * e.head_dim;
        pos_stride = e.head_dim;
        tps = e.tok_per_seq;
      }
      break;
    }
  }
  const float *src = tslices + 4 * (et & 31);
  constexpr int TU = 8;  // tokens per thread per round: 8 x 2 slices of loads in flight
  constexpr int TS = NT / 32;  // token step between a thread's tokens
  for (int tb = et >> 5; tb < M; tb += TS * TU) {
    float4 acc[TU];
#pragma unroll
    for (int i = 0; i < TU; ++i) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int s = 0; s < S; s += 2) {
      float4 v0[TU], v1[TU];
#pragma unroll
      for (int i = 0; i < TU; ++i) {
        const int tok = tb + TS * i;
        const float *p = src + (long long)s * sstride + (long long)tok * 128;
        v0[i] = tok < M ? __ldcg(reinterpret_cast<const float4 *>(p)) : make_float4(0.f, 0.f, 0.f, 0.f);
        v1[i] = tok < M && s + 1 < S ? __ldcg(reinterpret_cast<const float4 *>(p + sstride))
                                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < TU; ++i) {
        acc[i].x += v0[i].x;
        acc[i].y += v0[i].y;
        acc[i].z += v0[i].z;
        acc[i].w += v0[i].w;
        if (s + 1 < S) {
          acc[i].x += v1[i].x;
          acc[i].y += v1[i].y;
          acc[i].z += v1[i].z;
          acc[i].w += v1[i].w;
        }
      }
    }
#pragma unroll
    for (int i = 0; i < TU; ++i) {
      const int tok = tb + TS * i;
      if (tok >= M) break;
      const float4 a = acc[i];
      switch (mode) {
        case 0:
          *reinterpret_cast<float4 *>(f32 + (long long)tok * tok_stride) = a;
          break;
        case 1:
          store4<CT>(dst + (long long)tok * tok_stride, (a.x + b4[0]) * scale,
                     (a.y + b4[1]) * scale, (a.z + b4[2]) * scale, (a.w + b4[3]) * scale);
          break;
        case 2: {
          const int b = tok / tps, p = tok - b * tps;
          store4<CT>(dst + (long long)b * tok_stride + (long long)p * pos_stride, a.x + b4[0],
                     a.y + b4[1], a.z + b4[2], a.w + b4[3]);
          break;
        }
        case 3:
          store4<CT>(dst + act_index(tok, n0, e.ldo, e.out_rows), fmaxf(a.x + b4[0], 0.f),
                     fmaxf(a.y + b4[1], 0.f), fmaxf(a.z + b4[2], 0.f), fmaxf(a.w + b4[3], 0.f));
          break;
      }
    }
  }
}

// Output element type of a stream-K tile's final epilogue: fp32 logits / partial
// sums (and the raw values EPI_ARGMAX reduces), else the activation type.
__host__ __device__ inline int tile_out_bytes(int kind, int ct_bytes) {
  return kind == EPI_STORE_F32 || kind == EPI_PARTIAL || kind == EPI_ARGMAX ? 4 : ct_bytes;
}


// Tokens of a tile that the staged reduction of the tile's owner handles at a
// time in `avail` bytes of shared memory (a multiple of W; 0 if not even W fit):
// per token, the S - 1 other slices' 128 fp32 values and the 128 fp32 outputs.
__host__ __device__ inline int tile_stage_tokens(int S, int M, int W, int avail) {
  const int per_tok = S * 512;
  int ch = avail / per_tok / W * W;
  const int m = (M + W - 1) / W * W;
  return ch < m ? ch : m;
}

// Where the outputs of feature n (and the following ones of its 16-byte group)
// go, for any token: the part that depends on n only, computed once.
struct TileOutRow {
  char *base;                       // element of token 0 (kind 0 / 1) or the buffer (kind 2)
  long long tok_stride, pos_stride;  // bytes
  int kind;                         // 0 base + tok * tok_stride; 1 KV cache; 2 act_index layout
  int tps, n, ldo, rows, esize;
};

template <typename CT>
__device__ __forceinline__ TileOutRow tile_out_row(const Epi &e, int n) {
  TileOutRow o{};
  o.n = n;
  switch (e.kind) {
    case EPI_QKV: {
      const int which = n / e.d_model, c = n - which * e.d_model;
      o.esize = (int)sizeof(CT);
      if (which == 0) {
        o.kind = 0;
        o.base = reinterpret_cast<char *>(static_cast<CT *>(e.out) + c);
        o.tok_stride = (long long)e.ldo * sizeof(CT);
      } else {
        const int hh = c / e.head_dim, dd = c - hh * e.head_dim;
        o.kind = 1;
        o.base = reinterpret_cast<char *>(static_cast<CT *>(which == 1 ? e.kc : e.vc) +
                                          ((long long)hh * e.max_seq + e.pos0) * e.head_dim + dd);
        o.tok_stride = (long long)e.n_heads * e.max_seq * e.head_dim * sizeof(CT);
        o.pos_stride = (long long)e.head_dim * sizeof(CT);
        o.tps = e.tok_per_seq;
      }
      break;
    }
    case EPI_RELU:
      o.kind = 2;
      o.esize = (int)sizeof(CT);
      o.base = static_cast<char *>(e.out);
      o.ldo = e.ldo;
      o.rows = e.out_rows;
      break;
    default:
      o.kind = 0;
      o.esize = 4;
      o.base = reinterpret_cast<char *>(e.partial + n);
      o.tok_stride = (long long)e.ldp * 4;
      break;
  }
  return o;
}

__device__ __forceinline__ void *tile_out_ptr(const TileOutRow &o, int tok) {
  switch (o.kind) {
    case 0:
      return o.base + tok * o.tok_stride;
    case 1: {
      const int b = tok / o.tps, p = tok - b * o.tps;
      return o.base + b * o.tok_stride + p * o.pos_stride;
    }
    default:
      return o.base + act_index(tok, o.n, o.ldo, o.rows) * o.esize;
  }
}

// Bias of output feature n for an element-wise epilogue (0 past N or without one).
__device__ __forceinline__ float tile_row_bias(const Epi &e, int n, int N) {
  if (n >= N) return 0.f;
  if (e.kind == EPI_RELU) return __bfloat162float(static_cast<const bf16 *>(e.bias[0])[n]);
  if (e.kind == EPI_QKV) {
    const int which = n / e.d_model;
    return __bfloat162float(static_cast<const bf16 *>(e.bias[which])[n - which * e.d_model]);
  }
  return 0.f;
}

// Final epilogue of stream-K tile t by its owner (the run holding the tile's first
// k-blocks, whose accumulator is in TMEM at `tl` for this thread's row), with the
// other S - 1 runs' fp32 slices in global memory (tile-contiguous: tslices +
// s * sstride + tok * 128 + feature), once they have all counted themselves in
// *cnt.  Runs on the NT (256) epilogue threads, two per TMEM lane (et and et +
// 128 take alternate W-column chunks), after the CTA's
// last MMA, so the pipeline's shared memory `stage` (avail bytes) is free: per
// chunk of ch tokens the other slices come in as one bulk copy each (completing
// on the mbarrier `bar`), each thread adds its row's values in slot order (its own
// slice is slot 0) and applies the epilogue into a [token][128] fp32 staging
// tile, which then leaves (rounded to the output type) as 16-byte stores.  `bias`
// is this thread's row's (tile_row_bias); `rs` scales this thread's own accumulator
// (the row scale of fp8 weights, else 1; the other slices arrive scaled).  `flag` is
// a shared int; returns with
// every epilogue thread past the same barriers.
template <typename CT, int W, int NT>
__device__ __forceinline__ void tile_owner_epilogue(const Epi &e, const float *tslices,
                                                    long long sstride, int N, int M, int t, int S,
                                                    uint32_t tl, bool live, int *cnt,
                                                    uint8_t *stage, int avail, uint64_t *bar,
                                                    int *flag, int *dev_err, float bias,
                                                    float rs = 1.f) {
  static_assert(NT == 256, "two threads per TMEM lane");
  const int et = threadIdx.x, r = et & 127, hf = et >> 7;  // row (feature) of the tile, half
  const int n_row = t * 128 + r;
  // per-row epilogue constants (`bias`, this row's, was read by the caller)
  float scale = 1.f;
  if (n_row < N && e.kind == EPI_QKV && n_row < e.d_model) scale = e.q_scale;
  epi_bar_sync<NT>();  // *flag may still be read from an earlier segment
  if (et == 0) {
    // acquire: the other runs' slices (written, fenced, then counted) are visible
    // to this thread and, through the barrier below, to the whole group
    bool ok = live;
    if (ok && S > 1 && !wait_count_at_least(cnt, S - 1)) {
      set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
      ok = false;
    }
    *flag = ok;
  }
  epi_bar_sync<NT>();
  const bool go = *flag != 0;
  const int ob = tile_out_bytes(e.kind, (int)sizeof(CT));
  const bool relu = e.kind == EPI_RELU;
  const int ch = tile_stage_tokens(S, M, W, avail);
  float *ps = reinterpret_cast<float *>(stage);      // [S-1][ch][128] other slices
  uint8_t *os = stage + (size_t)(S - 1) * ch * 512;  // [ch][128] fp32 outputs
  uint32_t phase = 0;
  for (int c0 = 0; c0 < M; c0 += ch) {
    const int cn = min(ch, M - c0);
    if (go && S > 1) {
      if (et == 0) {
        // earlier generic reads of the staging area come before these async writes
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        mbar_arrive_expect_tx(bar, (uint32_t)((S - 1) * cn * 512));
        for (int s = 1; s < S; ++s)
          bulk_load(ps + (size_t)(s - 1) * ch * 128, tslices + s * sstride + (size_t)c0 * 128,
                    (uint32_t)(cn * 512), bar);
      }
      if (!mbar_wait_bounded(bar, phase)) set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
      phase ^= 1;
    }
    epi_bar_sync<NT>();
    const uint32_t ps_s = smem_u32(ps), os_s = smem_u32(os);
#pragma unroll 1
    for (int j0 = hf * W; j0 < cn; j0 += 2 * W) {
      // own accumulator (slot 0), then the other slots in order; rows j0 .. j0+W-1
      // stay inside the chunk's staging (ch is a multiple of W)
      float v[W];
      tmem_load_cols<W>(tl + (uint32_t)(c0 + j0), v);
#pragma unroll
      for (int j = 0; j < W; ++j) v[j] *= rs;  // (the row's fp8 weight scale, else 1)
      for (int s = 0; s < S - 1; ++s) {
        const uint32_t src = ps_s + (uint32_t)((((size_t)s * ch + j0) * 128 + r) * 4);
        float p[W];
#pragma unroll
        for (int j = 0; j < W; ++j) p[j] = lds_f32(src + j * 512);
#pragma unroll
        for (int j = 0; j < W; ++j) v[j] += p[j];
      }
#pragma unroll
      for (int j = 0; j < W; ++j) {
        float y = v[j];
        if (ob != 4) {
          y = (y + bias) * scale;
          if (relu) y = fmaxf(y, 0.f);
        }
        sts_f32(os_s + (uint32_t)(((j0 + j) * 128 + r) * 4), y);
      }
    }
    epi_bar_sync<NT>();
    if (e.kind == EPI_ARGMAX) {
      // two threads per token, 64 features each, then merged: the tile's statistics
      float4 *stats = reinterpret_cast<float4 *>(e.partial);
      const int hf2 = et & 1;
      for (int jb = (et >> 1) & ~15; jb < cn; jb += NT / 2) {  // warp-uniform bound
        const int jj = jb + ((et >> 1) & 15);
        ArgStat st{-INFINITY, 0.f, 0};
        if (jj < cn) {
          const int f0 = 64 * hf2;
#pragma unroll 4
          for (int f = f0; f < f0 + 64; f += 4) {
            const uint4 q4 = lds_u128(os_s + (uint32_t)((jj * 128 + f) * 4));
            const float q[4] = {__uint_as_float(q4.x), __uint_as_float(q4.y),
                                __uint_as_float(q4.z), __uint_as_float(q4.w)};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (t * 128 + f + e < N) argstat_add(st, q[e], t * 128 + f + e);
          }
        }
        st = argstat_merge(st, argstat_shfl_xor(st, 1));
        if (go && jj < cn && hf2 == 0)
          stats[(size_t)t * e.ldp + c0 + jj] =
              make_float4(st.m, st.s, __int_as_float(st.i), 0.f);
      }
    } else if (go) {
      // 16-byte output groups (4 fp32 values, or 8 values rounded to CT): thread et
      // always takes group et % cpr of rows et / cpr, et / cpr + 128 / cpr, ...
      const int per = 16 / ob, cpr = 128 / per;
      const int k = et % cpr, n = t * 128 + k * per;
      if (n < N) {
        const TileOutRow orow = tile_out_row<CT>(e, n);
        for (int jj = et / cpr; jj < cn; jj += NT / cpr) {
          const uint32_t src = os_s + (uint32_t)((jj * 128 + k * per) * 4);
          uint4 o = lds_u128(src);
          if (ob != 4) {
            const uint4 hi = lds_u128(src + 16);
            const float f[8] = {__uint_as_float(o.x),  __uint_as_float(o.y),
                                __uint_as_float(o.z),  __uint_as_float(o.w),
                                __uint_as_float(hi.x), __uint_as_float(hi.y),
                                __uint_as_float(hi.z), __uint_as_float(hi.w)};
            union {
              uint4 u;
              CT c[8];
            } pk;
#pragma unroll
            for (int i = 0; i < 8; ++i) pk.c[i] = from_f<CT>(f[i]);
            o = pk.u;
          }
          *reinterpret_cast<uint4 *>(tile_out_ptr(orow, c0 + jj)) = o;
        }
      }
    }
    epi_bar_sync<NT>();  // the next chunk reuses the staging memory
  }
  if (go && S > 1 && et == 0) *cnt = 0;  // every other run of t has counted itself
}

}  // namespace he
