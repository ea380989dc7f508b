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

}  // namespace he
