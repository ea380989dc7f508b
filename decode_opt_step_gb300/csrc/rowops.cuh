// Row helpers of the residual + LayerNorm kernels: the slice sums (in slot order, so
// every variant gives the same bits) and 16-byte parameter loads / output stores.
#pragma once
#include <type_traits>

#include "common.cuh"

namespace he {

// Sum of the split slices of one float4 of a row, in slice order (loads of four
// slices are issued together; the additions keep the order 0, 1, 2, ...).
__device__ __forceinline__ float4 sum_slices(const float *p, int split, long long stride) {
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int s = 0;
  for (; s + 4 <= split; s += 4) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = __ldcg(reinterpret_cast<const float4 *>(p + (s + u) * stride));
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      acc.x += v[u].x;
      acc.y += v[u].y;
      acc.z += v[u].z;
      acc.w += v[u].w;
    }
  }
  for (; s < split; ++s) {
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(p + s * stride));
    acc.x += v.x;
    acc.y += v.y;
    acc.z += v.z;
    acc.w += v.w;
  }
  return acc;
}

// The same sums for eight consecutive values of a row (two float4s at p): the loads
// of NB slices of both halves are issued together, so a row's slices arrive in
// ceil(split / NB) round trips; each half is still added in slice order 0, 1, 2, ...
template <int NB>
__device__ __forceinline__ void sum_slices8(const float *p, int split, long long stride,
                                            float4 &a0, float4 &a1) {
  a0 = make_float4(0.f, 0.f, 0.f, 0.f);
  a1 = a0;
  for (int s = 0; s < split; s += NB) {
    float4 v0[NB], v1[NB];
#pragma unroll
    for (int u = 0; u < NB; ++u)
      if (s + u < split) {
        v0[u] = __ldcg(reinterpret_cast<const float4 *>(p + (s + u) * stride));
        v1[u] = __ldcg(reinterpret_cast<const float4 *>(p + 4 + (s + u) * stride));
      }
#pragma unroll
    for (int u = 0; u < NB; ++u)
      if (s + u < split) {
        a0.x += v0[u].x;
        a0.y += v0[u].y;
        a0.z += v0[u].z;
        a0.w += v0[u].w;
        a1.x += v1[u].x;
        a1.y += v1[u].y;
        a1.z += v1[u].z;
        a1.w += v1[u].w;
      }
  }
}

// Eight consecutive parameters (16-bit: one 16-byte load; fp32: two).
template <typename PT>
__device__ __forceinline__ void load8(const PT *p, float (&v)[8]) {
  if constexpr (std::is_same<PT, float>::value) {
    const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
    const float4 b = __ldg(reinterpret_cast<const float4 *>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  } else {
    const uint4 u = __ldg(reinterpret_cast<const uint4 *>(p));
    const PT *e = reinterpret_cast<const PT *>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = to_f<PT>(e[i]);
  }
}

template <typename OT>
__device__ __forceinline__ void store8(OT *p, const float (&v)[8]) {
  if constexpr (std::is_same<OT, float>::value) {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  } else {
    uint4 u;
    OT *e = reinterpret_cast<OT *>(&u);
#pragma unroll
    for (int i = 0; i < 8; ++i) e[i] = from_f<OT>(v[i]);
    *reinterpret_cast<uint4 *>(p) = u;
  }
}

}  // namespace he
