// Prefill (causal) attention for bf16 or fp16 on tensor cores (mma.sync m16n8k16, fp32
// accumulation), flash-style: one CTA = 4 warps = 64 queries of one (b, h); key
// and value blocks of 64 rows are staged in shared memory (rows padded by 16
// bytes so ldmatrix reads are conflict-free), two blocks in flight: the next
// block's asynchronous copies (cp.async) run while the current one is used; the
// query tile passes through the second buffer first.  Scores, the running softmax
// and the output stay in registers.  Scores S = Q K^T use ldmatrix fragments of Q
// (A, row-major) and K (B, "col" = K rows); the probabilities are re-packed from
// the S accumulators into A fragments for O += P V, with V read by ldmatrix.trans.
#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace he {

namespace {

__device__ __forceinline__ void ldm_x4(uint32_t (&r)[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldm_x4_t(uint32_t (&r)[4], const void *p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}
template <typename T>
__device__ __forceinline__ void mma_16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
  if constexpr (std::is_same<T, bf16>::value)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (std::is_same<T, bf16>::value) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
  }
}

// Asynchronous copy of a [64][HD] 16-bit tile (row stride `ld` elements; rows >= nrows
// are zero-filled, reading nothing) into shared memory with row stride HD + 8; one
// 16-byte cp.async per chunk, completed by cp.async.wait_group.
template <int HD>
__device__ __forceinline__ void load_tile_async(uint16_t *dst, const uint16_t *src, long long ld,
                                                int nrows) {
  constexpr int CH = HD / 8;  // 16-byte chunks per row
#pragma unroll
  for (int e = threadIdx.x; e < 64 * CH; e += 128) {
    const int r = e / CH, c = e - r * CH;
    const bool ok = r < nrows;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(
                     smem_u32(dst + r * (HD + 8) + c * 8)),
                 "l"(src + (ok ? (long long)r * ld : 0) + c * 8), "r"(ok ? 16 : 0)
                 : "memory");
  }
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <typename T, int HD>
__global__ void __launch_bounds__(128, 3)  // three CTAs (and their 70 KB of tiles) per SM
    k_attn_prefill_mma(const uint16_t *__restrict__ q, const uint16_t *__restrict__ kc,
                       const uint16_t *__restrict__ vc, T *__restrict__ ctx, int H, int Lp,
                       int max_seq) {
  constexpr int LD = HD + 8;
  constexpr int KS = HD / 16;  // k-steps of Q K^T
  constexpr int DT = HD / 8;   // 8-wide output tiles
  extern __shared__ __align__(16) uint8_t smraw[];
  // two (K, V) buffers of 64 x LD each; the query tile is staged in buffer 1's K
  uint16_t *const kbuf0 = reinterpret_cast<uint16_t *>(smraw);
  const int bstride = 2 * 64 * LD;  // elements per (K, V) buffer
  const int qb = blockIdx.x, bh = blockIdx.y;
  const int b = bh / H, h = bh - b * H;
  const int d = H * HD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, tg = lane & 3;
  const long long row0 = ((long long)b * H + h) * max_seq;

  pdl_wait();
  uint16_t *qs = kbuf0 + bstride;
  load_tile_async<HD>(qs, q + ((long long)b * Lp + qb * 64) * d + h * HD, d, Lp - qb * 64);
  cp_commit();
  load_tile_async<HD>(kbuf0, kc + row0 * HD, HD, min(64, Lp));
  load_tile_async<HD>(kbuf0 + 64 * LD, vc + row0 * HD, HD, min(64, Lp));
  cp_commit();
  cp_wait<1>();  // this thread's query copies
  __syncthreads();
  // Q fragments of this warp's 16 rows, all k-steps
  uint32_t qa[KS][4];
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) {
    const int r = warp * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
    const int c = kk * 16 + 8 * (lane >> 4);
    ldm_x4(qa[kk], qs + r * LD + c);
  }
  __syncthreads();  // buffer 1 is free for key block 1
  float o[DT][4];
#pragma unroll
  for (int i = 0; i < DT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int tq0 = qb * 64 + warp * 16 + g;  // query positions of rows g and g + 8
  const int tq1 = tq0 + 8;

  for (int kb = 0; kb <= qb; ++kb) {
    if (kb < qb) {  // the next key block into the other buffer, then wait for this one
      uint16_t *nb = kbuf0 + ((kb + 1) & 1) * bstride;
      const int nk = min(64, Lp - (kb + 1) * 64);
      load_tile_async<HD>(nb, kc + (row0 + (kb + 1) * 64) * HD, HD, nk);
      load_tile_async<HD>(nb + 64 * LD, vc + (row0 + (kb + 1) * 64) * HD, HD, nk);
      cp_commit();
      cp_wait<1>();
    } else {
      cp_wait<0>();
    }
    __syncthreads();  // every thread's copies of this block have landed
    const uint16_t *ks = kbuf0 + (kb & 1) * bstride;
    const uint16_t *vs = ks + 64 * LD;
    // S = Q K^T for 64 keys: 8 n-tiles of 8 keys
    float s[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.f;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
#pragma unroll
      for (int jp = 0; jp < 4; ++jp) {  // pairs of n-tiles (16 keys)
        uint32_t kf[4];
        const int r = jp * 16 + (lane & 7) + 8 * (lane >> 4);
        const int c = kk * 16 + 8 * ((lane >> 3) & 1);
        ldm_x4(kf, ks + r * LD + c);
        mma_16<T>(s[2 * jp], qa[kk], kf[0], kf[1]);
        mma_16<T>(s[2 * jp + 1], qa[kk], kf[2], kf[3]);
      }
    }
    // causal mask and running max
    float mx0 = m0, mx1 = m1;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int tk = kb * 64 + j * 8 + 2 * tg;
      if (tk > tq0) s[j][0] = -INFINITY;
      if (tk + 1 > tq0) s[j][1] = -INFINITY;
      if (tk > tq1) s[j][2] = -INFINITY;
      if (tk + 1 > tq1) s[j][3] = -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(s[j][0], s[j][1]));
      mx1 = fmaxf(mx1, fmaxf(s[j][2], s[j][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    // key kb*64 <= every query of this block, so mx0 and mx1 are finite
    const float c0 = expf(m0 - mx0), c1 = expf(m1 - mx1);
    m0 = mx0;
    m1 = mx1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      s[j][0] = expf(s[j][0] - mx0);
      s[j][1] = expf(s[j][1] - mx0);
      s[j][2] = expf(s[j][2] - mx1);
      s[j][3] = expf(s[j][3] - mx1);
      rs0 += s[j][0] + s[j][1];
      rs1 += s[j][2] + s[j][3];
    }
    l0 = l0 * c0 + rs0;  // per-thread partial row sums (reduced over the quad at the end)
    l1 = l1 * c1 + rs1;
#pragma unroll
    for (int i = 0; i < DT; ++i) {
      o[i][0] *= c0;
      o[i][1] *= c0;
      o[i][2] *= c1;
      o[i][3] *= c1;
    }
    // O += P V: 4 k-steps of 16 keys
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack2<T>(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack2<T>(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack2<T>(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack2<T>(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < DT / 2; ++dp) {  // pairs of 8-wide output tiles
        uint32_t vf[4];
        const int r = kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1);
        const int c = dp * 16 + 8 * (lane >> 4);
        ldm_x4_t(vf, vs + r * LD + c);
        mma_16<T>(o[2 * dp], pa, vf[0], vf[1]);
        mma_16<T>(o[2 * dp + 1], pa, vf[2], vf[3]);
      }
    }
    __syncthreads();  // this buffer is refilled at the next block
  }
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  const float i0 = 1.f / l0, i1 = 1.f / l1;
#pragma unroll
  for (int i = 0; i < DT; ++i) {
    const int c = h * HD + i * 8 + 2 * tg;
    if (tq0 < Lp)
      *reinterpret_cast<uint32_t *>(ctx + ((long long)b * Lp + tq0) * d + c) =
          pack2<T>(o[i][0] * i0, o[i][1] * i0);
    if (tq1 < Lp)
      *reinterpret_cast<uint32_t *>(ctx + ((long long)b * Lp + tq1) * d + c) =
          pack2<T>(o[i][2] * i1, o[i][3] * i1);
  }
}

template <typename T, int HD>
cudaError_t run(const void *q, const void *kc, const void *vc, void *ctx, int B, int Lp, int H,
                int max_seq, cudaStream_t st) {
  const size_t sm = (size_t)4 * 64 * (HD + 8) * sizeof(uint16_t);
  cudaError_t e = ensure_smem_limit<k_attn_prefill_mma<T, HD>>((int)sm);
  if (e != cudaSuccess) return e;
  dim3 grid((Lp + 63) / 64, B * H);
  return launch_k(k_attn_prefill_mma<T, HD>, grid, dim3(128), sm, st, g_pdl, (const uint16_t *)q,
                  (const uint16_t *)kc, (const uint16_t *)vc, (T *)ctx, H, Lp, max_seq);
}

}  // namespace

cudaError_t launch_attn_prefill_mma(int act, const void *q, const void *kc, const void *vc,
                                    void *ctx, int B, int Lp, int H, int hd, int max_seq,
                                    cudaStream_t st) {
  auto go = [&](auto tag) -> cudaError_t {
    using T = decltype(tag);
    if (hd == 128) return run<T, 128>(q, kc, vc, ctx, B, Lp, H, max_seq, st);
    if (hd == 64) return run<T, 64>(q, kc, vc, ctx, B, Lp, H, max_seq, st);
    if (hd == 32) return run<T, 32>(q, kc, vc, ctx, B, Lp, H, max_seq, st);
    return cudaErrorInvalidValue;
  };
  if (act == ACT_BF16) return go(bf16{});
  if (act == ACT_F16) return go(f16{});
  return cudaErrorInvalidValue;
}

}  // namespace he
