// Prefill (causal) attention on the 5th-generation tensor cores (tcgen05 + TMEM +
// TMA), sm_103a, for 16-bit activations and head sizes 64 and 128.
//
// One CTA = one (sequence b, head h) and 128 consecutive query positions (the UMMA
// M dimension; query row r of the block lives on TMEM lane r).  Key blocks of 128:
//   S  = Q K^T            tcgen05.mma, Q and K from shared memory (K-major), S fp32 in
//                         TMEM columns [0, 128)
//   P  = exp(S - m)       one thread per query row reads its S row from TMEM, applies
//                         the causal mask, updates the running maximum m and sum l, and
//                         writes P (16-bit, two keys per 32-bit column) back over the
//                         first 64 columns of S
//   O  = O * c + P V      the running output (fp32, TMEM columns [128, 128 + hd)) is
//                         rescaled by the thread that owns its row when m moved, then
//                         tcgen05.mma accumulates P (A operand read from TMEM) times V
//                         (B operand from shared memory, MN-major: V rows are keys)
// and at the end ctx = O / l.  Q, K and V tiles arrive by 3-D TMA (128-byte swizzle);
// the maps stop at the prompt length, so key rows past it read as zeros and no stale
// cache entry (possibly not a number) reaches the P V product.  The next key block is
// loaded while the current one is in use: K(kb+1) as soon as S(kb) is done, V(kb+1)
// once P(kb) V(kb) is done.  Thread 0 issues copies and MMAs; every wait is bounded
// and a timeout records DEVERR_WAIT_TIMEOUT, drains what is in flight, frees TMEM and
// returns.  Two CTAs share an SM (256 TMEM columns each), so one CTA's softmax
// overlaps the other's copies and MMAs.
//
// Scaling: q arrives already multiplied by 1 / sqrt(hd) (QKV epilogue), as in the
// other attention kernels.  Accumulation is fp32; P is rounded to the activation
// type for the P V product while l sums the unrounded fp32 values.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"

namespace he {

bool make_tmap_3d_16(CUtensorMap *m, const void *ptr, long long d0, long long d1, long long d2,
                     long long stride1_bytes, long long stride2_bytes, int box0, int box1,
                     bool fp16);

namespace {

constexpr int QB = 128;     // query rows per CTA (UMMA M)
constexpr int KBLK = 128;   // keys per block (N of Q K^T, K of P V)
constexpr int BOX = 16384;  // one 128-row x 64-column 16-bit TMA box
constexpr uint32_t TCOLS = 256, S_COL = 0, O_COL = 128;
constexpr int NBAR = 5;     // qk, v, s, o, drain

__device__ __forceinline__ void tma_load_3d(void *dst, const void *tmap, uint64_t *bar, int c0,
                                            int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// Shared-memory operand descriptors (128-byte swizzle, descriptor version 1).
// K-major: rows of 128 bytes (64 elements along K), 8-row atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t desc_kmajor(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
         (2ull << 61);
}
// MN-major: each 128-byte line holds 64 consecutive N elements of one K index, 8 lines
// (K indices) per 1024-byte atom; `lbo` = bytes between groups of 64 N elements,
// `sbo` = bytes between groups of 8 K indices.
__device__ __forceinline__ uint64_t desc_mnmajor(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: fp32 D, A and B of type T, M = 128, N = n; B
// MN-major when b_mn (A is K-major or read from TMEM).
template <typename T>
__host__ __device__ constexpr uint32_t idesc_attn(int n, bool b_mn) {
  constexpr uint32_t fmt = std::is_same<T, bf16>::value ? 1u : 0u;
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((b_mn ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(QB >> 4) << 24);
}

constexpr float kLog2e = 1.4426950408889634f;
// 2^x by the SFU's approximate base-2 exponential (ex2.approx; 2^-inf = 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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

template <int HD>
struct TcCfg {
  static constexpr int NB = HD / 64;         // TMA boxes per tile
  static constexpr int TILE = NB * BOX;      // one Q, K or V tile
  // V, K, Q tiles, then barriers; sized so that exactly two CTAs fit an SM (their
  // 2 x 256 TMEM columns fill it)
  static constexpr int USED = 1024 + 3 * TILE + 128;
  static constexpr int SMEM = USED > 80 * 1024 ? USED : 80 * 1024;
};

template <typename T, int HD>
__global__ void __launch_bounds__(128, 1)
    k_attn_prefill_tc(const __grid_constant__ CUtensorMap tm_q,
                      const __grid_constant__ CUtensorMap tm_k,
                      const __grid_constant__ CUtensorMap tm_v, T *__restrict__ ctx, int H,
                      int Lp, int *dev_err) {
  using C = TcCfg<HD>;
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t *sV = sm, *sK = sm + C::TILE, *sQ = sm + 2 * C::TILE;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sm + 3 * C::TILE);
  uint64_t *bar_qk = bars, *bar_v = bars + 1, *bar_s = bars + 2, *bar_o = bars + 3,
           *bar_drain = bars + 4;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(bars + NBAR);
  volatile int *sabort = reinterpret_cast<volatile int *>(tslot + 1);

  const int qb = (int)(gridDim.x - 1 - blockIdx.x);  // the longest key ranges first
  const int bh = blockIdx.y, b = bh / H, h = bh - b * H;
  const int d = H * HD;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rr = warp * 32 + lane;  // this thread's query row in the block (its TMEM lane)
  const int qrow = qb * QB + rr;
  const int nkb = qb + 1;           // causal: key blocks 0 .. qb
  const bool t0 = threadIdx.x == 0;

  if (t0) {
    for (int i = 0; i < NBAR; ++i) mbar_init(&bars[i], 1);
    *sabort = 0;
    fence_mbar_init();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 0) {
    tmem_alloc(tslot, TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  const uint32_t tS = tbase + S_COL, tO = tbase + O_COL;
  const uint32_t lrow = (uint32_t)(warp * 32) << 16;  // this warp's TMEM lane quarter

  // copies issued / completions consumed on bar_qk and bar_v (thread 0's bookkeeping,
  // used to drain in-flight copies on a timeout)
  int qk_issued = 0, qk_done = 0, v_issued = 0, v_done = 0;
  pdl_wait();  // q and the caches come from the QKV projection
  if (t0) {
    mbar_arrive_expect_tx(bar_qk, 2 * C::TILE);
#pragma unroll
    for (int j = 0; j < C::NB; ++j) {
      tma_load_3d(sQ + j * BOX, &tm_q, bar_qk, h * HD + 64 * j, qb * QB, b);
      tma_load_3d(sK + j * BOX, &tm_k, bar_qk, 64 * j, 0, bh);
    }
    mbar_arrive_expect_tx(bar_v, C::TILE);
#pragma unroll
    for (int j = 0; j < C::NB; ++j) tma_load_3d(sV + j * BOX, &tm_v, bar_v, 64 * j, 0, bh);
    qk_issued = 1;
    v_issued = 1;
  }

  constexpr uint32_t IDESC_S = idesc_attn<T>(KBLK, false);
  constexpr uint32_t IDESC_PV = idesc_attn<T>(HD, true);
  float m = -INFINITY, l = 0.f;
  bool ok = true;
  for (int kb = 0; kb < nkb; ++kb) {
    // ---- S = Q K(kb)^T (thread 0) ----
    if (t0) {
      bool w = mbar_wait_bounded(bar_qk, (uint32_t)(kb & 1));
      if (w) ++qk_done;
      if (w && kb > 0) {
        // P(kb-1) V(kb-1) done: the S columns and the V tile are free
        w = mbar_wait_bounded(bar_o, (uint32_t)((kb - 1) & 1));
        if (w) {
          mbar_arrive_expect_tx(bar_v, C::TILE);
#pragma unroll
          for (int j = 0; j < C::NB; ++j)
            tma_load_3d(sV + j * BOX, &tm_v, bar_v, 64 * j, kb * KBLK, bh);
          ++v_issued;
        }
      }
      if (!w) {
        *sabort = 1;
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
      } else {
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t off = (uint32_t)((kk >> 2) * BOX + (kk & 3) * 32);
          tc_mma_f16(tS, desc_kmajor(smem_u32(sQ) + off), desc_kmajor(smem_u32(sK) + off),
                     IDESC_S, kk > 0 ? 1u : 0u);
        }
      }
      tc_commit(bar_s);  // also on a timeout, so that the other threads are released
    }
    if (!mbar_wait_bounded(bar_s, (uint32_t)(kb & 1))) {
      *sabort = 1;
      set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
    }
    tc_fence_after();
    __syncthreads();
    if (*sabort) {
      ok = false;
      break;
    }
    // K(kb) has been consumed: fetch K(kb+1) while this block's softmax runs
    if (t0 && kb + 1 < nkb) {
      mbar_arrive_expect_tx(bar_qk, C::TILE);
#pragma unroll
      for (int j = 0; j < C::NB; ++j)
        tma_load_3d(sK + j * BOX, &tm_k, bar_qk, 64 * j, (kb + 1) * KBLK, bh);
      ++qk_issued;
    }

    // ---- softmax of this thread's row ----
    float s[KBLK];
    {
      uint32_t r[KBLK / 32][32];
#pragma unroll
      for (int c = 0; c < KBLK / 32; ++c) tmem_ld32_nowait(tS + lrow + (uint32_t)(c * 32), r[c]);
      tmem_wait_ld();
#pragma unroll
      for (int c = 0; c < KBLK / 32; ++c)
#pragma unroll
        for (int i = 0; i < 32; ++i) s[c * 32 + i] = __uint_as_float(r[c][i]);
    }
    const int last = kb == qb ? rr : KBLK - 1;  // keys past the query are masked
    // maximum and sum over eight independent partials (short dependency chains)
    float ma[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) ma[i] = m;
#pragma unroll
    for (int c = 0; c < KBLK; ++c) {
      if (c > last) s[c] = -INFINITY;
      ma[c & 7] = fmaxf(ma[c & 7], s[c]);
    }
    const float mx = fmaxf(fmaxf(fmaxf(ma[0], ma[1]), fmaxf(ma[2], ma[3])),
                           fmaxf(fmaxf(ma[4], ma[5]), fmaxf(ma[6], ma[7])));
    // key kb*128 precedes every query of the block, so mx is finite
    const float corr = ex2_approx((m - mx) * kLog2e);
    m = mx;
    const float mxl = mx * kLog2e;
    float ra[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) ra[i] = 0.f;
#pragma unroll
    for (int c = 0; c < KBLK / 32; ++c) {
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float p0 = ex2_approx(fmaf(s[c * 32 + 2 * i], kLog2e, -mxl));
        const float p1 = ex2_approx(fmaf(s[c * 32 + 2 * i + 1], kLog2e, -mxl));
        ra[i & 7] += p0 + p1;
        pk[i] = pack2<T>(p0, p1);
      }
      tmem_st16(tS + lrow + (uint32_t)(c * 16), pk);  // over S columns already read
    }
    l = l * corr + (((ra[0] + ra[1]) + (ra[2] + ra[3])) + ((ra[4] + ra[5]) + (ra[6] + ra[7])));
    if (kb > 0 && __any_sync(0xffffffffu, corr != 1.f)) {
      // the previous P V is complete (S(kb) was issued after it), so O is stable
#pragma unroll
      for (int c = 0; c < HD / 32; ++c) {
        uint32_t r[32];
        tmem_ld32_nowait(tO + lrow + (uint32_t)(c * 32), r);
        tmem_wait_ld();
        uint32_t lo[16], hi[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          lo[i] = __float_as_uint(__uint_as_float(r[i]) * corr);
          hi[i] = __float_as_uint(__uint_as_float(r[16 + i]) * corr);
        }
        tmem_st16(tO + lrow + (uint32_t)(c * 32), lo);
        tmem_st16(tO + lrow + (uint32_t)(c * 32 + 16), hi);
      }
    }
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();

    // ---- O += P V(kb) (thread 0) ----
    if (t0) {
      tc_fence_after();
      if (!mbar_wait_bounded(bar_v, (uint32_t)(kb & 1))) {
        *sabort = 1;
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
      } else {
        ++v_done;
#pragma unroll
        for (int kk = 0; kk < KBLK / 16; ++kk)
          tc_mma_f16_tmem_a(tO, tS + (uint32_t)(kk * 8),
                            desc_mnmajor(smem_u32(sV) + (uint32_t)(kk * 2048), BOX, 1024),
                            IDESC_PV, (kb > 0 || kk > 0) ? 1u : 0u);
      }
      tc_commit(bar_o);
    }
  }
  pdl_trigger();

  // ---- ctx = O / l ----
  if (ok) {
    if (!mbar_wait_bounded(bar_o, (uint32_t)((nkb - 1) & 1))) {
      set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
      ok = false;
    }
  }
  tc_fence_after();
  if (__all_sync(0xffffffffu, ok)) {
    const float inv = 1.f / l;
    T *dst = ctx + ((long long)b * Lp + qrow) * d + h * HD;
#pragma unroll
    for (int c = 0; c < HD / 32; ++c) {
      uint32_t r[32];
      tmem_ld32_nowait(tO + lrow + (uint32_t)(c * 32), r);
      tmem_wait_ld();
      if (qrow < Lp) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          pk[i] = pack2<T>(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
        uint4 *o4 = reinterpret_cast<uint4 *>(dst + c * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          o4[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
      }
    }
  }

  // ---- teardown: every MMA and copy of this CTA finished, then TMEM freed ----
  if (t0) {
    tc_commit(bar_drain);
    if (!mbar_wait_bounded(bar_drain, 0)) set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
    for (; qk_done < qk_issued; ++qk_done)
      if (!mbar_wait_bounded(bar_qk, (uint32_t)(qk_done & 1))) break;
    for (; v_done < v_issued; ++v_done)
      if (!mbar_wait_bounded(bar_v, (uint32_t)(v_done & 1))) break;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tbase, TCOLS);
}

template <typename T, int HD>
cudaError_t run(const void *q, const void *kc, const void *vc, void *ctx, int B, int Lp, int H,
                int max_seq, int *dev_err, cudaStream_t st) {
  using C = TcCfg<HD>;
  constexpr bool fp16 = std::is_same<T, f16>::value;
  const int d = H * HD;
  CUtensorMap tq, tk, tv;
  // q: [B][Lp][d]; caches: [B*H][max_seq][HD], read up to the prompt length
  if (!make_tmap_3d_16(&tq, q, d, Lp, B, (long long)d * 2, (long long)Lp * d * 2, 64, QB, fp16) ||
      !make_tmap_3d_16(&tk, kc, HD, Lp, (long long)B * H, HD * 2, (long long)max_seq * HD * 2, 64,
                       KBLK, fp16) ||
      !make_tmap_3d_16(&tv, vc, HD, Lp, (long long)B * H, HD * 2, (long long)max_seq * HD * 2, 64,
                       KBLK, fp16))
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem_limit<k_attn_prefill_tc<T, HD>>(C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((Lp + QB - 1) / QB, B * H);
  return launch_k(k_attn_prefill_tc<T, HD>, grid, dim3(128), (size_t)C::SMEM, st, g_pdl, tq, tk,
                  tv, (T *)ctx, H, Lp, dev_err);
}

}  // namespace

bool attn_prefill_tc_supported(int act, int hd) {
  return (act == ACT_BF16 || act == ACT_F16) && (hd == 64 || hd == 128);
}

cudaError_t launch_attn_prefill_tc(int act, const void *q, const void *kc, const void *vc,
                                   void *ctx, int B, int Lp, int H, int hd, int max_seq,
                                   int *dev_err, cudaStream_t st) {
  if (B < 1 || H < 1 || Lp < 1 || Lp > max_seq) return cudaErrorInvalidValue;
  if ((uintptr_t)q % 16 || (uintptr_t)kc % 16 || (uintptr_t)vc % 16 || (uintptr_t)ctx % 16)
    return cudaErrorInvalidValue;
  auto go = [&](auto tag) -> cudaError_t {
    using T = decltype(tag);
    if (hd == 128) return run<T, 128>(q, kc, vc, ctx, B, Lp, H, max_seq, dev_err, st);
    if (hd == 64) return run<T, 64>(q, kc, vc, ctx, B, Lp, H, max_seq, dev_err, st);
    return cudaErrorInvalidValue;
  };
  if (act == ACT_BF16) return go(bf16{});
  if (act == ACT_F16) return go(f16{});
  return cudaErrorInvalidValue;
}

}  // namespace he
