// LoRA fuse of one projection into the fp16 tiled streaming layout with the rank-r
// product on the tensor cores: out = fp16(W + scale * B A) for W bf16 [rows][cols],
// A bf16 [r][cols], B bf16 [rows][r], r = 8 or 16 ("DeepSpeed-Chat: Easy, Fast and
// Affordable RLHF Training of ChatGPT-like Models at All Scales", §3.4 "Training
// Mode", Optimization 2: the weight is used as W + B A; the selection guide's §三: the
// LoRA weights are fused into the inference weights before generation).
//
// Work: 128 x 64 tiles of W.  Per tile, the delta B[n0..n0+128) A[:, k0..k0+64) is one
// tcgen05.mma (M = 128 rows, N = 64 columns, K = 16 with the factors zero-padded past r)
// into a 64-column TMEM accumulator, so the SIMT pipes only widen, add and round.
// Persistent CTAs (two per SM) walk tiles blockIdx.x, + gridDim.x, ...:
//   warp 8 (one thread)  TMA: the W tile (128-byte swizzle), the r x 64 block of A as
//                        16 zero-padded rows (the MMA's B operand, MN-major, 128-byte
//                        swizzle) and the 128 x r block of B as 16-element rows (the
//                        MMA's A operand, K-major, 32-byte swizzle), into a 4-stage ring
//   warp 9 (one thread)  the MMA of each tile into one of two TMEM accumulators
//   warps 0-7            warp w reads TMEM lanes 32 (w % 4) .. + 31 (tile rows) and
//                        columns 32 (w / 4) .. + 31 and the matching 64 bytes of its W row
//                        from shared memory, and writes fp16(w + scale * delta) back over
//                        them: the swizzled W tile (row n's logical 16-byte chunk c at
//                        c ^ (n % 8)) is already the order of the tiled output layout
//   warp 10 (one thread) stores each finished tile with one 16 KB bulk copy and hands
//                        the stage back to the producer once the copy has read it
// The products are exact in fp32 and summed by the tensor core in fp32, then one
// rounding to fp16.  Every wait is bounded; a timeout records DEVERR_WAIT_TIMEOUT, and
// each role drains what it issued before the CTA frees its TMEM and exits.
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.h"

namespace he {

bool make_tmap_2d_16sw(CUtensorMap *m, const void *ptr, int rows, int cols, int ld, int box_cols,
                       int box_rows, int swizzle_bytes, bool fp16);

namespace {

constexpr int FC_STAGES = 4;
constexpr int FC_W = 128 * 64 * 2;         // W tile, 128-byte swizzle
constexpr int FC_A = 16 * 128;             // A block: 16 rows of 64 columns
constexpr int FC_B = 128 * 32;             // B block: 128 rows of 16 factors
constexpr int FC_A_OFF = FC_W, FC_B_OFF = FC_W + FC_A;
constexpr int FC_STAGE = FC_W + FC_A + FC_B;  // 22528, a multiple of 1024
constexpr int FC_CONSUMER_WARPS = 8;
constexpr int FC_THREADS = (FC_CONSUMER_WARPS + 3) * 32;
constexpr int FC_PRODUCER = FC_CONSUMER_WARPS, FC_MMA = FC_CONSUMER_WARPS + 1,
              FC_STORER = FC_CONSUMER_WARPS + 2;
constexpr uint32_t FC_TCOLS = 128;         // two 64-column accumulators
constexpr int FC_NBAR = 3 * FC_STAGES + 2 * 2 + 1;
// + 1 KB slack at the end: operand descriptors stay inside the allocation whatever
// stride the hardware takes for an unused field
constexpr int FC_SMEM = 1024 + FC_STAGES * FC_STAGE + FC_NBAR * 8 + 16 + 1024;

// Bulk store shared -> global (16-byte aligned, size a multiple of 16), its commit
// group, and the waits: until at most N groups still read shared memory, or until at
// most N groups are still in flight at all.
__device__ __forceinline__ void bulk_store(void *gdst, const void *ssrc, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(
                   reinterpret_cast<uint64_t>(gdst)),
               "r"(smem_u32(ssrc)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
template <int N>
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void sts_u128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w));
}

// K-major, 32-byte swizzle: rows of 32 bytes (16 elements), 8-row atoms 256 bytes apart.
__device__ __forceinline__ uint64_t desc_k_sw32(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | ((uint64_t)(256 >> 4) << 32) |
         (1ull << 46) | (6ull << 61);
}
// MN-major, 128-byte swizzle: 128-byte lines of 64 N elements, 8 K lines per 1024-byte
// atom (stride byte offset); one 64-wide N group here (the leading offset is unused).
__device__ __forceinline__ uint64_t desc_mn_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(1024 >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | (1ull << 46) | (2ull << 61);
}
// kind::f16, D fp32, A and B bf16, A K-major, B MN-major, M = 128, N = 64.
constexpr uint32_t FC_IDESC = (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((64u >> 3) << 17) |
                              ((128u >> 4) << 24);

__global__ void __launch_bounds__(FC_THREADS, 2)
    k_fuse_tc(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_a,
              const __grid_constant__ CUtensorMap tm_b, uint4 *__restrict__ out, int rows,
              int cols, float scale, int *dev_err) {
  extern __shared__ uint8_t smraw[];
  uint8_t *sm = reinterpret_cast<uint8_t *>(
      (reinterpret_cast<uintptr_t>(smraw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + FC_STAGES * FC_STAGE);
  uint64_t *empty = full + FC_STAGES;
  uint64_t *d_full = empty + FC_STAGES;  // [2]
  uint64_t *d_empty = d_full + 2;        // [2]
  uint64_t *done = d_empty + 2;          // [STAGES]: the stage's output tile is written
  uint64_t *drain = done + FC_STAGES;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(drain + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KT = cols / 64;
  const long long T = (long long)(rows / 128) * KT;
  const long long first = blockIdx.x, step = gridDim.x;
  const long long n_mine = first < T ? (T - first + step - 1) / step : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < FC_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);  // the storer, once its bulk copy has read the stage
      mbar_init(&done[s], FC_CONSUMER_WARPS);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&d_full[b], 1);
      mbar_init(&d_empty[b], FC_CONSUMER_WARPS);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  }
  if (warp == FC_MMA) {
    tmem_alloc(tslot, FC_TCOLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;

  if (warp == FC_PRODUCER) {
    if (lane == 0) {
      prefetch_tmap(&tm_w);
      prefetch_tmap(&tm_a);
      prefetch_tmap(&tm_b);
      long long issued = 0;
      for (long long i = 0; i < n_mine; ++i) {
        const int s = (int)(i % FC_STAGES);
        if (i >= FC_STAGES &&
            !mbar_wait_bounded(&empty[s], (uint32_t)(((i / FC_STAGES) - 1) & 1))) {
          set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
          break;
        }
        const long long t = first + i * step;
        const int kx = (int)(t % KT) * 64, ny = (int)(t / KT) * 128;
        uint8_t *st = sm + s * FC_STAGE;
        mbar_arrive_expect_tx(&full[s], FC_STAGE);
        tma_load_2d(st, &tm_w, &full[s], kx, ny);
        tma_load_2d(st + FC_A_OFF, &tm_a, &full[s], kx, 0);  // rows r..15 read as zeros
        tma_load_2d(st + FC_B_OFF, &tm_b, &full[s], 0, ny);  // factors r..15 read as zeros
        issued = i + 1;
      }
      // no copy may still be landing when the CTA exits
      for (long long i = issued > FC_STAGES ? issued - FC_STAGES : 0; i < issued; ++i)
        if (!mbar_wait_bounded(&full[i % FC_STAGES], (uint32_t)((i / FC_STAGES) & 1))) {
          set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
          break;
        }
    }
  } else if (warp == FC_MMA) {
    if (lane == 0) {
      for (long long i = 0; i < n_mine; ++i) {
        const int s = (int)(i % FC_STAGES), b = (int)(i & 1);
        if (!mbar_wait_bounded(&full[s], (uint32_t)((i / FC_STAGES) & 1)) ||
            (i >= 2 && !mbar_wait_bounded(&d_empty[b], (uint32_t)(((i >> 1) - 1) & 1)))) {
          set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
          break;
        }
        tc_fence_after();
        const uint32_t st = smem_u32(sm + s * FC_STAGE);
        tc_mma_f16(tbase + (uint32_t)(b * 64), desc_k_sw32(st + FC_B_OFF),
                   desc_mn_sw128(st + FC_A_OFF), FC_IDESC, 0u);
        tc_commit(&d_full[b]);
      }
      tc_commit(drain);  // every MMA of this CTA complete before TMEM is freed
      if (!mbar_wait_bounded(drain, 0)) set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
    }
  } else if (warp == FC_STORER) {
    if (lane == 0) {
      long long stored = 0;
      for (long long i = 0; i < n_mine; ++i) {
        const int s = (int)(i % FC_STAGES);
        if (!mbar_wait_bounded(&done[s], (uint32_t)((i / FC_STAGES) & 1))) {
          set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
          break;
        }
        const long long t = first + i * step;
        bulk_store(out + t * 1024, sm + s * FC_STAGE, FC_W);
        bulk_commit();
        stored = i + 1;
        bulk_wait_read<1>();  // the copy of tile i - 1 has read its stage
        if (i >= 1) mbar_arrive(&empty[(i - 1) % FC_STAGES]);
      }
      bulk_wait_read<0>();
      if (stored >= 1) mbar_arrive(&empty[(stored - 1) % FC_STAGES]);
      bulk_wait_all<0>();  // every tile in global memory before the CTA exits
    }
  } else {
    // ---------------- consumers ----------------
    const int quarter = warp & 3, half = warp >> 2;
    const int n = quarter * 32 + lane;  // tile row = TMEM lane
    const uint32_t tl = ((uint32_t)(quarter * 32) << 16) + (uint32_t)(half * 32);
    for (long long i = 0; i < n_mine; ++i) {
      const int s = (int)(i % FC_STAGES), b = (int)(i & 1);
      if (!mbar_wait_bounded(&d_full[b], (uint32_t)((i >> 1) & 1))) {
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
        break;
      }
      tc_fence_after();
      uint32_t dr[32];
      tmem_ld32_nowait(tbase + (uint32_t)(b * 64) + tl, dr);
      const uint32_t wrow = smem_u32(sm + s * FC_STAGE) + (uint32_t)(n * 128);
      uint4 wv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        wv[q] = lds_u128(wrow + (uint32_t)((((half * 4 + q) ^ (n & 7))) * 16));
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&d_empty[b]);  // the accumulator may be reused
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t w4[4] = {wv[q].x, wv[q].y, wv[q].z, wv[q].w};
        uint32_t res[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float w0 = __uint_as_float(w4[e] << 16), w1 = __uint_as_float(w4[e] & 0xFFFF0000u);
          const float d0 = __uint_as_float(dr[q * 8 + 2 * e]);
          const float d1 = __uint_as_float(dr[q * 8 + 2 * e + 1]);
          __half2 hv = __floats2half2_rn(w0 + scale * d0, w1 + scale * d1);
          res[e] = *reinterpret_cast<uint32_t *>(&hv);
        }
        sts_u128(wrow + (uint32_t)((((half * 4 + q) ^ (n & 7))) * 16),
                 make_uint4(res[0], res[1], res[2], res[3]));
      }
      fence_proxy_async_smem();  // visible to the bulk copy that stores the tile
      __syncwarp();
      if (lane == 0) mbar_arrive(&done[s]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == FC_MMA) tmem_dealloc(tbase, FC_TCOLS);
}

}  // namespace

bool fuse_tc_supported(int r, const void *a, const void *bm) {
  return a != nullptr && bm != nullptr && (r == 8 || r == 16) && (uintptr_t)a % 16 == 0 &&
         (uintptr_t)bm % 16 == 0;
}

cudaError_t launch_fuse_tc(void *out, const void *src, const void *a, const void *bm, int rows,
                           int cols, int r, float scale, int num_sms, int *dev_err,
                           cudaStream_t st) {
  if (rows % 128 || cols % 64 || rows <= 0 || cols <= 0 || !fuse_tc_supported(r, a, bm))
    return cudaErrorInvalidValue;
  if ((uintptr_t)src % 16 || (uintptr_t)out % 16) return cudaErrorInvalidValue;
  const long long tiles = (long long)(rows / 128) * (cols / 64);
  CUtensorMap tw, ta, tb;
  if (!make_tmap_2d_16sw(&tw, src, rows, cols, cols, 64, 128, 128, false) ||
      !make_tmap_2d_16sw(&ta, a, r, cols, cols, 64, 16, 128, false) ||
      !make_tmap_2d_16sw(&tb, bm, rows, r, r, 16, 128, 32, false))
    return cudaErrorInvalidValue;
  cudaError_t e = ensure_smem_limit<k_fuse_tc>(FC_SMEM);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::min<long long>(tiles, 2LL * (num_sms > 0 ? num_sms : 148));
  k_fuse_tc<<<grid, FC_THREADS, FC_SMEM, st>>>(tw, ta, tb, (uint4 *)out, rows, cols, scale,
                                              dev_err);
  return cudaGetLastError();
}

}  // namespace he
