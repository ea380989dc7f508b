// bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), sm_103a.
//
// C[tok][n] = sum_k X[tok][k] * W[n][k] with both operands K-major, as nn.Linear
// stores them.  The weight is the UMMA A operand (M = 128 output features per
// tile) and the activations are the B operand (N = up to 256 tokens per tile):
// in decode the token count is the batch, so a tile streams 128 weight rows once
// for every sequence of the batch.  Accumulators live in TMEM (fp32, one lane
// per output feature, one column per token).
//
// Warp roles (192 threads): warps 0-3 read TMEM and run the epilogue (warp w
// owns TMEM lanes 32w..32w+31), warp 4 issues TMA loads into a STAGES-deep ring
// of 128B-swizzled tiles, warp 5 owns the TMEM allocation and one elected thread
// issues tcgen05.mma.  Every mbarrier wait is bounded; on a timeout the kernel
// records DEVERR_WAIT_TIMEOUT, stops issuing, drains its own copies and frees
// its TMEM.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "row_epilogue.cuh"

namespace he {

namespace {

constexpr int BM = 128;        // UMMA M: output features per tile
constexpr int BK = 64;         // K per stage: one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;     // K per tcgen05.mma (kind::f16)
constexpr int A_BYTES = BM * BK * 2;

// UMMA shared-memory descriptor, K-major operand with 128-byte swizzle: rows of
// 128 bytes, 8-row atoms of 1024 bytes (stride byte offset), version 1, swizzle
// mode 2 (128B).  The leading byte offset is unused for this layout.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
         (2ull << 61);
}

// Instruction descriptor, kind::f16: D fp32, A and B both bf16 (format 1) or both
// fp16 (format 0), both K-major, M = 128.
template <typename CT>
__host__ __device__ constexpr uint32_t idesc_f16kind(int n) {
  constexpr uint32_t fmt = std::is_same<CT, bf16>::value ? 1u : 0u;
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(BM >> 4) << 24);
}

constexpr uint32_t tmem_cols_for(int bn) { return bn <= 32 ? 32u : (bn <= 64 ? 64u : (bn <= 128 ? 128u : 256u)); }

template <int BN, int STAGES>
struct Cfg {
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int SMEM = 1024 /*align slack*/ + STAGES * STAGE_BYTES + 256;
  static constexpr uint32_t TMEM_COLS = tmem_cols_for(BN);
};

struct WTiles {
  const uint16_t *p[3];  // tiled weights of each row group (ABULK), 16-bit elements
  int kt;                // 64-wide k tiles per 128-row tile row
  // per-row scales of each row group, or null: the weights hold fp8 codes (as exact
  // 16-bit values) and output row n is scaled by its group's scale[n - group start]
  const float *scale[3];
  int group_rows;
};

// The scale of output feature `row` (1 without scales).
__device__ __forceinline__ float wt_row_scale(const WTiles &wt, int row, int N) {
  if (!wt.scale[0] || row >= N) return 1.f;
  const int g = wt.group_rows > 0 ? row / wt.group_rows : 0;
  return wt.scale[g][row - g * wt.group_rows];
}

template <typename CT, int BN, int STAGES, bool ABULK>
__global__ void __launch_bounds__(192, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
              const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_x,
              int tiles_per_group, int M, int N, int kb_total, int kb_per_split,
              const __grid_constant__ Epi epi, WTiles wt, int *dev_err) {
  using C = Cfg<BN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t *smA = base;                                   // STAGES x A tile
  uint8_t *smB = base + STAGES * A_BYTES;                // STAGES x B tile
  uint64_t *full = reinterpret_cast<uint64_t *>(base + STAGES * C::STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *accum = empty + STAGES;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(accum + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x, n_tile = blockIdx.y, split = blockIdx.z;
  const int kb0 = split * kb_per_split;
  const int nkb = min(kb_per_split, kb_total - kb0);

  if (warp == 4 && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accum, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();

  if (warp == 4 && lane == 0) {
    // ---------------- TMA producer ----------------
    const int group = m_tile / tiles_per_group;
    const CUtensorMap *tw = group == 0 ? &tm_w0 : (group == 1 ? &tm_w1 : &tm_w2);
    const int m_row = (m_tile - group * tiles_per_group) * BM;
    if (!ABULK) prefetch_tmap(tw);
    prefetch_tmap(&tm_x);
    pdl_wait();
    // tiled weights: this CTA's k-blocks of tile row `m_row / BM` are contiguous
    const uint16_t *wtile =
        ABULK ? wt.p[group] + ((long long)(m_row / BM) * wt.kt + kb0) * (BM * BK) : nullptr;
    int issued = 0;
    for (int i = 0; i < nkb; ++i) {
      const int s = i % STAGES;
      if (i >= STAGES && !mbar_wait_bounded(&empty[s], ((i / STAGES) - 1) & 1)) {
        *abort_flag = 1;
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
        break;
      }
      if (*(volatile int *)abort_flag) break;
      mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
      const int kc = (kb0 + i) * BK;
      if (ABULK)
        bulk_load(smA + s * A_BYTES, wtile + (long long)i * (BM * BK), A_BYTES, &full[s]);
      else
        tma_load_2d(smA + s * A_BYTES, tw, &full[s], kc, m_row);
      tma_load_2d(smB + s * C::B_BYTES, &tm_x, &full[s], kc, n_tile * BN);
      issued = i + 1;
    }
    // Drain: the last load issued into each stage must have landed before exit.
    for (int i = max(0, issued - STAGES); i < issued; ++i)
      if (!mbar_wait_bounded(&full[i % STAGES], (i / STAGES) & 1))
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
  } else if (warp == 5 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = idesc_f16kind<CT>(BN);
    for (int i = 0; i < nkb; ++i) {
      const int s = i % STAGES;
      if (!mbar_wait_bounded(&full[s], (i / STAGES) & 1)) {
        *(volatile int *)abort_flag = 1;
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
        break;
      }
      if (*(volatile int *)abort_flag) break;
      tc_fence_after();
      const uint32_t a0 = smem_u32(smA + s * A_BYTES);
      const uint32_t b0 = smem_u32(smB + s * C::B_BYTES);
#pragma unroll
      for (int kk = 0; kk < BK / UMMA_K; ++kk)
        tc_mma_f16(tmem_base, sdesc_sw128(a0 + kk * UMMA_K * 2), sdesc_sw128(b0 + kk * UMMA_K * 2),
                   idesc, (i | kk) != 0);
      tc_commit(&empty[s]);  // frees the stage once these MMAs have read it
    }
    tc_commit(accum);        // arrives when every MMA issued above is complete
  } else if (warp < 4) {
    // ---------------- epilogue ----------------
    pdl_wait();
    const bool ok = mbar_wait_bounded(accum, 0);
    if (!ok) set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
    tc_fence_after();
    const bool live = ok && !*(volatile int *)abort_flag && nkb > 0;
    const int row = m_tile * BM + warp * 32 + lane;  // output feature n
    const uint32_t tl = tmem_base + ((uint32_t)(warp * 32) << 16);
    constexpr int W = BN >= 32 ? 32 : 16;
    const bool part = epi.kind == EPI_PARTIAL;
    const RowEpi<CT> re = row_epi_prepare<CT>(epi, row < N ? row : 0, part ? epi.partial : nullptr,
                                              epi.split_stride, split, epi.ldp);
    const int tok_base = n_tile * BN;
    const float rs = wt_row_scale(wt, row, N);
#pragma unroll 1
    for (int c0 = 0; c0 < BN; c0 += W) {
      float v[W];
      tmem_load_cols<W>(tl + c0, v);
#pragma unroll
      for (int j = 0; j < W; ++j) v[j] *= rs;
      if (live && row < N && tok_base + c0 < M)
        row_epi_store<CT, W>(re, tok_base + c0, min(W, M - tok_base - c0), v);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------------------
// Persistent variant for many tiles (prefill: every prompt token at once).  One
// CTA per SM walks the (128-feature, 256-token) tiles c, c + P, c + 2P, ... in an
// order that groups kTokGroup token tiles, so the tiles in flight at one time
// share operands in L2 (about 19 weight tiles x 8 token tiles per wave).  Two
// TMEM accumulators (2 x 256 columns): the epilogue of one tile runs while the
// MMAs of the next one accumulate, and the load ring never drains between tiles.
// ---------------------------------------------------------------------------
constexpr int PBN = 256, PSTAGES = 4, kTokGroup = 8;

__host__ __device__ inline void tcp_tile(long long L, int MT, int NT, int *mt, int *nt) {
  const long long gsz = (long long)kTokGroup * MT;
  const long long g = L / gsz, rem = L - g * gsz;
  const int gnt = min(kTokGroup, NT - (int)g * kTokGroup);  // the last group may be narrower
  *mt = (int)(rem / gnt);
  *nt = (int)g * kTokGroup + (int)(rem % gnt);
}

// PAIR: CTAs run in clusters of two on weight tiles 2m and 2m + 1 of the same token
// tile; each loads its own weight tile and half of the token tile, multicast into both
// CTAs' shared memory, so the pair reads the activations from L2 once, and each MMA
// releases a stage in both CTAs (multicast commit).
template <typename CT, bool ABULK, bool PAIR>
__global__ void __launch_bounds__(192, 1)
    k_gemm_tcp(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
               const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_x,
               int tiles_per_group, int M, int N, int kb_total, int MT, int NT,
               const __grid_constant__ Epi epi, WTiles wt, int *dev_err) {
  using C = Cfg<PBN, PSTAGES>;
  constexpr uint32_t kCols = 2 * PBN;  // two accumulators
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t *smA = base;
  uint8_t *smB = base + PSTAGES * A_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(base + PSTAGES * C::STAGE_BYTES);
  uint64_t *empty = full + PSTAGES;
  uint64_t *acc_full = empty + PSTAGES;  // [2]
  uint64_t *acc_empty = acc_full + 2;    // [2]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + 2);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = PAIR ? (int)(blockIdx.x & 1) : 0;  // rank in the cluster of two
  const int P = PAIR ? (int)(gridDim.x >> 1) : (int)gridDim.x;
  const int c = PAIR ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
  const int MTL = PAIR ? MT / 2 : MT;  // weight tiles (pairs of tiles) in the tile order
  const long long T = (long long)MTL * NT;
  auto tile_of = [&](long long L, int *mt, int *nt) {
    tcp_tile(L, MTL, NT, mt, nt);
    if (PAIR) *mt = 2 * *mt + rank;
  };

  if (warp == 4 && lane == 0) {
    for (int s = 0; s < PSTAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], PAIR ? 2 : 1);  // the MMAs of both CTAs read a stage's token half
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 4);  // one arrival per epilogue warp
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 5) {
    tmem_alloc(tmem_slot, kCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // the peer's barriers exist before anything targets them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();

  if (warp == 4 && lane == 0) {
    // ---------------- TMA producer ----------------
    if (!ABULK) {
      prefetch_tmap(&tm_w0);
      prefetch_tmap(&tm_w1);
      prefetch_tmap(&tm_w2);
    }
    prefetch_tmap(&tm_x);
    pdl_wait();  // the activations come from the kernel before this one
    long long it = 0, issued = 0;
    bool stop = false;
    for (long long L = c; L < T && !stop; L += P) {
      int mt, nt;
      tile_of(L, &mt, &nt);
      const int group = mt / tiles_per_group;
      const CUtensorMap *tw = group == 0 ? &tm_w0 : (group == 1 ? &tm_w1 : &tm_w2);
      const int m_row = (mt - group * tiles_per_group) * BM;
      const uint16_t *wtile =
          ABULK ? wt.p[group] + (long long)(m_row / BM) * wt.kt * (BM * BK) : nullptr;
      for (int kb = 0; kb < kb_total; ++kb, ++it) {
        const int s = (int)(it % PSTAGES);
        if (it >= PSTAGES && !mbar_wait_bounded(&empty[s], (uint32_t)((it / PSTAGES - 1) & 1))) {
          *(volatile int *)abort_flag = 1;
          set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
          stop = true;
          break;
        }
        if (*(volatile int *)abort_flag) {
          stop = true;
          break;
        }
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        if (ABULK)
          bulk_load(smA + s * A_BYTES, wtile + (long long)kb * (BM * BK), A_BYTES, &full[s]);
        else
          tma_load_2d(smA + s * A_BYTES, tw, &full[s], kb * BK, m_row);
        if (PAIR)  // this CTA's half of the token tile, into both CTAs
          tma_load_2d_mc(smB + s * C::B_BYTES + rank * (C::B_BYTES / 2), &tm_x, &full[s],
                         kb * BK, nt * PBN + rank * (PBN / 2), 0x3);
        else
          tma_load_2d(smB + s * C::B_BYTES, &tm_x, &full[s], kb * BK, nt * PBN);
        issued = it + 1;
      }
    }
    // the last load issued into each stage must have landed before exit
    for (long long i = issued > PSTAGES ? issued - PSTAGES : 0; i < issued; ++i)
      if (!mbar_wait_bounded(&full[i % PSTAGES], (uint32_t)((i / PSTAGES) & 1)))
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
  } else if (warp == 5 && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = idesc_f16kind<CT>(PBN);
    long long it = 0;
    int tcount = 0;
    bool ok = true;
    for (long long L = c; L < T && ok; L += P, ++tcount) {
      const int buf = tcount & 1;
      if (tcount >= 2 &&
          !mbar_wait_bounded(&acc_empty[buf], (uint32_t)(((tcount >> 1) - 1) & 1))) {
        *(volatile int *)abort_flag = 1;
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem_base + (uint32_t)(buf * PBN);
      for (int kb = 0; kb < kb_total; ++kb, ++it) {
        const int s = (int)(it % PSTAGES);
        if (!mbar_wait_bounded(&full[s], (uint32_t)((it / PSTAGES) & 1)) ||
            *(volatile int *)abort_flag) {
          *(volatile int *)abort_flag = 1;
          set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a0 = smem_u32(smA + s * A_BYTES);
        const uint32_t b0 = smem_u32(smB + s * C::B_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / UMMA_K; ++kk)
          tc_mma_f16(acc, sdesc_sw128(a0 + kk * UMMA_K * 2), sdesc_sw128(b0 + kk * UMMA_K * 2),
                     idesc, (kb | kk) != 0);
        if (PAIR)
          tc_commit_mc(&empty[s], 0x3);
        else
          tc_commit(&empty[s]);
      }
      tc_commit(&acc_full[buf]);  // also issued on abort so the epilogue is released
    }
  } else if (warp < 4) {
    // ---------------- epilogue ----------------
    pdl_wait();  // outputs may still be read by the kernel before this one
    constexpr int W = 32;
    const bool part = epi.kind == EPI_PARTIAL;
    int tcount = 0;
    for (long long L = c; L < T; L += P, ++tcount) {
      if (*(volatile int *)abort_flag) break;
      int mt, nt;
      tile_of(L, &mt, &nt);
      const int buf = tcount & 1;
      const bool ok = mbar_wait_bounded(&acc_full[buf], (uint32_t)((tcount >> 1) & 1));
      if (!ok) {
        *(volatile int *)abort_flag = 1;
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
      }
      tc_fence_after();
      const bool live = ok && !*(volatile int *)abort_flag;
      const int row = mt * BM + warp * 32 + lane;  // output feature n
      const uint32_t tl = tmem_base + ((uint32_t)(warp * 32) << 16) + (uint32_t)(buf * PBN);
      const RowEpi<CT> re = row_epi_prepare<CT>(epi, row < N ? row : 0,
                                                part ? epi.partial : nullptr, epi.split_stride,
                                                0, epi.ldp);
      const int tok_base = nt * PBN;
      const float rs = wt_row_scale(wt, row, N);
#pragma unroll 1
      for (int c0 = 0; c0 < PBN; c0 += W) {
        float v[W];
        tmem_load_cols<W>(tl + c0, v);
#pragma unroll
        for (int j = 0; j < W; ++j) v[j] *= rs;
        if (live && row < N && tok_base + c0 < M)
          row_epi_store<CT, W>(re, tok_base + c0, min(W, M - tok_base - c0), v);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acc_empty[buf]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();  // no CTA leaves while its peer may still signal or fill it
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kCols);
  }
}

// ---------------------------------------------------------------------------
// Host side: tensor maps and launch.
// ---------------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D bf16 map over a [rows][cols] matrix with row stride `ld` elements, box
// {64 (K), box_rows}, 128-byte swizzle, zero fill out of bounds.
bool make_tmap(CUtensorMap *m, const void *ptr, int rows, int cols, int ld, int box_rows,
               CUtensorMapDataType dt = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, dt, 2, const_cast<void *>(ptr), dims, strides,
                   box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename CT>
constexpr CUtensorMapDataType tmap_type() {
  return std::is_same<CT, bf16>::value ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                       : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
}

template <typename CT, int BN, int STAGES, bool ABULK>
cudaError_t launch_bn(const GemmArgs &a, int *dev_err, cudaStream_t st) {
  using C = Cfg<BN, STAGES>;
  CUtensorMap tw[3], tx;
  WTiles wt{};
  memset(tw, 0, sizeof tw);
  for (int g = 0; g < 3; ++g) {
    const void *p = a.w[g < a.n_groups ? g : 0];
    if (ABULK)
      wt.p[g] = static_cast<const uint16_t *>(p);
    else if (!make_tmap(&tw[g], p, a.group_rows, a.K, a.K, BM, tmap_type<CT>()))
      return cudaErrorInvalidValue;
  }
  wt.kt = a.K / BK;
  wt.group_rows = a.group_rows;
  if (a.w_scale[0])
    for (int g = 0; g < 3; ++g) wt.scale[g] = a.w_scale[g < a.n_groups ? g : 0];
  if (!make_tmap(&tx, a.x, a.M, a.K, a.ldx, BN, tmap_type<CT>())) return cudaErrorInvalidValue;
  cudaError_t ae = ensure_smem_limit<k_gemm_tc<CT, BN, STAGES, ABULK>>(C::SMEM);
  if (ae != cudaSuccess) return ae;
  const int kb_total = (a.K + BK - 1) / BK;
  const int kb_per_split = split_kblocks(a.K, a.split);
  if (effective_split(a.K, a.split) != a.split) return cudaErrorInvalidValue;
  const int tiles_per_group = a.n_groups > 1 ? a.group_rows / BM : (1 << 30);
  dim3 grid(a.N / BM + (a.N % BM != 0), (a.M + BN - 1) / BN, a.split);
  return launch_k(k_gemm_tc<CT, BN, STAGES, ABULK>, grid, dim3(192), C::SMEM, st, g_pdl, tw[0],
                  tw[1], tw[2], tx, tiles_per_group, a.M, a.N, kb_total, kb_per_split, a.epi, wt,
                  dev_err);
}

template <typename CT, bool ABULK, bool PAIR>
cudaError_t launch_tcp(const GemmArgs &a, int num_sms, int *dev_err, cudaStream_t st) {
  using C = Cfg<PBN, PSTAGES>;
  CUtensorMap tw[3], tx;
  WTiles wt{};
  memset(tw, 0, sizeof tw);
  for (int g = 0; g < 3; ++g) {
    const void *p = a.w[g < a.n_groups ? g : 0];
    if (ABULK)
      wt.p[g] = static_cast<const uint16_t *>(p);
    else if (!make_tmap(&tw[g], p, a.group_rows, a.K, a.K, BM, tmap_type<CT>()))
      return cudaErrorInvalidValue;
  }
  wt.kt = a.K / BK;
  wt.group_rows = a.group_rows;
  if (a.w_scale[0])
    for (int g = 0; g < 3; ++g) wt.scale[g] = a.w_scale[g < a.n_groups ? g : 0];
  if (!make_tmap(&tx, a.x, a.M, a.K, a.ldx, PAIR ? PBN / 2 : PBN, tmap_type<CT>()))
    return cudaErrorInvalidValue;
  cudaError_t ae = ensure_smem_limit<k_gemm_tcp<CT, ABULK, PAIR>>(C::SMEM);
  if (ae != cudaSuccess) return ae;
  const int kb_total = (a.K + BK - 1) / BK;
  const int tiles_per_group = a.n_groups > 1 ? a.group_rows / BM : (1 << 30);
  const int MT = a.N / BM + (a.N % BM != 0), NT = (a.M + PBN - 1) / PBN;
  if (PAIR) {
    // as many clusters as can be resident at once (a cluster's two CTAs share a GPC)
    static int max_clusters[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    int &mc = max_clusters[dev & 63];
    if (!mc) {
      cudaLaunchConfig_t qc = {};
      qc.gridDim = dim3(num_sms);
      qc.blockDim = dim3(192);
      qc.dynamicSmemBytes = C::SMEM;
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = 2;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      qc.attrs = qa;
      qc.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, k_gemm_tcp<CT, ABULK, PAIR>, &qc) != cudaSuccess ||
          n <= 0)
        return cudaErrorInvalidValue;
      mc = n;
    }
    const long long T = (long long)(MT / 2) * NT;
    const int P = (int)(T < mc ? T : mc);
    return launch_k_cluster2(k_gemm_tcp<CT, ABULK, PAIR>, dim3(2 * P), dim3(192), C::SMEM, st,
                             g_pdl, tw[0], tw[1], tw[2], tx, tiles_per_group, a.M, a.N, kb_total,
                             MT, NT, a.epi, wt, dev_err);
  }
  const long long T = (long long)MT * NT;
  const int P = (int)(T < num_sms ? T : num_sms);
  return launch_k(k_gemm_tcp<CT, ABULK, PAIR>, dim3(P), dim3(192), C::SMEM, st, g_pdl, tw[0],
                  tw[1], tw[2], tx, tiles_per_group, a.M, a.N, kb_total, MT, NT, a.epi, wt,
                  dev_err);
}

int device_sms() {
  static int sms[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!sms[dev]) cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
  return sms[dev];
}

}  // namespace

bool make_tmap_16(CUtensorMap *m, const void *ptr, int rows, int cols, int ld, int box_rows,
                  bool fp16) {
  return make_tmap(m, ptr, rows, cols, ld, box_rows,
                   fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16);
}

// 2-D 16-bit map over [rows][cols] (row stride ld elements), box {box_cols, box_rows},
// swizzle of `swizzle_bytes` (0, 32 or 128; the box's inner extent in bytes must not
// exceed it), zero fill out of bounds.
bool make_tmap_2d_16sw(CUtensorMap *m, const void *ptr, int rows, int cols, int ld, int box_cols,
                       int box_rows, int swizzle_bytes, bool fp16) {
  auto enc = get_encode();
  if (!enc) return false;
  const CUtensorMapSwizzle sw = swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                      : CU_TENSOR_MAP_SWIZZLE_NONE;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 3-D 16-bit map {d0 (innermost), d1, d2} with byte strides stride1 (d1) and stride2
// (d2), box {box0, box1, 1}, 128-byte swizzle, zero fill out of bounds.
bool make_tmap_3d_16(CUtensorMap *m, const void *ptr, long long d0, long long d1, long long d2,
                     long long stride1_bytes, long long stride2_bytes, int box0, int box1,
                     bool fp16) {
  auto enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d0, (cuuint64_t)d1, (cuuint64_t)d2};
  cuuint64_t strides[2] = {(cuuint64_t)stride1_bytes, (cuuint64_t)stride2_bytes};
  cuuint32_t box[3] = {(cuuint32_t)box0, (cuuint32_t)box1, 1};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = enc(m, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void *>(ptr), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

cudaError_t launch_gemm_tc(const GemmArgs &a, int *dev_err, cudaStream_t st) {
  // Shape rules of this kernel (checked again by the engine at create time):
  // K rows 16-byte aligned (K % 8), row groups whole tiles, pointers 16-byte aligned.
  if (a.K <= 0 || a.K % 8 || a.ldx % 8 || a.M <= 0 || a.N <= 0) return cudaErrorInvalidValue;
  if (a.n_groups < 1 || a.n_groups > 3) return cudaErrorInvalidValue;
  if (a.n_groups > 1 && a.group_rows % BM) return cudaErrorInvalidValue;
  if (a.n_groups * a.group_rows != a.N) return cudaErrorInvalidValue;
  if (a.epi.kind == EPI_QKV && a.epi.d_model % BM) return cudaErrorInvalidValue;
  // One CTA per SM with the deepest ring that fits (~190 KB of stages): the decode
  // GEMMs are weight streams, so bytes in flight per SM set their bandwidth.
  if (a.w_tiled) {
    // the tiled layout covers whole 128 x 64 tiles only
    if (a.group_rows % BM || a.K % BK) return cudaErrorInvalidValue;
    for (int g = 0; g < a.n_groups; ++g)
      if ((uintptr_t)a.w[g] % 16) return cudaErrorInvalidValue;
  }
  // many token tiles and no split: the persistent kernel
  const int sms = device_sms();
  const bool persist = a.split == 1 && a.M > PBN && sms > 0;
  auto pick = [&](auto ct) -> cudaError_t {
    using CT = decltype(ct);
    if (persist) {
      // clusters of two sharing each token tile when the weight tiles pair up
      const int MT = a.N / BM + (a.N % BM != 0);
      const bool pair = MT % 2 == 0;
      if (pair)
        return a.w_tiled ? launch_tcp<CT, true, true>(a, sms, dev_err, st)
                         : launch_tcp<CT, false, true>(a, sms, dev_err, st);
      return a.w_tiled ? launch_tcp<CT, true, false>(a, sms, dev_err, st)
                       : launch_tcp<CT, false, false>(a, sms, dev_err, st);
    }
    if (a.w_tiled) {
      if (a.M <= 16) return launch_bn<CT, 16, 10, true>(a, dev_err, st);
      if (a.M <= 32) return launch_bn<CT, 32, 9, true>(a, dev_err, st);
      if (a.M <= 64) return launch_bn<CT, 64, 8, true>(a, dev_err, st);
      if (a.M <= 128) return launch_bn<CT, 128, 6, true>(a, dev_err, st);
      return launch_bn<CT, 256, 4, true>(a, dev_err, st);
    }
    if (a.M <= 16) return launch_bn<CT, 16, 10, false>(a, dev_err, st);
    if (a.M <= 32) return launch_bn<CT, 32, 9, false>(a, dev_err, st);
    if (a.M <= 64) return launch_bn<CT, 64, 8, false>(a, dev_err, st);
    if (a.M <= 128) return launch_bn<CT, 128, 6, false>(a, dev_err, st);
    return launch_bn<CT, 256, 4, false>(a, dev_err, st);
  };
  if (a.act == ACT_BF16) return pick(bf16{});
  if (a.act == ACT_F16) return pick(f16{});
  return cudaErrorInvalidValue;
}

}  // namespace he
