// Persistent stream-K GEMM (bf16 or fp16 operands) for the decode projections
// (tcgen05 + TMEM).
//
// In decode every SM has to stream weights all the time for the projections to
// run at HBM speed (one SM moves about 1/152 of the HBM bandwidth), so tiles
// are not handed out whole: the T x KB (tile, 64-wide k-block) units of one
// GEMM are cut into P equal contiguous runs, one per CTA (P = SM count).  A run
// crosses tile boundaries; each piece of a tile it covers is a "segment".
// Segments accumulate in TMEM (two accumulators, so the epilogue of one segment
// overlaps the MMAs of the next) and are written as fp32 slices, slot = CTA
// index - first CTA of the tile (sk_segments gives how many).  For a row-wise
// consumer (EPI_PARTIAL: residual + LayerNorm) they stay as partial[slot][tok][n]
// and the consumer adds them in slot order.  Element-wise epilogues finish in the
// kernel: the tile's first run (its owner; for it the tile is the last segment,
// while the other runs' parts are their first segments) waits on a per-tile
// counter for the other slices, adds them to its own accumulator in slot order
// and stores the outputs; those slices are tile-contiguous,
// partial[slot][tile][tok][128], so each arrives as one bulk copy.  A tile
// covered by a single segment gets the element-wise epilogue directly.
//
// Warp roles (320 threads): warps 0-7 epilogue (warp w reads TMEM lanes
// 32 (w % 4) .. +31, warps w and w + 4 splitting the token columns), warp 8 loads (per stage one bulk copy of KPS tiled 128 x 64
// weight tiles, or KPS TMA boxes of row-major weights, plus one bulk copy of the
// KPS row-tiled activation k-blocks), warp 9 owns TMEM and issues the MMAs.
// The SM's copy engine spends a roughly fixed time per request (about 0.3 us for
// a bulk copy, 0.55 us for a tensor-tiled box, nearly independent of size up to
// 32 KB), so a stage is two large bulk requests.  All waits are bounded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "row_epilogue.cuh"

namespace he {

bool make_tmap_16(CUtensorMap *m, const void *ptr, int rows, int cols, int ld, int box_rows,
                  bool fp16);

namespace {

constexpr int BM = 128, BK = 64, UMMA_K = 16, A_BYTES = BM * BK * 2;

__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) |
         (2ull << 61);
}
template <typename CT>
__host__ __device__ constexpr uint32_t idesc_f16kind(int n) {
  constexpr uint32_t fmt = std::is_same<CT, bf16>::value ? 1u : 0u;
  return (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(n >> 3) << 17) |
         ((uint32_t)(BM >> 4) << 24);
}
constexpr uint32_t pow2_cols(int c) { return c <= 32 ? 32u : c <= 64 ? 64u : c <= 128 ? 128u : c <= 256 ? 256u : 512u; }

// KPS 64-wide k-blocks per pipeline stage: with tiled weights the KPS weight
// tiles of a stage are contiguous and arrive in one bulk copy (a bulk request
// costs the SM's copy engine a roughly fixed time, so bigger requests stream faster).
template <int BN, int STAGES, int KPS>
struct SkCfg {
  static constexpr int B_BYTES = BN * BK * 2;  // one k-block of activations
  static constexpr int STAGE_A = KPS * A_BYTES;
  static constexpr int STAGE_B = KPS * B_BYTES;
  static constexpr int STAGE_BYTES = STAGE_A + STAGE_B;
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + 256;  // + barriers and flags
  static constexpr uint32_t TMEM_COLS = pow2_cols(2 * BN);
};

// FP8 weights (W8): the weights of a stage are KPS / 2 consecutive 128 x 128 E4M3
// tiles (16 KB each, one bulk copy) that converter warps decode to fp16 (exactly:
// every E4M3 value is an fp16 value) and store into tensor memory as the MMA's A
// operand; the stage's activations still come from shared memory.  Weights and
// activations have rings of their own (S8 and SB stages).  The SM's copy engine
// takes a roughly fixed time per bulk request, so a stage spans 256 k (KPS 4): one
// 32 KB weight request and one activation request per stage.  TMEM holds the two
// accumulators (2 BN columns) and SA decoded A stages of 32 KPS columns each.
constexpr int W8_TILE = 128 * 128;  // one fp8 tile: 128 rows x 128 k
template <int BN, int KPS> struct Sk8Cfg {
  static constexpr int W8_STAGE = KPS / 2 * W8_TILE;
  static constexpr int STAGE_B = KPS * BN * BK * 2;
  static constexpr int SB = BN >= 128 ? 2 : BN == 64 ? 3 : BN == 32 ? 4 : 5;  // activation stages
  static constexpr int S8 = BN >= 128 ? 3 : BN == 64 ? 4 : 5;                 // weight stages
  static constexpr int A_COLS = 32 * KPS;
  static constexpr int SA = (512 - 2 * BN) / A_COLS < 4 ? (512 - 2 * BN) / A_COLS : 4;
  static constexpr uint32_t A_COL0 = 2 * BN;
  static constexpr int RING = S8 * W8_STAGE + SB * STAGE_B;
  static constexpr int SMEM = 1024 + RING + 512;
};

struct SkArgs {
  const uint16_t *wt[3]; // tiled weights per row group (tiled == 1), 16-bit elements
  const uint8_t *w8[3];  // fp8 tiled weights per row group (W8 kernels)
  const float *wscale[3];// per-row fp32 scales of the fp8 weights (W8 kernels)
  int tiled;
  int tiles_per_group;   // 128-row tiles per group (multiple groups only)
  int n_groups;
  int M, N, KB;          // tokens, output features, units (KPS k-blocks) per tile
  long long U;           // units = tiles * KB
  float *slices;         // fp32 slices: [slot][M][N], or [slot][tile][M][128] with tile_cnt
  long long slice_stride;
  int *tile_cnt;         // per-tile arrival counters (zero between launches); null: no fix-up
  // Stream-K + data-parallel split (dp > 0): run c first takes its stream-K share
  // [c U_sk / P_sk, (c + 1) U_sk / P_sk) of the units of the leftover tiles t_sk0 .. T-1
  // (none for c >= P_sk), then its dp whole tiles c dp .. c dp + dp - 1.  dp == 0:
  // plain stream-K over all U units on the P runs.
  int dp, P_sk, t_sk0;
  long long U_sk;
};

constexpr int EPW = 8;              // epilogue warps
constexpr int EPT = 32 * EPW;        // epilogue threads
constexpr int SK_THREADS = EPT + 64; // + producer warp + MMA warp
constexpr int PRODUCER = EPW, MMA = EPW + 1;
constexpr int CONV0 = EPW + 2;       // W8: converter warps, two per TMEM lane quarter
constexpr int NCONV = 8;             // (a pair of warps per quarter takes alternate stages)
constexpr int SK8_THREADS = SK_THREADS + 32 * NCONV;

// EPI_ARGMAX for a tile stored directly (one run): the greedy statistics of each
// token column over the tile's 128 rows (features n >= N left out).  Rounds of 32
// columns, 16 per column half; a warp reduces its 32 rows for 16 columns (a
// butterfly step over lanes l and l + 16, then a halving exchange after which lane l
// holds column l % 16), the four lane quarters meet in shared memory and the first
// warp of each half merges them in quarter order.  Every epilogue warp runs the same
// rounds (both barriers).
template <int BN>
__device__ __forceinline__ void argmax_tile_direct(const Epi &epi, uint32_t tl, int t, int row,
                                                   int N, int M, int quarter, int half, int lane,
                                                   bool live, ArgStat (*part)[4][16]) {
  float4 *stats = reinterpret_cast<float4 *>(epi.partial);
  for (int r0 = 0; r0 < BN; r0 += 32) {
    const int c0 = r0 + 16 * half;  // this warp's 16 columns
    const bool any = c0 < BN;       // (BN 16: the second half has none)
    ArgStat st[16];
    if (any) {
      float v[16];
      tmem_load_cols<16>(tl + (uint32_t)c0, v);
#pragma unroll
      for (int j = 0; j < 16; ++j) st[j] = row < N ? ArgStat{v[j], 1.f, row} : ArgStat{-INFINITY, 0.f, 0};
#pragma unroll
      for (int j = 0; j < 16; ++j) st[j] = argstat_merge(st[j], argstat_shfl_xor(st[j], 16));
#pragma unroll
      for (int w = 8; w >= 1; w >>= 1) {
        const bool up = (lane & w) != 0;
#pragma unroll
        for (int j = 0; j < w; ++j) {
          const ArgStat keep = up ? st[j + w] : st[j];
          const ArgStat give = up ? st[j] : st[j + w];
          st[j] = argstat_merge(keep, argstat_shfl_xor(give, w));
        }
      }
      if (lane < 16) part[half][quarter][lane] = st[0];
    }
    epi_bar_sync<EPT>();
    if (any && quarter == 0 && lane < 16) {
      ArgStat m = part[half][0][lane];
#pragma unroll
      for (int q = 1; q < 4; ++q) m = argstat_merge(m, part[half][q][lane]);
      const int tok = c0 + lane;
      if (live && tok < M)
        stats[(size_t)t * epi.ldp + tok] = make_float4(m.m, m.s, __int_as_float(m.i), 0.f);
    }
    epi_bar_sync<EPT>();
  }
}

template <typename CT, int BN, int STAGES, int KPS, bool W8 = false>
__global__ void __launch_bounds__(W8 ? SK8_THREADS : SK_THREADS, 1)
    k_gemm_sk(const __grid_constant__ CUtensorMap tm_w0, const __grid_constant__ CUtensorMap tm_w1,
              const __grid_constant__ CUtensorMap tm_w2, const __grid_constant__ CUtensorMap tm_x,
              const __grid_constant__ SkArgs a, const __grid_constant__ Epi epi, const uint16_t *x,
              int ldx, int *dev_err) {
  using C = SkCfg<BN, STAGES, KPS>;
  using C8 = Sk8Cfg<BN, KPS>;
  static_assert(!W8 || ((KPS == 2 || KPS == 4) && BN <= 128), "fp8 weights: 128- or 256-k stages, at most 128 tokens");
  constexpr uint32_t kTmemCols = W8 ? 512u : C::TMEM_COLS;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  // 16-bit weights: [STAGES x (A | B)]; W8: [S8 fp8 weight stages][SB activation stages]
  uint8_t *smA = base;
  uint8_t *smW8 = base;
  uint8_t *smB = W8 ? base + C8::S8 * C8::W8_STAGE : base + STAGES * C::STAGE_A;
  uint64_t *full = reinterpret_cast<uint64_t *>(base + (W8 ? C8::RING : STAGES * C::STAGE_BYTES));
  uint64_t *empty = full + (W8 ? C8::SB : STAGES);
  uint64_t *acc_full = empty + (W8 ? C8::SB : STAGES);  // [2]
  uint64_t *acc_empty = acc_full + 2;    // [2]
  uint64_t *fix_bar = acc_empty + 2;     // the owner's slice copies (tile_owner_epilogue)
  uint64_t *w8_full = fix_bar + 1;       // W8 only: [S8]
  uint64_t *w8_empty = w8_full + (W8 ? C8::S8 : 0);  // [S8]
  uint64_t *a_full = w8_empty + (W8 ? C8::S8 : 0);   // [SA] decoded A stage in TMEM
  uint64_t *a_empty = a_full + (W8 ? C8::SA : 0);    // [SA]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(a_empty + (W8 ? C8::SA : 0));
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
  int *last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = gridDim.x, c = blockIdx.x;
  // This run's units in order: v = 0 .. nv-1 -> global unit unit_of(v) (tile * KB + k-block).
  long long sk_b = 0, sk_n = 0, dp_t0 = 0;
  int dp_n = 0;
  if (a.dp == 0) {
    sk_b = (long long)c * a.U / P;
    sk_n = (long long)(c + 1) * a.U / P - sk_b;
  } else {
    if (c < a.P_sk) {
      sk_b = (long long)c * a.U_sk / a.P_sk;
      sk_n = (long long)(c + 1) * a.U_sk / a.P_sk - sk_b;
    }
    dp_t0 = (long long)c * a.dp;
    dp_n = a.dp;
  }
  const long long nv = sk_n + (long long)dp_n * a.KB;
  auto unit_of = [&](long long v) -> long long {
    return v < sk_n ? (long long)a.t_sk0 * a.KB + sk_b + v : dp_t0 * a.KB + (v - sk_n);
  };
  // units of the segment starting at v (k-block kb0 of its tile): to the tile's end, and
  // the stream-K share never runs into the whole tiles
  auto seg_len = [&](long long v, int kb0) -> int {
    return (int)(v < sk_n ? min((long long)(a.KB - kb0), sk_n - v) : (long long)(a.KB - kb0));
  };

  if (warp == PRODUCER && lane == 0) {
    const int nst = W8 ? C8::SB : STAGES;
    for (int s = 0; s < nst; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], EPW);  // one arrival per epilogue warp
    }
    mbar_init(fix_bar, 1);
    if constexpr (W8) {
      for (int s = 0; s < C8::S8; ++s) {
        mbar_init(&w8_full[s], 1);
        mbar_init(&w8_empty[s], 4);  // one arrival per converter warp
      }
      for (int s = 0; s < C8::SA; ++s) {
        mbar_init(&a_full[s], 4);
        mbar_init(&a_empty[s], 1);  // the MMAs reading the stage have completed
      }
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();  // one CTA per SM: the next kernel may start its set-up

  if (W8 && warp == PRODUCER && lane < 2) {
    // ---------------- loads, fp8 weights ----------------
    // lane 0 streams the weight stages (before waiting on the kernel before this one:
    // they do not depend on it), lane 1 the activation stages; each ring runs on its
    // own, so the weights may run ahead of the activations.
    const bool wts = lane == 0;
    const int NS = wts ? C8::S8 : C8::SB;
    const uint32_t bytes = wts ? (uint32_t)C8::W8_STAGE : (uint32_t)C8::STAGE_B;
    uint64_t *fb = wts ? w8_full : full;
    uint64_t *eb = wts ? w8_empty : empty;
    const uint64_t pol = l2_evict_first_policy();
    if (!wts) pdl_wait();
    long long issued = 0;
    for (long long i = 0; i < nv; ++i) {
      const long long u = unit_of(i);
      const int s = (int)(i % NS);
      if (i >= NS && !mbar_wait_bounded(&eb[s], (uint32_t)((i / NS - 1) & 1))) {
        *(volatile int *)abort_flag = 1;
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
        break;
      }
      if (*(volatile int *)abort_flag) break;
      const int t = (int)(u / a.KB), kb = (int)(u - (long long)t * a.KB);
      mbar_arrive_expect_tx(&fb[s], bytes);
      if (wts) {
        const int group = a.n_groups > 1 ? t / a.tiles_per_group : 0;
        const int lt = t - group * (a.n_groups > 1 ? a.tiles_per_group : 0);
        bulk_load_hint(smW8 + s * C8::W8_STAGE,
                       a.w8[group] + ((long long)lt * a.KB + kb) * C8::W8_STAGE, bytes, &fb[s],
                       pol);
      } else {
        bulk_load(smB + s * C8::STAGE_B, x + (long long)kb * KPS * BN * BK, bytes, &fb[s]);
      }
      issued = i + 1;
    }
    // every requested stage lands before the CTA can finish
    for (long long i = issued > NS ? issued - NS : 0; i < issued; ++i)
      if (!mbar_wait_bounded(&fb[i % NS], (uint32_t)((i / NS) & 1)))
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
  } else if (W8 && warp >= CONV0) {
    // ---------------- fp8 -> fp16 into TMEM (A operand) ----------------
    // Thread = weight row r (TMEM lane r; warp w reaches lanes 32 (w % 4) ..): in each
    // fp8 tile of the stage its 128 values are eight 16-byte chunks, chunk j (k = 16 j
    // ..) at slot j ^ (r % 8) of the row's 128 bytes; decoded pairs go to TMEM columns
    // 64 tt + 8 j .. + 7 of the stage (tile tt).
    const int quarter = warp & 3, r = quarter * 32 + lane;
    const int pair = (warp - CONV0) / 4;  // this warp's stages: pair, pair + 2, ...
    const uint32_t trow = tmem_base + ((uint32_t)(quarter * 32) << 16) + C8::A_COL0;
    for (long long i = pair; i < nv; i += NCONV / 4) {
      const int s8 = (int)(i % C8::S8), sa = (int)(i % C8::SA);
      bool ok = mbar_wait_bounded(&w8_full[s8], (uint32_t)((i / C8::S8) & 1));
      if (ok && i >= C8::SA)
        ok = mbar_wait_bounded(&a_empty[sa], (uint32_t)((i / C8::SA - 1) & 1));
      if (!ok || *(volatile int *)abort_flag) {
        if (!ok) set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
        *(volatile int *)abort_flag = 1;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int tt = 0; tt < KPS / 2; ++tt) {  // the stage's fp8 tiles, 64 TMEM columns each
        const uint32_t row_s = smem_u32(smW8 + s8 * C8::W8_STAGE + tt * W8_TILE + r * 128);
        uint4 ch[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) ch[j] = lds_u128(row_s + (uint32_t)((j ^ (r & 7)) * 16));
        if (tt == KPS / 2 - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&w8_empty[s8]);  // the fp8 stage may be refilled
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t w[16];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const uint32_t *q = reinterpret_cast<const uint32_t *>(&ch[2 * g + h]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __half2_raw lo = __nv_cvt_fp8x2_to_halfraw2(
                  (__nv_fp8x2_storage_t)(q[e] & 0xFFFFu), __NV_E4M3);
              const __half2_raw hi = __nv_cvt_fp8x2_to_halfraw2(
                  (__nv_fp8x2_storage_t)(q[e] >> 16), __NV_E4M3);
              w[8 * h + 2 * e] = (uint32_t)lo.x | ((uint32_t)lo.y << 16);
              w[8 * h + 2 * e + 1] = (uint32_t)hi.x | ((uint32_t)hi.y << 16);
            }
          }
          tmem_st16(trow + (uint32_t)(sa * C8::A_COLS + tt * 64 + g * 16), w);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&a_full[sa]);
    }
  } else if (!W8 && warp == PRODUCER && lane == 0) {
    // ---------------- loads ----------------
    if (!a.tiled) {
      prefetch_tmap(&tm_w0);
      if (a.n_groups > 1) prefetch_tmap(&tm_w1);
      if (a.n_groups > 2) prefetch_tmap(&tm_w2);
    }
    long long issued = 0;
    const uint64_t pol = l2_evict_first_policy();  // every weight byte is read once
    // Weights do not depend on the kernel before this one: the weight part of the
    // first stages is requested before waiting for it (programmatic dependent
    // launch), the activation part after.
    auto load_a = [&](long long u, int s) {
      const int t = (int)(u / a.KB), kb = (int)(u - (long long)t * a.KB);
      const int group = a.n_groups > 1 ? t / a.tiles_per_group : 0;
      const int lt = t - group * (a.n_groups > 1 ? a.tiles_per_group : 0);
      if (a.tiled) {
        const uint16_t *src = a.wt[group] + ((long long)lt * a.KB + kb) * (KPS * BM * BK);
        bulk_load_hint(smA + s * C::STAGE_A, src, C::STAGE_A, &full[s], pol);
      } else {
        const CUtensorMap *tw = group == 0 ? &tm_w0 : (group == 1 ? &tm_w1 : &tm_w2);
#pragma unroll
        for (int j = 0; j < KPS; ++j)
          tma_load_2d_hint(smA + s * C::STAGE_A + j * A_BYTES, tw, &full[s], (kb * KPS + j) * BK,
                           lt * BM, pol);
      }
    };
    auto load_b = [&](long long u, int s) {
      const int t = (int)(u / a.KB), kb = (int)(u - (long long)t * a.KB);
      bulk_load(smB + s * C::STAGE_B, x + (long long)kb * KPS * BN * BK, C::STAGE_B, &full[s]);
    };
    const long long pre = min((long long)STAGES, nv);
    for (long long i = 0; i < pre; ++i) {
      mbar_arrive_expect_tx(&full[i], C::STAGE_BYTES);
      load_a(unit_of(i), (int)i);
    }
    pdl_wait();
    for (long long i = 0; i < pre; ++i) load_b(unit_of(i), (int)i);
    issued = pre;
    for (long long i = pre; i < nv; ++i) {
      const long long u = unit_of(i);
      const int s = (int)(i % STAGES);
      if (!mbar_wait_bounded(&empty[s], (uint32_t)((i / STAGES - 1) & 1))) {
        *(volatile int *)abort_flag = 1;
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
        break;
      }
      if (*(volatile int *)abort_flag) break;
      mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
      load_a(u, s);
      load_b(u, s);
      issued = i + 1;
    }
    for (long long i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
      if (!mbar_wait_bounded(&full[i % STAGES], (uint32_t)((i / STAGES) & 1)))
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
  } else if (warp == MMA && lane == 0) {
    // ---------------- MMA ----------------
    constexpr uint32_t idesc = idesc_f16kind<CT>(BN);
    int seg = 0;
    bool ok = true;
    for (long long v = 0; v < nv && ok;) {
      const long long u = unit_of(v);
      const int t = (int)(u / a.KB), kb0 = (int)(u - (long long)t * a.KB);
      const int n = seg_len(v, kb0);
      const int buf = seg & 1;
      if (seg >= 2 && !mbar_wait_bounded(&acc_empty[buf], (uint32_t)(((seg >> 1) - 1) & 1))) {
        *(volatile int *)abort_flag = 1;
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t acc = tmem_base + (uint32_t)(buf * BN);
      if constexpr (W8) {
        for (int j = 0; j < n; ++j) {
          const long long i = v + j;
          const int sb = (int)(i % C8::SB), sa = (int)(i % C8::SA);
          if (!mbar_wait_bounded(&full[sb], (uint32_t)((i / C8::SB) & 1)) ||
              !mbar_wait_bounded(&a_full[sa], (uint32_t)((i / C8::SA) & 1)) ||
              *(volatile int *)abort_flag) {
            *(volatile int *)abort_flag = 1;
            set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int q = 0; q < KPS; ++q) {
            const uint32_t b0 = smem_u32(smB + sb * C8::STAGE_B + q * C::B_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
              tc_mma_f16_tmem_a(acc, tmem_base + C8::A_COL0 + (uint32_t)(sa * C8::A_COLS + (q * 4 + kk) * 8),
                                sdesc_sw128(b0 + kk * UMMA_K * 2), idesc, (j | q | kk) != 0);
          }
          tc_commit(&empty[sb]);
          tc_commit(&a_empty[sa]);
        }
        tc_commit(&acc_full[buf]);  // also issued on abort so the epilogue is released
        v += n;
        ++seg;
        continue;
      }
      for (int j = 0; j < n; ++j) {
        const long long i = v + j;
        const int s = (int)(i % STAGES);
        if (!mbar_wait_bounded(&full[s], (uint32_t)((i / STAGES) & 1)) ||
            *(volatile int *)abort_flag) {
          *(volatile int *)abort_flag = 1;
          set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < KPS; ++q) {
          const uint32_t a0 = smem_u32(smA + s * C::STAGE_A + q * A_BYTES);
          const uint32_t b0 = smem_u32(smB + s * C::STAGE_B + q * C::B_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / UMMA_K; ++kk)
            tc_mma_f16(acc, sdesc_sw128(a0 + kk * UMMA_K * 2), sdesc_sw128(b0 + kk * UMMA_K * 2),
                       idesc, (j | q | kk) != 0);
        }
        tc_commit(&empty[s]);
      }
      tc_commit(&acc_full[buf]);  // also issued on abort so the epilogue is released
      v += n;
      ++seg;
    }
  } else if (warp < EPW) {
    // ---------------- epilogue ----------------
    // With a.tile_cnt (element-wise epilogues) a tile split over S runs is finished
    // inside the kernel by its owner, the run holding its first k-blocks (slot 0;
    // for that run it is always the last segment, reached at the end of its
    // range): the other runs (whose part is their first segment, done early) write
    // fp32 slices and count themselves in the tile's counter; the owner waits for
    // the count, adds the slices to its own accumulator in slot order, applies the
    // epilogue and clears the counter.  The owner's staged reduction reuses the
    // pipeline's shared memory, free after the CTA's last MMA.  Without
    // a.tile_cnt, tiles of one run are stored directly and the others are left as
    // slices for a second kernel.
    const bool fix = a.tile_cnt != nullptr && epi.kind != EPI_PARTIAL;
    __shared__ ArgStat am_part[W8 ? 1 : 2][4][16];  // EPI_ARGMAX (16-bit weights only)
    constexpr int W = BN >= 32 ? 32 : 16;
    constexpr int kStageAvail = W8 ? C8::RING : STAGES * C::STAGE_BYTES;
    // The bias of this thread's row in the tile of the last segment (the one an
    // owner finishes at the end of the run), read before waiting on the kernel
    // before this one: parameters do not depend on it.
    const int quarter = warp & 3, half = warp >> 2;  // TMEM lanes 32 quarter.., column half
    float last_bias = 0.f;
    if (fix && nv > 0) {
      const int t_last = (int)(unit_of(nv - 1) / a.KB);
      last_bias = tile_row_bias(epi, t_last * BM + quarter * 32 + lane, a.N);
    }
    pdl_wait();  // outputs may still be read by the kernel before this one
    int seg = 0;
    for (long long v = 0; v < nv;) {
      const long long u = unit_of(v);
      const int t = (int)(u / a.KB), kb0 = (int)(u - (long long)t * a.KB);
      const int n = seg_len(v, kb0);
      const int buf = seg & 1;
      const bool ok = !*(volatile int *)abort_flag &&
                      mbar_wait_bounded(&acc_full[buf], (uint32_t)((seg >> 1) & 1));
      if (!ok) set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
      tc_fence_after();
      const bool live = ok && !*(volatile int *)abort_flag;
      // the runs that share tile t: stream-K tiles among the P (or P_sk) runs, whole
      // tiles of the data-parallel part by this run alone
      int cf = c, S = 1;
      if (v < sk_n) {
        if (a.dp == 0)
          sk_segments(t, a.KB, P, a.U, &cf, &S);
        else
          sk_segments(t - a.t_sk0, a.KB, a.P_sk, a.U_sk, &cf, &S);
      }
      const int slot = c - cf;
      const int row = t * BM + quarter * 32 + lane;
      const uint32_t tl = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * BN);
      // W8: this row's fp8 scale, applied as the accumulator leaves TMEM
      float rs = 1.f;
      if constexpr (W8) {
        const int group = a.n_groups > 1 ? t / a.tiles_per_group : 0;
        const int gr = row - group * (a.n_groups > 1 ? a.tiles_per_group : 0) * BM;
        if (row < a.N) rs = a.wscale[group][gr];
      }
      // (all conditions below are uniform over the four epilogue warps)
      const bool staged = fix && slot == 0 && v + n == nv &&
                          tile_stage_tokens(S, a.M, W, kStageAvail) >= W;
      if (staged) {
        tile_owner_epilogue<CT, W, EPT>(epi, a.slices + (size_t)t * a.M * BM, a.slice_stride,
                                        a.N, a.M, t, S, tl, live, &a.tile_cnt[t], base,
                                        kStageAvail, fix_bar, last_flag, dev_err, last_bias, rs);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      } else if (S == 1 && epi.kind == EPI_ARGMAX) {
        argmax_tile_direct<BN>(epi, tl, t, row, a.N, a.M, quarter, half, lane, live, am_part);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
      } else {
        const bool direct = S == 1 && epi.kind != EPI_PARTIAL;
        RowEpi<CT> re = row_epi_prepare<CT>(epi, row < a.N ? row : 0,
                                            direct ? nullptr : a.slices, a.slice_stride, slot,
                                            a.N);
        if (fix && !direct) {  // tile-contiguous slices: [slot][tile][M][128]
          re.f32 = a.slices + slot * a.slice_stride + (size_t)t * a.M * BM + (row - t * BM);
          re.f32_stride = BM;
        }
        // the two warps of a lane quarter take one half of the columns each (BN 16:
        // the first one all 16)
        constexpr int WH = BN >= 64 ? 32 : 16;
        const int c_begin = BN >= 32 ? half * (BN / 2) : 0;
        const int c_end = BN >= 32 ? c_begin + BN / 2 : (half == 0 ? BN : 0);
#pragma unroll 1
        for (int c0 = c_begin; c0 < c_end; c0 += WH) {
          float v[WH];
          tmem_load_cols<WH>(tl + c0, v);
          if constexpr (W8) {
#pragma unroll
            for (int j = 0; j < WH; ++j) v[j] *= rs;
          }
          if (live && row < a.N && c0 < a.M) row_epi_store<CT, WH>(re, c0, min(WH, a.M - c0), v);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&acc_empty[buf]);
        if (fix && S > 1) {
          // this run's slice is complete: count it (release), every run of the
          // tile including an owner without room for the staged reduction
          __threadfence();
          epi_bar_sync<EPT>();
          if (threadIdx.x == 0 && live) atomicAdd(&a.tile_cnt[t], 1);
          if (slot == 0) {
            // owner: wait for all S slices, then reduce them through registers
            if (threadIdx.x == 0) {
              bool ok2 = live && wait_count_at_least(&a.tile_cnt[t], S);
              if (live && !ok2) set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
              *last_flag = ok2;
            }
            epi_bar_sync<EPT>();
            if (*last_flag) {
              __threadfence();
              tile_fixup<CT, EPT>(epi, a.slices + (size_t)t * a.M * BM, a.slice_stride, a.N,
                                  a.M, t, S, threadIdx.x);
              if (threadIdx.x == 0) a.tile_cnt[t] = 0;
            }
          }
        }
      }
      v += n;
      ++seg;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <typename CT, int BN, int STAGES, int KPS, bool W8 = false>
cudaError_t launch_sk_bn(const GemmArgs &g, int P, float *slices, long long slice_stride,
                         int *tile_cnt, int *dev_err, cudaStream_t st) {
  using C = SkCfg<BN, STAGES, KPS>;
  constexpr bool fp16 = !std::is_same<CT, bf16>::value;
  constexpr int kSmem = W8 ? Sk8Cfg<BN, KPS>::SMEM : C::SMEM;
  CUtensorMap tw[3], tx;
  memset(tw, 0, sizeof tw);
  SkArgs a{};
  a.tiled = g.w_tiled;
  a.n_groups = g.n_groups;
  a.tiles_per_group = g.n_groups > 1 ? g.group_rows / BM : 1;
  for (int i = 0; i < 3; ++i) {
    const void *p = g.w[i < g.n_groups ? i : 0];
    if (W8) {
      a.w8[i] = static_cast<const uint8_t *>(p);
      a.wscale[i] = g.w_scale[i < g.n_groups ? i : 0];
      if ((uintptr_t)p % 16 || !a.wscale[i]) return cudaErrorInvalidValue;
    } else if (g.w_tiled) {
      a.wt[i] = static_cast<const uint16_t *>(p);
    } else if (i < g.n_groups && !make_tmap_16(&tw[i], p, g.group_rows, g.K, g.K, BM, fp16)) {
      return cudaErrorInvalidValue;
    }
  }
  memset(&tx, 0, sizeof tx);  // activations arrive by bulk copy (row-tiled layout)
  if ((uintptr_t)g.x % 16) return cudaErrorInvalidValue;
  a.M = g.M;
  a.N = g.N;
  a.KB = g.K / (BK * KPS);
  a.U = (long long)((g.N + BM - 1) / BM) * a.KB;
  a.slices = slices;
  a.slice_stride = slice_stride;
  a.tile_cnt = tile_cnt;
  // With the in-kernel fix-up, at least one whole tile per run and 16-bit weights: each
  // run first takes its share of the leftover tiles, split stream-K over at most 15 runs
  // a tile, then its whole tiles, so that no run ends in an owner's fix-up (the owners
  // of the leftover tiles finish them while the whole tiles stream).
  const long long T = (g.N + BM - 1) / BM;
  if (g.sk_hybrid && !W8 && tile_cnt && g.epi.kind != EPI_ARGMAX && T >= P) {
    a.dp = (int)(T / P);
    a.t_sk0 = a.dp * P;
    const long long L = T - a.t_sk0;
    a.U_sk = L * a.KB;
    long long psk = P;
    if (psk > 15 * L) psk = 15 * L;
    if (psk > a.U_sk) psk = a.U_sk;
    a.P_sk = (int)psk;
  }
  cudaError_t ae = ensure_smem_limit<k_gemm_sk<CT, BN, STAGES, KPS, W8>>(kSmem);
  if (ae != cudaSuccess) return ae;
  return launch_k(k_gemm_sk<CT, BN, STAGES, KPS, W8>, dim3(P), dim3(W8 ? SK8_THREADS : SK_THREADS),
                  kSmem, st, g_pdl, tw[0], tw[1], tw[2], tx, a, g.epi,
                  static_cast<const uint16_t *>(g.x), g.ldx, dev_err);
}

}  // namespace

int sk_kps(const GemmArgs &g) {
  if (g.w_fp8) return 4;  // fp8 weights: 256-k stages (K % 256 == 0)
  return g.K % 128 == 0 ? 2 : 1;
}

long long sk_units(const GemmArgs &g) {
  return (long long)((g.N + 127) / 128) * (g.K / (64 * sk_kps(g)));
}

// Runs: one per SM, at most U runs and at most 15 runs per tile (so a tile never
// has more than 16 slices).  Without the in-kernel fix-up, whole tiles (P = T)
// when the tiles nearly fill the GPU, which needs no reduction.
int sk_ctas(const GemmArgs &g, int num_sms, bool fixup) {
  const long long T = (g.N + 127) / 128, U = sk_units(g);
  if (!fixup && T <= num_sms && 10 * T >= 7LL * num_sms) return (int)T;
  long long P = num_sms;
  if (P > U) P = U;
  if (U < 2 * P) {
    // under two units a run: the longest runs set the time, so give every run that many
    // and use fewer runs (fewer slices to add, fewer fix-ups)
    const long long per = (U + P - 1) / P;
    P = (U + per - 1) / per;
  }
  if (P > 15 * T) P = 15 * T;
  return (int)P;
}

// The in-kernel completion stores 16-byte groups of outputs (4 fp32 or 8 16-bit).
bool sk_fixup_ok(const GemmArgs &g) {
  const Epi &e = g.epi;
  auto al = [](const void *p) { return (uintptr_t)p % 16 == 0; };
  switch (e.kind) {
    case EPI_STORE_F32:
      return g.N % 4 == 0 && e.ldp % 4 == 0 && al(e.partial);
    case EPI_RELU:
      return g.N % 8 == 0 && al(e.out) && (e.out_rows > 0 || e.ldo % 8 == 0);
    case EPI_QKV:
      return g.N % 8 == 0 && e.head_dim % 8 == 0 && e.ldo % 8 == 0 && al(e.out) && al(e.kc) &&
             al(e.vc);
    case EPI_ARGMAX:
      return g.N % 4 == 0 && e.ldp >= g.M && al(e.partial);
    default:
      return false;
  }
}

// Shared memory of the pipeline stages of the kernel launch_gemm_sk picks for a.
static int sk_stage_avail(const GemmArgs &g) {
  struct Pick { int bn, stages, kps; };
  Pick p;
  if (sk_kps(g) == 2)
    p = g.M <= 16 ? Pick{16, 5, 2} : g.M <= 32 ? Pick{32, 5, 2} : g.M <= 64 ? Pick{64, 4, 2}
        : g.M <= 128 ? Pick{128, 3, 2} : Pick{256, 2, 2};
  else
    p = g.M <= 16 ? Pick{16, 10, 1} : g.M <= 32 ? Pick{32, 9, 1} : g.M <= 64 ? Pick{64, 8, 1}
        : g.M <= 128 ? Pick{128, 6, 1} : Pick{256, 4, 1};
  return p.stages * p.kps * (BM * BK * 2 + p.bn * BK * 2);
}

bool sk_argmax_ok(const GemmArgs &g, int P) {
  if (g.epi.kind != EPI_ARGMAX || !sk_fixup_ok(g)) return false;
  const long long T = (g.N + BM - 1) / BM, U = sk_units(g);
  const int KB = (int)(U / T);
  int smax = 1;
  for (long long t = 0; t < T; ++t) {
    int cf, S;
    sk_segments((int)t, KB, P, U, &cf, &S);
    if (S > smax) smax = S;
  }
  const int W = g.M <= 16 ? 16 : 32;  // the owner's column chunk (BN >= 32: 32)
  return tile_stage_tokens(smax, g.M, W, sk_stage_avail(g)) >= W;
}

cudaError_t launch_gemm_sk(const GemmArgs &g, int P, float *slices, long long slice_stride,
                           int *tile_cnt, int *dev_err, cudaStream_t st) {
  // One row tile of tokens (M <= 256), whole 128 x 64 tiles, fp32 slices in epi.partial.
  if ((g.act != ACT_BF16 && g.act != ACT_F16) || g.M < 1 || g.M > 256 || g.K % BK)
    return cudaErrorInvalidValue;
  if (g.w_tiled && (g.group_rows % BM)) return cudaErrorInvalidValue;
  if (g.n_groups < 1 || g.n_groups > 3 || g.n_groups * g.group_rows != g.N) return cudaErrorInvalidValue;
  if (g.epi.kind == EPI_QKV && g.epi.d_model % BM) return cudaErrorInvalidValue;
  if (!slices || P < 1 || slice_stride < (long long)g.M * g.N) return cudaErrorInvalidValue;
  if (tile_cnt && (!sk_fixup_ok(g) || (uintptr_t)slices % 16 ||
                   slice_stride < (long long)g.M * ((g.N + BM - 1) / BM) * BM))
    return cudaErrorInvalidValue;
  if (g.epi.kind == EPI_ARGMAX && (!tile_cnt || !sk_argmax_ok(g, P))) return cudaErrorInvalidValue;
  if (g.w_fp8) {
    // fp8 weights (fp8 tiled layout, K % 128 == 0, whole 128-row tiles) with fp16
    // activations, at most 128 tokens
    if (g.act != ACT_F16 || g.M > 128 || g.K % 256 || (g.group_rows % BM) ||
        g.epi.kind == EPI_ARGMAX)
      return cudaErrorInvalidValue;
#define HE_SK8(BN) \
  return launch_sk_bn<f16, BN, Sk8Cfg<BN, 4>::SB, 4, true>(g, P, slices, slice_stride, tile_cnt, dev_err, st)
    if (g.M <= 16) HE_SK8(16);
    if (g.M <= 32) HE_SK8(32);
    if (g.M <= 64) HE_SK8(64);
    HE_SK8(128);
#undef HE_SK8
  }
  auto pick = [&](auto ct) -> cudaError_t {
    using CT = decltype(ct);
#define HE_SK(BN, ST, KPS) \
  return launch_sk_bn<CT, BN, ST, KPS>(g, P, slices, slice_stride, tile_cnt, dev_err, st)
    if (sk_kps(g) == 2) {
      // two k-blocks per stage: 32 KB weight requests
      if (g.M <= 16) HE_SK(16, 5, 2);
      if (g.M <= 32) HE_SK(32, 5, 2);
      if (g.M <= 64) HE_SK(64, 4, 2);
      if (g.M <= 128) HE_SK(128, 3, 2);
      HE_SK(256, 2, 2);
    }
    if (g.M <= 16) HE_SK(16, 10, 1);
    if (g.M <= 32) HE_SK(32, 9, 1);
    if (g.M <= 64) HE_SK(64, 8, 1);
    if (g.M <= 128) HE_SK(128, 6, 1);
    HE_SK(256, 4, 1);
#undef HE_SK
  };
  if (g.act == ACT_BF16) return pick(bf16{});
  return pick(f16{});
}

}  // namespace he
