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
//
// One launch can run several phases in order (SkChain): projections, and the
// residual + LayerNorm rows that follow an EPI_PARTIAL projection, separated by
// grid barriers.  In decode a layer's out projection, residual + LayerNorm, fc1,
// fc2, residual + LayerNorm and the next layer's QKV projection are one launch:
// the producer requests the next projection's weights while the CTAs wait at the
// barrier, so the weight stream does not stop between the projections the way
// it does at a kernel boundary.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstring>
#include <type_traits>

#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"
#include "row_epilogue.cuh"
#include "rowops.cuh"

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
  static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + 512;  // + barriers, flags, sums
  static constexpr uint32_t TMEM_COLS = pow2_cols(2 * BN);
};

// One projection of a launch (PH_GEMM): the stream-K work of the GEMM above.
struct SkGemm {
  const uint16_t *wt[3];  // tiled weights per row group (tiled == 1), 16-bit elements
  int map0;               // row-major weights: the launch's tensor maps map0 .. map0 + n_groups - 1
  int tiled;
  int tiles_per_group;    // 128-row tiles per group (multiple groups only)
  int n_groups;
  int N, KB, P;           // output features, units (KPS k-blocks) per tile, runs (CTAs 0..P-1)
  long long U;            // units = tiles * KB
  const uint16_t *x;      // activations, row-tiled with BN rows
  float *slices;          // fp32 slices: [slot][M][N], or [slot][tile][M][128] with tile_cnt
  long long slice_stride;
  int *tile_cnt;          // per-tile arrival counters (zero between uses); null: no fix-up
  Epi epi;
};

// Residual + LayerNorm of the M token rows after an EPI_PARTIAL projection (PH_ROWS):
// x[r] += sum of the slices + bias; h[r] = LayerNorm(x[r]) (parameters bf16).
struct SkRows {
  const float *partial;   // slice 0 of the projection before, [M][ldp]
  SliceInfo si;
  long long split_stride;
  int ldp;
  const bf16 *bias, *gamma, *beta;
  float *x;               // fp32 residual stream [M][d]
  float eps;
  void *h;                // LayerNorm output, act_index layout with h_rows rows
  int h_rows, d, out_bf16;  // out_bf16: h is bf16 (else the operand type CT)
};

struct SkPhase {
  int kind;  // PH_GEMM or PH_ROWS
  SkGemm gm;
  SkRows rw;
};

// The phases of one launch.  Phase p + 1 starts on any CTA only after every CTA has
// finished phase p: a grid barrier on the counter *gbar, which counts arrivals of
// the whole generation (bar_base of them came before this launch).  All CTAs are
// resident (one per SM), which the barrier relies on; its waits are bounded.
struct SkChain {
  int n, M;               // phases, tokens
  SkPhase ph[kMaxPhases];
  unsigned *gbar;
  unsigned bar_base;
};
struct SkMaps {
  CUtensorMap m[kMaxMaps];
};

constexpr int EPW = 8;              // epilogue warps
constexpr int EPT = 32 * EPW;        // epilogue threads
constexpr int SK_THREADS = EPT + 64; // + producer warp + MMA warp
constexpr int PRODUCER = EPW, MMA = EPW + 1;
constexpr int kRowGroups = 4;        // 8-element groups per epilogue thread in a rows phase

__device__ __forceinline__ void sk_run(const SkGemm &g, int c, long long *ub, long long *ue) {
  *ub = c < g.P ? (long long)c * g.U / g.P : 0;
  *ue = c < g.P ? (long long)(c + 1) * g.U / g.P : 0;
}

// Wait (acquire) until the grid-barrier counter reaches `target`.  Gives up after
// about half a second, or early once some CTA has reported a timed-out wait.
__device__ __forceinline__ bool grid_wait(const unsigned *p, unsigned target, int *dev_err) {
  for (uint32_t i = 0; i < (1u << 20); ++i) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    if (v >= target) return true;
    if ((i & 255) == 255 && (*(volatile int *)dev_err & DEVERR_WAIT_TIMEOUT)) return false;
    if (i >= 32) __nanosleep(64);
  }
  set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
  return false;
}

// Sum over the EPT epilogue threads of one value per "virtual" thread: vals[j] is
// the value of 8-element group et + EPT j, and the groups are added warp by warp
// in the order a block with one thread per group (d / 8 threads) adds them, so
// the result has the bits of block_sum in k_resid_ln8.
__device__ __forceinline__ float rows_sum(const float (&vals)[kRowGroups], int nwv, float *red) {
  const int et = threadIdx.x, lane = et & 31, w = et >> 5;
  epi_bar_sync<EPT>();  // red may still be read from the sum before
#pragma unroll
  for (int j = 0; j < kRowGroups; ++j) {
    const int vw = w + EPW * j;  // virtual warp of this thread's group j
    if (vw < nwv) {
      const float s = warp_sum(vals[j]);
      if (lane == 0) red[vw] = s;
    }
  }
  epi_bar_sync<EPT>();
  if (w == 0) {
    float t = lane < nwv ? red[lane] : 0.f;
    t = warp_sum(t);
    if (lane == 0) red[32] = t;
  }
  epi_bar_sync<EPT>();
  return red[32];
}

// A rows phase on the epilogue threads: rows c, c + G, ... of the M rows.  Per
// 8-element group the arithmetic of k_resid_ln8 (slices in slot order, then the
// bias, onto the residual; mean, then the biased variance of the centred values).
template <typename CT>
__device__ void sk_rows_phase(const SkRows &w, int M, int c, int G, float *red) {
  const int et = threadIdx.x, d = w.d, nwv = d >> 8;  // d / 256 virtual warps
#pragma unroll 1
  for (int r = c; r < M; r += G) {
    float v[kRowGroups][8];
    float part[kRowGroups];
#pragma unroll
    for (int j = 0; j < kRowGroups; ++j) {
      part[j] = 0.f;
      const int col = 8 * (et + EPT * j);
      if (col < d) {
        float bs[8];
        load8<bf16>(w.bias + col, bs);
        float4 *xr = reinterpret_cast<float4 *>(w.x + (long long)r * d + col);
        const float *pr = w.partial + (long long)r * w.ldp + col;
        const int S = w.si.slices(col);
        float4 x0 = __ldcg(xr), x1 = __ldcg(xr + 1);
        float4 a0, a1;
        sum_slices8<8>(pr, S, w.split_stride, a0, a1);
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
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) s += v[j][i];
        part[j] = s;
      }
    }
    const float mean = rows_sum(part, nwv, red) / (float)d;
#pragma unroll
    for (int j = 0; j < kRowGroups; ++j) {
      float q = 0.f;
      if (8 * (et + EPT * j) < d) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[j][i] -= mean;
          q += v[j][i] * v[j][i];
        }
      }
      part[j] = q;
    }
    const float var = rows_sum(part, nwv, red) / (float)d;
    const float rstd = 1.0f / sqrtf(var + w.eps);
#pragma unroll
    for (int j = 0; j < kRowGroups; ++j) {
      const int col = 8 * (et + EPT * j);
      if (col < d) {
        float gs[8], bt[8];
        load8<bf16>(w.gamma + col, gs);
        load8<bf16>(w.beta + col, bt);
#pragma unroll
        for (int i = 0; i < 8; ++i) v[j][i] = v[j][i] * rstd * gs[i] + bt[i];
        const long long o = act_index(r, col, d, w.h_rows);
        if (w.out_bf16)
          store8<bf16>(static_cast<bf16 *>(w.h) + o, v[j]);
        else
          store8<CT>(static_cast<CT *>(w.h) + o, v[j]);
      }
    }
  }
}

template <typename CT, int BN, int STAGES, int KPS>
__global__ void __launch_bounds__(SK_THREADS, 1)
    k_gemm_sk(const __grid_constant__ SkMaps maps, const __grid_constant__ SkChain ch,
              int *dev_err) {
  using C = SkCfg<BN, STAGES, KPS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t *base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  // stage s: KPS weight k-blocks, then KPS activation k-blocks (one contiguous block,
  // which the owner reduction of a split tile can borrow as a whole)
  auto stage_a = [&](int s) { return base + (size_t)s * C::STAGE_BYTES; };
  auto stage_b = [&](int s) { return base + (size_t)s * C::STAGE_BYTES + C::STAGE_A; };
  uint64_t *full = reinterpret_cast<uint64_t *>(base + STAGES * C::STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *acc_full = empty + STAGES;   // [2]
  uint64_t *acc_empty = acc_full + 2;    // [2]
  uint64_t *fix_bar = acc_empty + 2;     // the owner's slice copies (tile_owner_epilogue)
  uint64_t *epi_free = fix_bar + 1;      // the epilogue is done with a projection's stages
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(epi_free + 1);
  int *abort_flag = reinterpret_cast<int *>(tmem_slot + 1);
  int *last_flag = abort_flag + 1;
  int *gate = last_flag + 1;
  float *red = reinterpret_cast<float *>(gate + 1);  // [33]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = gridDim.x, c = blockIdx.x;

  if (warp == PRODUCER && lane == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], EPW);  // one arrival per epilogue warp
    }
    mbar_init(fix_bar, 1);
    mbar_init(epi_free, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == MMA) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_trigger();  // one CTA per SM: the next kernel may start its set-up

  if (warp == PRODUCER && lane == 0) {
    // ---------------- loads ----------------
    for (int p = 0; p < ch.n; ++p) {
      const SkGemm &g = ch.ph[p].gm;
      if (ch.ph[p].kind == PH_GEMM && !g.tiled)
        for (int k = 0; k < g.n_groups; ++k) prefetch_tmap(&maps.m[g.map0 + k]);
    }
    const uint64_t pol = l2_evict_first_policy();  // every weight byte is read once
    auto load_a = [&](const SkGemm &g, long long u, int s) {
      const int t = (int)(u / g.KB), kb = (int)(u - (long long)t * g.KB);
      const int group = g.n_groups > 1 ? t / g.tiles_per_group : 0;
      const int lt = t - group * (g.n_groups > 1 ? g.tiles_per_group : 0);
      if (g.tiled) {
        const uint16_t *src = g.wt[group] + ((long long)lt * g.KB + kb) * (KPS * BM * BK);
        bulk_load_hint(stage_a(s), src, C::STAGE_A, &full[s], pol);
      } else {
#pragma unroll
        for (int j = 0; j < KPS; ++j)
          tma_load_2d_hint(stage_a(s) + j * A_BYTES, &maps.m[g.map0 + group], &full[s],
                           (kb * KPS + j) * BK, lt * BM, pol);
      }
    };
    auto load_b = [&](const SkGemm &g, long long u, int s) {
      const int kb = (int)(u % g.KB);
      bulk_load(stage_b(s), g.x + (long long)kb * KPS * BN * BK, C::STAGE_B, &full[s]);
    };
    auto stop = [&]() {
      *(volatile int *)abort_flag = 1;
      set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
    };
    long long i = 0;  // units of this CTA so far, over all projections (the stage ring)
    int nph = 0;      // projections in which this CTA had units (all their loads issued)
    bool ok = true;
    for (int p = 0; p < ch.n && ok; ++p) {
      if (ch.ph[p].kind != PH_GEMM) continue;
      const SkGemm &g = ch.ph[p].gm;
      long long ub, ue;
      sk_run(g, c, &ub, &ue);
      const long long n = ue - ub;
      if (n == 0) continue;
      const long long pre = min((long long)STAGES, n);
      // The owner reduction at the end of this CTA's previous projection may borrow
      // the stage of that projection's last unit, which unit STAGES - 1 of this one
      // refills: wait for the epilogue to hand it back (epi_free) first.
      bool freed = nph == 0;
      const uint32_t fpar = (uint32_t)((nph - 1) & 1);
      // Weights do not depend on earlier phases or kernels: the weight part of the
      // first stages is requested before waiting for the inputs.
      long long k = 0;
      for (; k < pre; ++k) {
        const long long j = i + k;
        const int s = (int)(j % STAGES);
        if (!freed && k == STAGES - 1) {
          freed = true;
          if (!mbar_wait_bounded(epi_free, fpar)) {
            stop();
            ok = false;
            break;
          }
        }
        if (j >= STAGES && !mbar_wait_bounded(&empty[s], (uint32_t)((j / STAGES - 1) & 1))) {
          stop();
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        load_a(g, ub + k, s);
      }
      // inputs: the kernel before this one (first phase), else every CTA's phase p - 1
      if (ok) {
        if (p == 0) {
          pdl_wait();
        } else if (!grid_wait(ch.gbar, ch.bar_base + (unsigned)(p * G), dev_err)) {
          stop();
          ok = false;
        } else {
          // written by other CTAs' generic stores, read here by bulk copies
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
      }
      // (after a failed wait too: every requested stage must complete)
      for (long long q = 0; q < k; ++q) load_b(g, ub + q, (int)((i + q) % STAGES));
      for (; k < n && ok; ++k) {
        const long long j = i + k;
        const int s = (int)(j % STAGES);
        if (!mbar_wait_bounded(&empty[s], (uint32_t)((j / STAGES - 1) & 1))) {
          stop();
          ok = false;
          break;
        }
        if (*(volatile int *)abort_flag) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
        load_a(g, ub + k, s);
        load_b(g, ub + k, s);
      }
      i += k;
      if (ok && !freed && !mbar_wait_bounded(epi_free, fpar)) {
        stop();
        ok = false;
      }
      ++nph;
    }
    // no copy may still be in flight when the CTA exits
    for (long long j = i > STAGES ? i - STAGES : 0; j < i; ++j)
      if (!mbar_wait_bounded(&full[j % STAGES], (uint32_t)((j / STAGES) & 1)))
        set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
  } else if (warp == MMA && lane == 0) {
    // ---------------- MMA ----------------
    constexpr uint32_t idesc = idesc_f16kind<CT>(BN);
    int seg = 0;
    long long i = 0;
    bool ok = true;
    for (int p = 0; p < ch.n && ok; ++p) {
      if (ch.ph[p].kind != PH_GEMM) continue;
      const SkGemm &g = ch.ph[p].gm;
      long long ub, ue;
      sk_run(g, c, &ub, &ue);
      for (long long u = ub; u < ue && ok;) {
        const int t = (int)(u / g.KB), kb0 = (int)(u - (long long)t * g.KB);
        const int n = (int)min((long long)(g.KB - kb0), ue - u);
        const int buf = seg & 1;
        if (seg >= 2 && !mbar_wait_bounded(&acc_empty[buf], (uint32_t)(((seg >> 1) - 1) & 1))) {
          *(volatile int *)abort_flag = 1;
          set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t acc = tmem_base + (uint32_t)(buf * BN);
        for (int j = 0; j < n; ++j) {
          const long long q = i + (u - ub) + j;
          const int s = (int)(q % STAGES);
          if (!mbar_wait_bounded(&full[s], (uint32_t)((q / STAGES) & 1)) ||
              *(volatile int *)abort_flag) {
            *(volatile int *)abort_flag = 1;
            set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kq = 0; kq < KPS; ++kq) {
            const uint32_t a0 = smem_u32(stage_a(s) + kq * A_BYTES);
            const uint32_t b0 = smem_u32(stage_b(s) + kq * C::B_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / UMMA_K; ++kk)
              tc_mma_f16(acc, sdesc_sw128(a0 + kk * UMMA_K * 2), sdesc_sw128(b0 + kk * UMMA_K * 2),
                         idesc, (j | kq | kk) != 0);
          }
          tc_commit(&empty[s]);
        }
        tc_commit(&acc_full[buf]);  // also issued on abort so the epilogue is released
        u += n;
        ++seg;
      }
      i += ue - ub;
    }
  } else if (warp < EPW) {
    // ---------------- epilogue ----------------
    // With tile_cnt (element-wise epilogues) a tile split over S runs is finished
    // inside the kernel by its owner, the run holding its first k-blocks (slot 0;
    // for that run it is always the last segment, reached at the end of its
    // range): the other runs (whose part is their first segment, done early) write
    // fp32 slices and count themselves in the tile's counter; the owner waits for
    // the count, adds the slices to its own accumulator in slot order, applies the
    // epilogue and clears the counter.  The owner's staged reduction borrows
    // pipeline shared memory free after the CTA's last MMA of the projection: all
    // of it after the last projection of the launch, else the stage of that last
    // MMA (the producer refills it only after epi_free).  Without tile_cnt, tiles
    // of one run are stored directly and the others are left as slices for the
    // rows phase (or kernel) after.
    constexpr int W = BN >= 32 ? 32 : 16;
    const int quarter = warp & 3, half = warp >> 2;  // TMEM lanes 32 quarter.., column half
    int last_gemm = -1;
    for (int p = 0; p < ch.n; ++p)
      if (ch.ph[p].kind == PH_GEMM) last_gemm = p;
    // The bias of this thread's row in the tile an owner finishes at the end of its
    // run; for the first phase read before waiting on the kernel before this one.
    auto owner_bias = [&](const SkGemm &g, long long ue) {
      const int t_last = (int)((ue - 1) / g.KB);
      return tile_row_bias(g.epi, t_last * BM + quarter * 32 + lane, g.N);
    };
    float last_bias = 0.f;
    if (ch.ph[0].kind == PH_GEMM) {
      const SkGemm &g = ch.ph[0].gm;
      long long ub, ue;
      sk_run(g, c, &ub, &ue);
      if (g.tile_cnt && g.epi.kind != EPI_PARTIAL && ue > ub) last_bias = owner_bias(g, ue);
    }
    pdl_wait();  // outputs may still be read by the kernel before this one
    int seg = 0;
    long long i = 0;
    uint32_t fix_phase = 0;  // parity of fix_bar's next phase
    for (int p = 0; p < ch.n; ++p) {
      if (ch.ph[p].kind == PH_ROWS) {
        // every CTA's part of phase p - 1 is done
        if (threadIdx.x == 0)
          *gate = !*(volatile int *)abort_flag &&
                  grid_wait(ch.gbar, ch.bar_base + (unsigned)(p * G), dev_err);
        epi_bar_sync<EPT>();
        if (*gate) sk_rows_phase<CT>(ch.ph[p].rw, ch.M, c, G, red);
      } else {
        const SkGemm &g = ch.ph[p].gm;
        const Epi &epi = g.epi;
        long long ub, ue;
        sk_run(g, c, &ub, &ue);
        const bool fix = g.tile_cnt != nullptr && epi.kind != EPI_PARTIAL;
        if (p > 0 && fix && ue > ub) last_bias = owner_bias(g, ue);
        const bool last = p == last_gemm;
        uint8_t *stage_mem = last || ue == ub ? base : stage_a((int)((i + (ue - ub) - 1) % STAGES));
        const int avail = last ? STAGES * C::STAGE_BYTES : C::STAGE_BYTES;
        for (long long u = ub; u < ue;) {
          const int t = (int)(u / g.KB), kb0 = (int)(u - (long long)t * g.KB);
          const int n = (int)min((long long)(g.KB - kb0), ue - u);
          const int buf = seg & 1;
          const bool ok = !*(volatile int *)abort_flag &&
                          mbar_wait_bounded(&acc_full[buf], (uint32_t)((seg >> 1) & 1));
          if (!ok) set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
          tc_fence_after();
          const bool live = ok && !*(volatile int *)abort_flag;
          int cf, S;
          sk_segments(t, g.KB, g.P, g.U, &cf, &S);
          const int slot = c - cf;
          const int row = t * BM + quarter * 32 + lane;
          const uint32_t tl = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(buf * BN);
          // (all conditions below are uniform over the epilogue warps)
          const bool staged = fix && slot == 0 && u + n == ue &&
                              tile_stage_tokens(S, ch.M, W, avail) >= W;
          if (staged) {
            tile_owner_epilogue<CT, W, EPT>(epi, g.slices + (size_t)t * ch.M * BM, g.slice_stride,
                                            g.N, ch.M, t, S, tl, live, &g.tile_cnt[t], stage_mem,
                                            avail, fix_bar, fix_phase, last_flag, dev_err,
                                            last_bias);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
          } else {
            const bool direct = S == 1 && epi.kind != EPI_PARTIAL;
            RowEpi<CT> re = row_epi_prepare<CT>(epi, row < g.N ? row : 0,
                                                direct ? nullptr : g.slices, g.slice_stride,
                                                slot, g.N);
            if (fix && !direct) {  // tile-contiguous slices: [slot][tile][M][128]
              re.f32 = g.slices + slot * g.slice_stride + (size_t)t * ch.M * BM + (row - t * BM);
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
              if (live && row < g.N && c0 < ch.M)
                row_epi_store<CT, WH>(re, c0, min(WH, ch.M - c0), v);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            if (fix && S > 1) {
              // this run's slice is complete: count it (release), every run of the
              // tile including an owner without room for the staged reduction
              __threadfence();
              epi_bar_sync<EPT>();
              if (threadIdx.x == 0 && live) atomicAdd(&g.tile_cnt[t], 1);
              if (slot == 0) {
                // owner: wait for all S slices, then reduce them through registers
                if (threadIdx.x == 0) {
                  bool ok2 = live && wait_count_at_least(&g.tile_cnt[t], S);
                  if (live && !ok2) set_dev_error(dev_err, DEVERR_WAIT_TIMEOUT);
                  *last_flag = ok2;
                }
                epi_bar_sync<EPT>();
                if (*last_flag) {
                  __threadfence();
                  tile_fixup<CT, EPT>(epi, g.slices + (size_t)t * ch.M * BM, g.slice_stride, g.N,
                                      ch.M, t, S, threadIdx.x);
                  if (threadIdx.x == 0) g.tile_cnt[t] = 0;
                }
              }
            }
          }
          u += n;
          ++seg;
        }
        if (ue > ub) {
          // the borrowed stage is free again (generic accesses ordered before the
          // producer's bulk copies into it)
          fence_proxy_async_smem();
          epi_bar_sync<EPT>();
          if (threadIdx.x == 0) mbar_arrive(epi_free);
        }
        i += ue - ub;
      }
      if (p + 1 < ch.n) {
        // this CTA's part of phase p is written: arrive (release) at the grid barrier,
        // after having seen every CTA finish phase p - 1 (so that the counter passes
        // bar_base + (p + 1) G only once all CTAs are through phase p)
        __threadfence();
        epi_bar_sync<EPT>();
        if (threadIdx.x == 0) {
          if (p > 0) grid_wait(ch.gbar, ch.bar_base + (unsigned)(p * G), dev_err);
          atomicAdd(ch.gbar, 1u);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == MMA) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

template <typename CT, int BN, int STAGES, int KPS>
cudaError_t launch_sk_bn(const SkMaps &maps, const SkChain &chn, int G, int *dev_err,
                         cudaStream_t st) {
  using C = SkCfg<BN, STAGES, KPS>;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(k_gemm_sk<CT, BN, STAGES, KPS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  return launch_k(k_gemm_sk<CT, BN, STAGES, KPS>, dim3(G), dim3(SK_THREADS), C::SMEM, st, g_pdl,
                  maps, chn, dev_err);
}

}  // namespace

int sk_kps(const GemmArgs &g) { return g.K % 128 == 0 ? 2 : 1; }

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
    default:
      return false;
  }
}

namespace {

// One projection's kernel arguments (and tensor maps for row-major weights).
cudaError_t sk_gemm_phase(const GemmArgs &g, int P, float *slices, long long slice_stride,
                          int *tile_cnt, SkGemm *o, SkMaps *maps, int *n_maps) {
  // one row tile of tokens (M <= 256), whole 128 x 64 tiles, fp32 slices
  if ((g.act != ACT_BF16 && g.act != ACT_F16) || g.M < 1 || g.M > 256 || g.K % BK)
    return cudaErrorInvalidValue;
  if (g.w_tiled && (g.group_rows % BM)) return cudaErrorInvalidValue;
  if (g.n_groups < 1 || g.n_groups > 3 || g.n_groups * g.group_rows != g.N) return cudaErrorInvalidValue;
  if (g.epi.kind == EPI_QKV && g.epi.d_model % BM) return cudaErrorInvalidValue;
  if (!slices || P < 1 || slice_stride < (long long)g.M * g.N) return cudaErrorInvalidValue;
  if (tile_cnt && (!sk_fixup_ok(g) || (uintptr_t)slices % 16 ||
                   slice_stride < (long long)g.M * ((g.N + BM - 1) / BM) * BM))
    return cudaErrorInvalidValue;
  if ((uintptr_t)g.x % 16) return cudaErrorInvalidValue;  // activations arrive by bulk copy
  const bool fp16 = g.act == ACT_F16;
  memset(o, 0, sizeof *o);
  o->tiled = g.w_tiled;
  o->n_groups = g.n_groups;
  o->tiles_per_group = g.n_groups > 1 ? g.group_rows / BM : 1;
  o->map0 = *n_maps;
  for (int i = 0; i < 3; ++i) {
    const void *p = g.w[i < g.n_groups ? i : 0];
    if (g.w_tiled) {
      o->wt[i] = static_cast<const uint16_t *>(p);
    } else if (i < g.n_groups) {
      if (*n_maps >= kMaxMaps) return cudaErrorInvalidValue;
      if (!make_tmap_16(&maps->m[*n_maps], p, g.group_rows, g.K, g.K, BM, fp16))
        return cudaErrorInvalidValue;
      ++*n_maps;
    }
  }
  o->N = g.N;
  o->KB = g.K / (BK * sk_kps(g));
  o->U = (long long)((g.N + BM - 1) / BM) * o->KB;
  o->P = P;
  o->x = static_cast<const uint16_t *>(g.x);
  o->slices = slices;
  o->slice_stride = slice_stride;
  o->tile_cnt = tile_cnt;
  o->epi = g.epi;
  return cudaSuccess;
}

bool al16(const void *p) { return (uintptr_t)p % 16 == 0; }

}  // namespace

cudaError_t launch_gemm_chain(const ChainPhase *ph, int n, int G, unsigned *gbar,
                              unsigned bar_base, int *dev_err, cudaStream_t st) {
  if (!ph || n < 1 || n > kMaxPhases || G < 1 || (n > 1 && !gbar)) return cudaErrorInvalidValue;
  SkChain chn;
  SkMaps maps;
  memset(&chn, 0, sizeof chn);
  memset(&maps, 0, sizeof maps);
  chn.n = n;
  chn.gbar = gbar;
  chn.bar_base = bar_base;
  int n_maps = 0, act = -1, kps = 0, M = 0;
  for (int p = 0; p < n; ++p) {
    SkPhase &o = chn.ph[p];
    o.kind = ph[p].kind;
    if (ph[p].kind == PH_GEMM) {
      const GemmArgs &g = ph[p].g;
      if (ph[p].P > G || (act >= 0 && (g.act != act || sk_kps(g) != kps || g.M != M)))
        return cudaErrorInvalidValue;
      act = g.act;
      kps = sk_kps(g);
      M = g.M;
      cudaError_t e = sk_gemm_phase(g, ph[p].P, ph[p].slices, ph[p].slice_stride, ph[p].tile_cnt,
                                    &o.gm, &maps, &n_maps);
      if (e != cudaSuccess) return e;
    } else if (ph[p].kind != PH_ROWS) {
      return cudaErrorInvalidValue;
    }
  }
  if (act < 0) return cudaErrorInvalidValue;
  chn.M = M;
  for (int p = 0; p < n; ++p) {
    if (ph[p].kind != PH_ROWS) continue;
    const ChainPhase &r = ph[p];
    // the arithmetic of k_resid_ln8 (d / 8 <= 1024 groups in whole warps), here at
    // most kRowGroups per epilogue thread; 16-byte loads and stores
    if (r.d % 256 || r.d / 8 > kRowGroups * EPT || r.ldp % 4 || r.split_stride % 4)
      return cudaErrorInvalidValue;
    if (r.out_act != act && r.out_act != ACT_BF16) return cudaErrorInvalidValue;
    if (!al16(r.partial) || !al16(r.x) || !al16(r.h) || !al16(r.bias) || !al16(r.gamma) ||
        !al16(r.beta))
      return cudaErrorInvalidValue;
    SkRows &w = chn.ph[p].rw;
    w.partial = r.partial;
    w.si = r.si;
    w.split_stride = r.split_stride;
    w.ldp = r.ldp;
    w.bias = static_cast<const bf16 *>(r.bias);
    w.gamma = static_cast<const bf16 *>(r.gamma);
    w.beta = static_cast<const bf16 *>(r.beta);
    w.x = r.x;
    w.eps = r.eps;
    w.h = r.h;
    w.h_rows = r.h_rows;
    w.d = r.d;
    w.out_bf16 = r.out_act == ACT_BF16;
  }
  auto pick = [&](auto ct) -> cudaError_t {
    using CT = decltype(ct);
#define HE_SK(BN, ST, KPS) return launch_sk_bn<CT, BN, ST, KPS>(maps, chn, G, dev_err, st)
    if (kps == 2) {
      // two k-blocks per stage: 32 KB weight requests
      if (M <= 16) HE_SK(16, 5, 2);
      if (M <= 32) HE_SK(32, 5, 2);
      if (M <= 64) HE_SK(64, 4, 2);
      if (M <= 128) HE_SK(128, 3, 2);
      HE_SK(256, 2, 2);
    }
    if (M <= 16) HE_SK(16, 10, 1);
    if (M <= 32) HE_SK(32, 9, 1);
    if (M <= 64) HE_SK(64, 8, 1);
    if (M <= 128) HE_SK(128, 6, 1);
    HE_SK(256, 4, 1);
#undef HE_SK
  };
  if (act == ACT_BF16) return pick(bf16{});
  return pick(f16{});
}

cudaError_t launch_gemm_sk(const GemmArgs &g, int P, float *slices, long long slice_stride,
                           int *tile_cnt, int *dev_err, cudaStream_t st) {
  ChainPhase one{};
  one.kind = PH_GEMM;
  one.g = g;
  one.P = P;
  one.slices = slices;
  one.slice_stride = slice_stride;
  one.tile_cnt = tile_cnt;
  return launch_gemm_chain(&one, 1, P, nullptr, 0, dev_err, st);
}

}  // namespace he
