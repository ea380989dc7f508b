// fp32 GEMM on CUDA cores (the fp32 workload keeps full fp32 arithmetic, so it
// does not go through the bf16 tensor-core kernel), and the dtype dispatch.
#include "common.cuh"
#include "epilogue.cuh"
#include "kernels.h"

namespace he {

cudaError_t launch_gemm_tc(const GemmArgs &a, int *dev_err, cudaStream_t st);

namespace {

constexpr int TT = 64;   // tokens per tile
constexpr int TN = 64;   // output features per tile
constexpr int TK = 16;   // K per smem step

// C[tok][n] over a 64 x 64 tile; 256 threads, 4 x 4 outputs each; the K loop of
// split `blockIdx.z` covers 64-wide blocks [z * kb_per_split, ...).
template <typename T>
__global__ void __launch_bounds__(256)
    k_gemm_simt(const T *__restrict__ x, int ldx, const T *w0, const T *w1, const T *w2,
                int group_rows, int M, int N, int K, int kb_per_split,
                const __grid_constant__ Epi epi) {
  __shared__ float xs[TK][TT + 4];
  __shared__ float ws[TK][TN + 4];
  const int tok0 = blockIdx.y * TT, n0 = blockIdx.x * TN, split = blockIdx.z;
  const int k_begin = split * kb_per_split * 64;
  const int k_end = min(K, k_begin + kb_per_split * 64);
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int k0 = k_begin; k0 < k_end; k0 += TK) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int e = threadIdx.x + i * 256;
      const int r = e / TK, kk = e % TK, k = k0 + kk;
      const int tok = tok0 + r;
      xs[kk][r] = (tok < M && k < k_end) ? to_f<T>(x[(long long)tok * ldx + k]) : 0.f;
      const int n = n0 + r;
      float wv = 0.f;
      if (n < N && k < k_end) {
        const int g = n / group_rows;
        const T *wg = g == 0 ? w0 : (g == 1 ? w1 : w2);
        wv = to_f<T>(wg[(long long)(n - g * group_rows) * K + k]);
      }
      ws[kk][r] = wv;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < TK; ++kk) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = ws[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int tok = tok0 + ty * 4 + i, n = n0 + tx * 4 + j;
      if (tok < M && n < N) epi_store<T, T>(epi, split, tok, n, acc[i][j]);
    }
}

}  // namespace

cudaError_t launch_gemm(const GemmArgs &a, int *dev_err, cudaStream_t st) {
  if (a.act != ACT_F32) return launch_gemm_tc(a, dev_err, st);
  if (a.M <= 0 || a.N <= 0 || a.K <= 0 || a.n_groups < 1 || a.n_groups > 3)
    return cudaErrorInvalidValue;
  if (a.n_groups * a.group_rows != a.N) return cudaErrorInvalidValue;
  if (effective_split(a.K, a.split) != a.split) return cudaErrorInvalidValue;
  dim3 grid((a.N + TN - 1) / TN, (a.M + TT - 1) / TT, a.split);
  const float *w0 = static_cast<const float *>(a.w[0]);
  const float *w1 = static_cast<const float *>(a.n_groups > 1 ? a.w[1] : a.w[0]);
  const float *w2 = static_cast<const float *>(a.n_groups > 2 ? a.w[2] : a.w[0]);
  k_gemm_simt<float><<<grid, 256, 0, st>>>(static_cast<const float *>(a.x), a.ldx, w0, w1, w2,
                                           a.group_rows, a.M, a.N, a.K,
                                           split_kblocks(a.K, a.split), a.epi);
  return cudaGetLastError();
}

// Split-K for the skinny decode GEMMs.  A cost model picks S: one CTA per SM,
// each SM streams ceil(units / SMs) units of 128 weight rows x K/S at a per-SM
// rate, while the whole GEMM moves the weights plus the fp32 partial slices
// (written and read back) at the HBM rate; the slower of the two is the time.
int gemm_pick_split(const GemmArgs &a, int num_sms) {
  const bool tc = a.act != ACT_F32;
  const int bm = tc ? 128 : TN;
  const int bn = tc ? (a.M <= 16 ? 16 : a.M <= 32 ? 32 : a.M <= 64 ? 64 : a.M <= 128 ? 128 : 256) : TT;
  const long long tiles = (long long)((a.N + bm - 1) / bm) * ((a.M + bn - 1) / bn);
  const int kb = (a.K + 63) / 64;
  const double esz = tc ? 2.0 : 4.0;
  const double hbm = 6.5e12, per_sm = 80e9;
  const double wbytes = (double)a.N * a.K * esz;
  int best = 1;
  double best_t = 1e30;
  for (int s = 1; s <= 16 && s <= kb; ++s) {
    if (effective_split(a.K, s) != s) continue;
    const long long units = tiles * s;
    const long long per = (units + num_sms - 1) / num_sms;
    const double unit_bytes = (double)bm * split_kblocks(a.K, s) * 64 * esz;
    const double t_sm = per * unit_bytes / per_sm;
    const double partial = s > 1 ? 2.0 * s * (double)a.M * a.N * 4.0 : 0.0;
    const double t = (t_sm > (wbytes + partial) / hbm ? t_sm : (wbytes + partial) / hbm) +
                     (s > 1 ? 2e-6 : 0.0);
    if (t < best_t * 0.98) {
      best_t = t;
      best = s;
    }
  }
  return best;
}

}  // namespace he
