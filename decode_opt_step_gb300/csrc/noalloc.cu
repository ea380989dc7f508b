// he_op_attn_decode_noalloc: the decode attention with its split-over-keys
// partial results kept in a fixed, statically allocated device array instead of a
// caller-provided buffer.
//
// Why: some callers of this library cannot allocate device memory at the moment
// they need the attention.  Runtimes whose device memory is owned by a pooling
// allocator or a fixed budget cannot hand out an extra buffer on demand; plugins
// hosted by another framework may have no allocator of their own; and
// latency-critical loops avoid cudaMalloc because it can synchronise the device.
// This entry point needs nothing from them but inputs and outputs.
//
// The scratch is one file-scope __device__ array, so every GPU that loads the
// library holds it (kNoAllocScratchFloats floats, 16 MiB) until the process ends.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "../../include/he.h"
#include "../../include/he_ops.h"
#include "kernels.h"

namespace {

constexpr long long kNoAllocScratchFloats = 4LL * 1024 * 1024;  // 16 MiB of fp32

static __device__ __align__(256) float g_attn_partials[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;

// The array's device address is looked up once per device with that device
// current, and kept with the context it was looked up in: a later call in another
// context of the same ordinal (after cudaDeviceReset, say) looks it up again.
// The address is stored before its context, so a reader that finds its context
// also finds that context's address.
struct ScratchAddr {
  std::atomic<CUcontext> ctx{nullptr};
  std::atomic<float *> addr{nullptr};
};
ScratchAddr g_scratch[kMaxDevices];
std::mutex g_lookup_mu;  // serialises the lookups, not the reads

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<CtxGetCurrentFn>(p);
  }();
  return fn;
}

// Device address of g_attn_partials in the current context, or null.
float *scratch_address(int dev) {
  CtxGetCurrentFn get_ctx = ctx_get_current();
  CUcontext cur = nullptr;
  if (!get_ctx || get_ctx(&cur) != CUDA_SUCCESS || !cur) return nullptr;
  ScratchAddr &s = g_scratch[dev];
  if (s.ctx.load(std::memory_order_acquire) == cur) return s.addr.load(std::memory_order_relaxed);
  std::lock_guard<std::mutex> lock(g_lookup_mu);
  if (s.ctx.load(std::memory_order_acquire) == cur) return s.addr.load(std::memory_order_relaxed);
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_attn_partials) != cudaSuccess || !p) return nullptr;
  s.addr.store(static_cast<float *>(p), std::memory_order_relaxed);
  s.ctx.store(cur, std::memory_order_release);
  return static_cast<float *>(p);
}

}  // namespace

namespace he {
he_status set_error(he_status s, const char *msg);  // engine.cu
}

extern "C" he_status he_op_attn_decode_noalloc(int dtype, const void *q, const void *kc,
                                               const void *vc, void *ctx, int B, int H, int hd,
                                               int max_seq, int n_keys, int split,
                                               void *stream) {
  if (!q || !kc || !vc || !ctx) return he::set_error(HE_ERR_ARG, "NULL buffer");
  if (dtype != HE_DTYPE_F32 && dtype != HE_DTYPE_BF16 && dtype != HE_DTYPE_F16)
    return he::set_error(HE_ERR_ARG, "bad dtype");
  if (B < 1 || H < 1 || n_keys < 1 || n_keys > max_seq || split < 1 || split > n_keys)
    return he::set_error(HE_ERR_ARG, "bad sizes");
  if (hd != 32 && hd != 64 && hd != 128) return he::set_error(HE_ERR_UNSUPPORTED, "bad head_dim");
  const long long need = split > 1 ? (long long)B * H * split * (hd + 2) : 0;
  if (need > kNoAllocScratchFloats)
    return he::set_error(HE_ERR_ARG,
                         "B * H * split * (head_dim + 2) exceeds the 4194304-float (16 MiB) "
                         "built-in scratch of he_op_attn_decode_noalloc; lower split");
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return he::set_error(HE_ERR_CUDA, "cudaGetDevice failed");
  // First call on a device (or in a new context): look up the array's device
  // address with that device current.  Host-side set-up only; it allocates nothing.
  float *part = scratch_address(dev);
  if (!part) {
    cudaGetLastError();
    return he::set_error(HE_ERR_CUDA, "device address of the built-in scratch not found");
  }
  // Every slot of the scratch the launch reads is written by the same launch's
  // first kernel before the combine kernel reads it, so nothing is cleared.
  const cudaError_t r = he::launch_attn_decode(dtype, q, kc, vc, ctx, 0, B, H, hd, max_seq,
                                               n_keys, split, part,
                                               static_cast<cudaStream_t>(stream));
  if (r != cudaSuccess) return he::set_error(HE_ERR_CUDA, cudaGetErrorString(r));
  return he::set_error(HE_OK, "");
}
