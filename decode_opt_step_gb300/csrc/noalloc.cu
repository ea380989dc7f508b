// he_op_attn_decode_noalloc: the decode attention with its split-over-keys
// partial results kept in a fixed, statically allocated device array instead of a
// caller-provided buffer.
//
// Why: some callers of this library cannot allocate device memory at the moment
// they need the attention.  Code recorded into a CUDA graph must not call
// cudaMalloc / cudaFree while capturing; runtimes whose device memory is owned by
// a pooling allocator or a fixed budget cannot hand out an extra buffer on
// demand; and latency-critical loops avoid cudaMalloc because it can synchronise
// the device.  This entry point needs nothing from them but inputs and outputs.
//
// The scratch is one file-scope __device__ array, so every GPU that loads the
// library holds it (kNoAllocScratchFloats floats, 16 MiB) until the process ends.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/he.h"
#include "../../include/he_ops.h"
#include "kernels.h"

namespace {

constexpr long long kNoAllocScratchFloats = 4LL * 1024 * 1024;  // 16 MiB of fp32

static __device__ __align__(256) float g_attn_partials[kNoAllocScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_addr_mu;
float *g_addr[kMaxDevices] = {};  // device address of g_attn_partials, per device

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
  float *part = nullptr;
  {
    // First call on a device: look up the array's device address (with that device
    // current).  This is host-side set-up only; it allocates nothing.
    std::lock_guard<std::mutex> lock(g_addr_mu);
    if (!g_addr[dev]) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_attn_partials) != cudaSuccess || !p)
        return he::set_error(HE_ERR_CUDA, "cudaGetSymbolAddress of the built-in scratch failed");
      g_addr[dev] = static_cast<float *>(p);
    }
    part = g_addr[dev];
  }
  // Every slot of the scratch the launch reads is written by the same launch's
  // first kernel before the combine kernel reads it, so nothing is cleared.
  const cudaError_t r = he::launch_attn_decode(dtype, q, kc, vc, ctx, 0, B, H, hd, max_seq,
                                               n_keys, split, part,
                                               static_cast<cudaStream_t>(stream));
  if (r != cudaSuccess) return he::set_error(HE_ERR_CUDA, cudaGetErrorString(r));
  return he::set_error(HE_OK, "");
}
