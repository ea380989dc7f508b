// Per-element GEMM epilogue shared by the tcgen05 GEMM, the fp32 CUDA-core GEMM
// and the split-K reduction.
#pragma once
#include "common.cuh"
#include "kernels.h"

namespace he {

// Store one finished element C[tok][n] (split slice `s` for EPI_PARTIAL).  PT: bias
// type; CT: type of the q / K / V / ReLU outputs.
template <typename PT, typename CT>
__device__ __forceinline__ void epi_store(const Epi &e, int s, int tok, int n, float acc) {
  switch (e.kind) {
    case EPI_PARTIAL:
      e.partial[(long long)s * e.split_stride + (long long)tok * e.ldp + n] = acc;
      break;
    case EPI_STORE_F32:
      e.partial[(long long)tok * e.ldp + n] = acc;
      break;
    case EPI_RELU: {
      float v = acc + to_f<PT>(static_cast<const PT *>(e.bias[0])[n]);
      static_cast<CT *>(e.out)[act_index(tok, n, e.ldo, e.out_rows)] = from_f<CT>(fmaxf(v, 0.f));
      break;
    }
    case EPI_QKV: {
      const int which = n / e.d_model;  // 0 = q, 1 = k, 2 = v
      const int c = n - which * e.d_model;
      float v = acc + to_f<PT>(static_cast<const PT *>(e.bias[which])[c]);
      if (which == 0) {
        static_cast<CT *>(e.out)[(long long)tok * e.ldo + c] = from_f<CT>(v * e.q_scale);
      } else {
        const int b = tok / e.tok_per_seq;
        const int t = e.pos0 + (tok - b * e.tok_per_seq);
        const int hh = c / e.head_dim, dd = c - hh * e.head_dim;
        CT *cache = static_cast<CT *>(which == 1 ? e.kc : e.vc);
        cache[(((long long)b * e.n_heads + hh) * e.max_seq + t) * e.head_dim + dd] = from_f<CT>(v);
      }
      break;
    }
  }
}

}  // namespace he
