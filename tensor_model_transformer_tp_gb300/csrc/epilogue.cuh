// Per-element GEMM epilogue shared by the SIMT and tensor-core kernels.
#pragma once
#include "common.cuh"

namespace oases {

// Applies g.epi to one accumulator value of output element (m, n).
__device__ __forceinline__ void epi_apply(const GemmArgs& g, int m, int n, float acc) {
  const int64_t ci = (int64_t)m * g.ldc + n;
  switch (g.epi) {
    case Epi::Store:
      store_any(g.C, g.c_t, ci, acc);
      break;
    case Epi::Bias:
      store_any(g.C, g.c_t, ci, acc + load_any(g.bias, g.in_t, n));
      break;
    case Epi::BiasGelu: {
      const float a = acc + load_any(g.bias, g.in_t, n);
      if (g.C2) store_any(g.C2, g.c_t, ci, gelu_grad_f(a));
      store_any(g.C, g.c_t, ci, gelu_f(a));
      break;
    }
    case Epi::BiasResid:
      store_any(g.C, g.c_t, ci,
                acc + load_any(g.bias, g.in_t, n) +
                    load_any(g.aux, g.aux_t, (int64_t)m * g.ld_aux + n));
      break;
    case Epi::Mul:
      store_any(g.C, g.c_t, ci, acc * load_any(g.aux, g.aux_t, (int64_t)m * g.ld_aux + n));
      break;
    case Epi::Accum: {
      float* c = static_cast<float*>(g.C);
      c[ci] += acc;
      break;
    }
  }
}

}  // namespace oases
