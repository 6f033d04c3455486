// CUDA-core (FFMA) GEMM with the block's fused epilogues.
//
// Serves the fp32 workloads (fp32 tensor cores would round operands to TF32,
// which cannot meet a 1e-5 relative error) and any operand shape the
// tensor-core kernel does not take (unaligned leading dimensions).  Tiles of
// 64 x 64 outputs, K staged 16 at a time through shared memory as fp32; each
// of the 256 threads owns a 4 x 4 register block whose rows are 16 apart and
// whose columns are 16 apart, so the epilogue stores are coalesced.
#include "epilogue.cuh"

namespace oases {
namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

template <typename T>
__global__ void __launch_bounds__(NT) gemm_simt_kernel(const GemmArgs g) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN + 4];
  pdl_wait();
  pdl_trigger();
  const T* A = static_cast<const T*>(g.A);
  const T* B = static_cast<const T*>(g.B);
  const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
  const int m0 = blockIdx.y * BM, n0 = blockIdx.x * BN;
  float acc[4][4] = {};
  for (int k0 = 0; k0 < g.K; k0 += BK) {
#pragma unroll
    for (int r = 0; r < (BM * BK) / NT; ++r) {
      const int idx = tid + r * NT;
      int m, k;
      if (g.a_kmajor) { m = idx / BK; k = idx % BK; } else { k = idx / BM; m = idx % BM; }
      const int gm = m0 + m, gk = k0 + k;
      float v = 0.f;
      if (gm < g.M && gk < g.K)
        v = ld_elem(A, g.a_kmajor ? (int64_t)gm * g.lda + gk : (int64_t)gk * g.lda + gm);
      As[k][m] = v;
    }
#pragma unroll
    for (int r = 0; r < (BN * BK) / NT; ++r) {
      const int idx = tid + r * NT;
      int n, k;
      if (g.b_kmajor) { n = idx / BK; k = idx % BK; } else { k = idx / BN; n = idx % BN; }
      const int gn = n0 + n, gk = k0 + k;
      float v = 0.f;
      if (gn < g.N && gk < g.K)
        v = ld_elem(B, g.b_kmajor ? (int64_t)gn * g.ldb + gk : (int64_t)gk * g.ldb + gn);
      Bs[k][n] = v;
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < BK; ++k) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[k][ty + 16 * i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[k][tx + 16 * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int m = m0 + ty + 16 * i;
    if (m >= g.M) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx + 16 * j;
      if (n < g.N) epi_apply(g, m, n, acc[i][j]);
    }
  }
}

}  // namespace

cudaError_t gemm_simt(const GemmArgs& g, cudaStream_t st) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  if (g.in_t == DType::E4M3) return cudaErrorNotSupported;  // E4M3 runs on the MX path only
  dim3 grid((g.N + BN - 1) / BN, (g.M + BM - 1) / BM);
  if (grid.y > 65535) return cudaErrorInvalidConfiguration;
  if (g.in_t == DType::F32) return launch_pdl(gemm_simt_kernel<float>, grid, dim3(NT), 0, st, g);
  return launch_pdl(gemm_simt_kernel<__nv_bfloat16>, grid, dim3(NT), 0, st, g);
}

}  // namespace oases
