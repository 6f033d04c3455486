// LayerNorm forward / backward and deterministic column reductions.
//
// These kernels are HBM-bound: one warp owns one row for the row-wise passes
// (mean, variance, normalise; or the two row means of the backward), and the
// column sums (dgamma, dbeta, bias gradients) are taken in two fixed-order
// stages — per block of ROWS_PER_PART rows into a partial buffer, then over the
// partials — so the result does not depend on scheduling.
#include <algorithm>

#include "common.cuh"

namespace oases {
namespace {

constexpr int ROWS_PER_PART = 64;
constexpr int WARPS = 8;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <typename T>
__global__ void __launch_bounds__(WARPS * 32)
ln_fwd_kernel(const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
              T* __restrict__ u, float* __restrict__ mean, float* __restrict__ rstd, int M, int H,
              float eps) {
  const int row = blockIdx.x * WARPS + threadIdx.x / 32, lane = threadIdx.x % 32;
  if (row >= M) return;
  const T* xr = x + (int64_t)row * H;
  float s = 0.f;
  for (int c = lane; c < H; c += 32) s += ld_elem(xr, c);
  const float mu = warp_sum(s) / H;
  float v = 0.f;
  for (int c = lane; c < H; c += 32) {
    const float d = ld_elem(xr, c) - mu;
    v = fmaf(d, d, v);
  }
  const float rs = rsqrtf(warp_sum(v) / H + eps);
  T* ur = u + (int64_t)row * H;
  for (int c = lane; c < H; c += 32)
    st_elem(ur, c, (ld_elem(xr, c) - mu) * rs * ld_elem(gamma, c) + ld_elem(beta, c));
  if (lane == 0) {
    mean[row] = mu;
    rstd[row] = rs;
  }
}

// dx = rstd * (g - mean(g) - xhat * mean(g * xhat)) (+ dres), g = du * gamma.
template <typename T>
__global__ void __launch_bounds__(WARPS * 32)
ln_bwd_dx_kernel(const float* __restrict__ du, const T* __restrict__ x,
                 const float* __restrict__ mean, const float* __restrict__ rstd,
                 const T* __restrict__ gamma, const T* __restrict__ dres, T* __restrict__ dx,
                 int M, int H) {
  const int row = blockIdx.x * WARPS + threadIdx.x / 32, lane = threadIdx.x % 32;
  if (row >= M) return;
  const float* dur = du + (int64_t)row * H;
  const T* xr = x + (int64_t)row * H;
  const float mu = mean[row], rs = rstd[row];
  float s1 = 0.f, s2 = 0.f;
  for (int c = lane; c < H; c += 32) {
    const float gg = dur[c] * ld_elem(gamma, c);
    const float xh = (ld_elem(xr, c) - mu) * rs;
    s1 += gg;
    s2 = fmaf(gg, xh, s2);
  }
  const float m1 = warp_sum(s1) / H, m2 = warp_sum(s2) / H;
  T* dxr = dx + (int64_t)row * H;
  const T* dr = dres ? dres + (int64_t)row * H : nullptr;
  for (int c = lane; c < H; c += 32) {
    const float gg = dur[c] * ld_elem(gamma, c);
    const float xh = (ld_elem(xr, c) - mu) * rs;
    float v = rs * (gg - m1 - xh * m2);
    if (dr) v += ld_elem(dr, c);
    st_elem(dxr, c, v);
  }
}

// part_g[blk, n] = sum_{m in blk} du[m, n] * xhat[m, n]; part_b[blk, n] = sum du.
template <typename T>
__global__ void ln_bwd_param_part_kernel(const float* __restrict__ du, const T* __restrict__ x,
                                         const float* __restrict__ mean,
                                         const float* __restrict__ rstd, float* __restrict__ pg,
                                         float* __restrict__ pb, int M, int H) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= H) return;
  const int m0 = blockIdx.y * ROWS_PER_PART, m1 = min(M, m0 + ROWS_PER_PART);
  float sg = 0.f, sb = 0.f;
  for (int m = m0; m < m1; ++m) {
    const float d = du[(int64_t)m * H + n];
    sg = fmaf(d, (ld_elem(x, (int64_t)m * H + n) - mean[m]) * rstd[m], sg);
    sb += d;
  }
  pg[(int64_t)blockIdx.y * H + n] = sg;
  pb[(int64_t)blockIdx.y * H + n] = sb;
}

template <typename T>
__global__ void colsum_part_kernel(const T* __restrict__ in, int64_t ld, int M, int N,
                                   float* __restrict__ part) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  const int m0 = blockIdx.y * ROWS_PER_PART, m1 = min(M, m0 + ROWS_PER_PART);
  float s = 0.f;
  for (int m = m0; m < m1; ++m) s += ld_elem(in, (int64_t)m * ld + n);
  part[(int64_t)blockIdx.y * N + n] = s;
}

// out[n] += sum_b part[b, n] in order b = 0, 1, ...; two outputs at once when
// part2/out2 are given.
__global__ void part_reduce_kernel(const float* __restrict__ part, float* __restrict__ out,
                                   const float* __restrict__ part2, float* __restrict__ out2,
                                   int nb, int N) {
  const int n = blockIdx.x * blockDim.x + threadIdx.x;
  if (n >= N) return;
  float s = 0.f;
  for (int b = 0; b < nb; ++b) s += part[(int64_t)b * N + n];
  out[n] += s;
  if (part2) {
    float s2 = 0.f;
    for (int b = 0; b < nb; ++b) s2 += part2[(int64_t)b * N + n];
    out2[n] += s2;
  }
}

template <typename T>
__global__ void add_into_kernel(const T* __restrict__ a, const float* __restrict__ b,
                                T* __restrict__ out, int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v = b[i];
    if (a) v += ld_elem(a, i);
    st_elem(out, i, v);
  }
}

}  // namespace

int ln_bwd_blocks(int M) { return (M + ROWS_PER_PART - 1) / ROWS_PER_PART; }
int colsum_blocks(int M) { return (M + ROWS_PER_PART - 1) / ROWS_PER_PART; }

cudaError_t layer_norm_fwd(const void* x, const void* gamma, const void* beta, void* u,
                           float* mean, float* rstd, int M, int H, float eps, DType t,
                           cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  const int grid = (M + WARPS - 1) / WARPS;
  if (t == DType::F32)
    ln_fwd_kernel<float><<<grid, WARPS * 32, 0, st>>>(
        (const float*)x, (const float*)gamma, (const float*)beta, (float*)u, mean, rstd, M, H, eps);
  else
    ln_fwd_kernel<__nv_bfloat16><<<grid, WARPS * 32, 0, st>>>(
        (const __nv_bfloat16*)x, (const __nv_bfloat16*)gamma, (const __nv_bfloat16*)beta,
        (__nv_bfloat16*)u, mean, rstd, M, H, eps);
  OASES_COUNT_LAUNCH();
  return cudaGetLastError();
}

cudaError_t layer_norm_bwd(const float* du, const void* x, const float* mean, const float* rstd,
                           const void* gamma, const void* dres, void* dx, float* part_g,
                           float* part_b, float* dgamma, float* dbeta, int M, int H, DType t,
                           cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  const int grid = (M + WARPS - 1) / WARPS;
  const int nb = ln_bwd_blocks(M);
  dim3 pgrid((H + 255) / 256, nb);
  if (t == DType::F32) {
    ln_bwd_dx_kernel<float><<<grid, WARPS * 32, 0, st>>>(du, (const float*)x, mean, rstd,
                                                         (const float*)gamma, (const float*)dres,
                                                         (float*)dx, M, H);
    ln_bwd_param_part_kernel<float><<<pgrid, 256, 0, st>>>(du, (const float*)x, mean, rstd,
                                                           part_g, part_b, M, H);
  } else {
    ln_bwd_dx_kernel<__nv_bfloat16><<<grid, WARPS * 32, 0, st>>>(
        du, (const __nv_bfloat16*)x, mean, rstd, (const __nv_bfloat16*)gamma,
        (const __nv_bfloat16*)dres, (__nv_bfloat16*)dx, M, H);
    ln_bwd_param_part_kernel<__nv_bfloat16><<<pgrid, 256, 0, st>>>(
        du, (const __nv_bfloat16*)x, mean, rstd, part_g, part_b, M, H);
  }
  part_reduce_kernel<<<(H + 255) / 256, 256, 0, st>>>(part_g, dgamma, part_b, dbeta, nb, H);
  g_launch_count += 3;
  return cudaGetLastError();
}

cudaError_t colsum_accum(const void* in, int64_t ld, int M, int N, DType t, float* part,
                         float* out, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  const int nb = colsum_blocks(M);
  dim3 pgrid((N + 255) / 256, nb);
  if (t == DType::F32)
    colsum_part_kernel<float><<<pgrid, 256, 0, st>>>((const float*)in, ld, M, N, part);
  else
    colsum_part_kernel<__nv_bfloat16><<<pgrid, 256, 0, st>>>((const __nv_bfloat16*)in, ld, M,
                                                             N, part);
  part_reduce_kernel<<<(N + 255) / 256, 256, 0, st>>>(part, out, nullptr, nullptr, nb, N);
  g_launch_count += 2;
  return cudaGetLastError();
}

cudaError_t add_into(const void* a, const float* b, void* out, int64_t n, DType t,
                     cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int grid = (int)std::min<int64_t>((n + 255) / 256, 152 * 16);
  if (t == DType::F32)
    add_into_kernel<float><<<grid, 256, 0, st>>>((const float*)a, b, (float*)out, n);
  else
    add_into_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)a, b,
                                                         (__nv_bfloat16*)out, n);
  OASES_COUNT_LAUNCH();
  return cudaGetLastError();
}

}  // namespace oases
