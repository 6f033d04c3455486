// Causal softmax attention, forward and backward, on CUDA cores.
//
// O_h = softmax(Q_h K_h^T / sqrt(d) + mask) V_h for every (sequence, head),
// computed flash-style: keys are streamed through shared memory in tiles and
// each query keeps a running max m, running sum l and an unnormalised output
// (online softmax), so the S x S score matrix is never stored.  The forward
// saves LSE = m + log(l) per (head, row); the backward rebuilds
// P = exp(s - LSE) from it:
//   delta_i = sum_c dO[i,c] O[i,c]
//   dQ_i = scale * sum_j P_ij (dO_i . V_j - delta_i) K_j        (query-major pass)
//   dV_j = sum_i P_ij dO_i,  dK_j = scale * sum_i dS_ij Q_i      (key-major pass)
// Each pass owns its outputs, so no atomics are needed and results are
// deterministic.  Eight threads share one query (or key) row, each holding
// d/8 of its dimensions; d <= 128 and d % 8 == 0.
#include <math.h>

#include "common.cuh"

namespace oases {
namespace {

constexpr int ROWS = 16;       // query (or key) rows per CTA
constexpr int TPR = 8;         // threads per row
constexpr int NT = ROWS * TPR; // 128 threads
constexpr int KT = 32;         // keys (or queries) per shared-memory tile
constexpr int DMAX = 128;
constexpr int DPT = DMAX / TPR;  // dims per thread, max

__device__ __forceinline__ float group_sum(float v) {
  v += __shfl_xor_sync(0xffffffffu, v, 1);
  v += __shfl_xor_sync(0xffffffffu, v, 2);
  v += __shfl_xor_sync(0xffffffffu, v, 4);
  return v;
}

struct Geo {
  int S, H, d, heads;
  int64_t ld;  // qkv row stride = 3H
};

// Forward: grid (ceil(S/ROWS), heads, batch).
template <typename T>
__global__ void __launch_bounds__(NT)
attn_fwd_kernel(const T* __restrict__ qkv, T* __restrict__ o, float* __restrict__ lse, Geo g,
                int M, bool causal, float scale) {
  __shared__ float Ks[KT][DMAX + 1];
  __shared__ float Vs[KT][DMAX + 1];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.z, h = blockIdx.y;
  const int r = threadIdx.x / TPR, t = threadIdx.x % TPR;
  const int i = blockIdx.x * ROWS + r;  // query position in the sequence
  const int dp = g.d / TPR;
  const int64_t row0 = (int64_t)b * g.S;
  float q[DPT], acc[DPT];
  const bool valid = i < g.S;
#pragma unroll
  for (int c = 0; c < DPT; ++c) {
    acc[c] = 0.f;
    q[c] = (valid && c < dp) ? ld_elem(qkv, (row0 + i) * g.ld + h * g.d + t * dp + c) * scale : 0.f;
  }
  float m = -INFINITY, l = 0.f;
  const int last_q = min(g.S, (int)(blockIdx.x + 1) * ROWS) - 1;
  const int kend = causal ? last_q + 1 : g.S;
  for (int k0 = 0; k0 < kend; k0 += KT) {
    __syncthreads();
    for (int e = threadIdx.x; e < KT * g.d; e += NT) {
      const int kk = e / g.d, c = e % g.d, j = k0 + kk;
      float kv = 0.f, vv = 0.f;
      if (j < g.S) {
        kv = ld_elem(qkv, (row0 + j) * g.ld + g.H + h * g.d + c);
        vv = ld_elem(qkv, (row0 + j) * g.ld + 2 * g.H + h * g.d + c);
      }
      Ks[kk][c] = kv;
      Vs[kk][c] = vv;
    }
    __syncthreads();
    const int nk = min(KT, kend - k0);
    for (int kk = 0; kk < nk; ++kk) {
      const int j = k0 + kk;
      float s = 0.f;
#pragma unroll
      for (int c = 0; c < DPT; ++c)
        if (c < dp) s = fmaf(q[c], Ks[kk][t * dp + c], s);
      s = group_sum(s);
      if (!valid || (causal && j > i)) continue;
      const float mn = fmaxf(m, s);
      const float corr = expf(m - mn), p = expf(s - mn);
      l = l * corr + p;
#pragma unroll
      for (int c = 0; c < DPT; ++c)
        if (c < dp) acc[c] = fmaf(p, Vs[kk][t * dp + c], acc[c] * corr);
      m = mn;
    }
  }
  if (!valid) return;
  const float inv = 1.f / l;
#pragma unroll
  for (int c = 0; c < DPT; ++c)
    if (c < dp) st_elem(o, (row0 + i) * g.H + h * g.d + t * dp + c, acc[c] * inv);
  if (t == 0) lse[(int64_t)h * M + row0 + i] = m + logf(l);
}

// delta[h, row] = sum_c dO[row, h*d + c] * O[row, h*d + c]; one warp per (row, head).
template <typename T>
__global__ void attn_delta_kernel(const T* __restrict__ o, const T* __restrict__ d_o,
                                  float* __restrict__ delta, int M, int H, int d, int heads) {
  pdl_wait();
  pdl_trigger();
  const int w = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32, lane = threadIdx.x % 32;
  if (w >= M * heads) return;
  const int row = w / heads, h = w % heads;
  float s = 0.f;
  for (int c = lane; c < d; c += 32) {
    const int64_t idx = (int64_t)row * H + h * d + c;
    s = fmaf(ld_elem(o, idx), ld_elem(d_o, idx), s);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane == 0) delta[(int64_t)h * M + row] = s;
}

// The same for bf16 with d = 128: sixteen threads per (row, head), each
// taking 8 elements (16-byte loads) of O and dO; the two (row, head) pairs of
// a warp are adjacent in memory.  Grid-stride over M * heads pairs.
__global__ void __launch_bounds__(256)
attn_delta_bf16_d128_kernel(const __nv_bfloat16* __restrict__ o, const __nv_bfloat16* __restrict__ d_o,
                            float* __restrict__ delta, int M, int H, int heads) {
  pdl_wait();
  pdl_trigger();
  const int64_t pairs = (int64_t)M * heads;
  const int grp = threadIdx.x >> 4, sl = threadIdx.x & 15;
  for (int64_t p = (int64_t)blockIdx.x * 16 + grp; p < pairs; p += (int64_t)gridDim.x * 16) {
    const int row = (int)(p / heads), h = (int)(p % heads);
    const int64_t idx = (int64_t)row * H + h * 128 + sl * 8;
    const uint4 x = __ldg(reinterpret_cast<const uint4*>(o + idx));
    const uint4 y = __ldg(reinterpret_cast<const uint4*>(d_o + idx));
    const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&xs[k]));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ys[k]));
      s = fmaf(a.x, b.x, s);
      s = fmaf(a.y, b.y, s);
    }
#pragma unroll
    for (int off = 8; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (sl == 0) delta[(int64_t)h * M + row] = s;
  }
}

// dQ pass: grid (ceil(S/ROWS), heads, batch).
template <typename T>
__global__ void __launch_bounds__(NT)
attn_bwd_dq_kernel(const T* __restrict__ qkv, const T* __restrict__ d_o,
                   const float* __restrict__ lse, const float* __restrict__ delta,
                   T* __restrict__ dqkv, Geo g, int M, bool causal, float scale) {
  __shared__ float Ks[KT][DMAX + 1];
  __shared__ float Vs[KT][DMAX + 1];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.z, h = blockIdx.y;
  const int r = threadIdx.x / TPR, t = threadIdx.x % TPR;
  const int i = blockIdx.x * ROWS + r;
  const int dp = g.d / TPR;
  const int64_t row0 = (int64_t)b * g.S;
  const bool valid = i < g.S;
  float q[DPT], dov[DPT], dq[DPT];
#pragma unroll
  for (int c = 0; c < DPT; ++c) {
    dq[c] = 0.f;
    const bool ok = valid && c < dp;
    q[c] = ok ? ld_elem(qkv, (row0 + i) * g.ld + h * g.d + t * dp + c) * scale : 0.f;
    dov[c] = ok ? ld_elem(d_o, (row0 + i) * g.H + h * g.d + t * dp + c) : 0.f;
  }
  const float L = valid ? lse[(int64_t)h * M + row0 + i] : 0.f;
  const float D = valid ? delta[(int64_t)h * M + row0 + i] : 0.f;
  const int last_q = min(g.S, (int)(blockIdx.x + 1) * ROWS) - 1;
  const int kend = causal ? last_q + 1 : g.S;
  for (int k0 = 0; k0 < kend; k0 += KT) {
    __syncthreads();
    for (int e = threadIdx.x; e < KT * g.d; e += NT) {
      const int kk = e / g.d, c = e % g.d, j = k0 + kk;
      float kv = 0.f, vv = 0.f;
      if (j < g.S) {
        kv = ld_elem(qkv, (row0 + j) * g.ld + g.H + h * g.d + c);
        vv = ld_elem(qkv, (row0 + j) * g.ld + 2 * g.H + h * g.d + c);
      }
      Ks[kk][c] = kv;
      Vs[kk][c] = vv;
    }
    __syncthreads();
    const int nk = min(KT, kend - k0);
    for (int kk = 0; kk < nk; ++kk) {
      const int j = k0 + kk;
      float s = 0.f, dp_ = 0.f;
#pragma unroll
      for (int c = 0; c < DPT; ++c)
        if (c < dp) {
          s = fmaf(q[c], Ks[kk][t * dp + c], s);
          dp_ = fmaf(dov[c], Vs[kk][t * dp + c], dp_);
        }
      s = group_sum(s);
      dp_ = group_sum(dp_);
      if (!valid || (causal && j > i)) continue;
      const float p = expf(s - L);
      const float ds = p * (dp_ - D);
#pragma unroll
      for (int c = 0; c < DPT; ++c)
        if (c < dp) dq[c] = fmaf(ds, Ks[kk][t * dp + c], dq[c]);
    }
  }
  if (!valid) return;
#pragma unroll
  for (int c = 0; c < DPT; ++c)
    if (c < dp) st_elem(dqkv, (row0 + i) * g.ld + h * g.d + t * dp + c, dq[c] * scale);
}

// dK / dV pass: grid (ceil(S/ROWS), heads, batch); rows are keys here.
template <typename T>
__global__ void __launch_bounds__(NT)
attn_bwd_dkv_kernel(const T* __restrict__ qkv, const T* __restrict__ d_o,
                    const float* __restrict__ lse, const float* __restrict__ delta,
                    T* __restrict__ dqkv, Geo g, int M, bool causal, float scale) {
  __shared__ float Qs[KT][DMAX + 1];
  __shared__ float dOs[KT][DMAX + 1];
  __shared__ float Ls[KT], Ds[KT];
  pdl_wait();
  pdl_trigger();
  const int b = blockIdx.z, h = blockIdx.y;
  const int r = threadIdx.x / TPR, t = threadIdx.x % TPR;
  const int j = blockIdx.x * ROWS + r;  // key position
  const int dp = g.d / TPR;
  const int64_t row0 = (int64_t)b * g.S;
  const bool valid = j < g.S;
  float k[DPT], v[DPT], dk[DPT], dv[DPT];
#pragma unroll
  for (int c = 0; c < DPT; ++c) {
    dk[c] = dv[c] = 0.f;
    const bool ok = valid && c < dp;
    k[c] = ok ? ld_elem(qkv, (row0 + j) * g.ld + g.H + h * g.d + t * dp + c) : 0.f;
    v[c] = ok ? ld_elem(qkv, (row0 + j) * g.ld + 2 * g.H + h * g.d + t * dp + c) : 0.f;
  }
  const int first_k = blockIdx.x * ROWS;
  const int qbeg = causal ? first_k - first_k % KT : 0;
  for (int q0 = qbeg; q0 < g.S; q0 += KT) {
    __syncthreads();
    for (int e = threadIdx.x; e < KT * g.d; e += NT) {
      const int qq = e / g.d, c = e % g.d, i = q0 + qq;
      float qv = 0.f, dv_ = 0.f;
      if (i < g.S) {
        qv = ld_elem(qkv, (row0 + i) * g.ld + h * g.d + c) * scale;
        dv_ = ld_elem(d_o, (row0 + i) * g.H + h * g.d + c);
      }
      Qs[qq][c] = qv;
      dOs[qq][c] = dv_;
    }
    if (threadIdx.x < KT) {
      const int i = q0 + threadIdx.x;
      Ls[threadIdx.x] = i < g.S ? lse[(int64_t)h * M + row0 + i] : 0.f;
      Ds[threadIdx.x] = i < g.S ? delta[(int64_t)h * M + row0 + i] : 0.f;
    }
    __syncthreads();
    const int nq = min(KT, g.S - q0);
    for (int qq = 0; qq < nq; ++qq) {
      const int i = q0 + qq;
      float s = 0.f, dp_ = 0.f;
#pragma unroll
      for (int c = 0; c < DPT; ++c)
        if (c < dp) {
          s = fmaf(Qs[qq][t * dp + c], k[c], s);
          dp_ = fmaf(dOs[qq][t * dp + c], v[c], dp_);
        }
      s = group_sum(s);
      dp_ = group_sum(dp_);
      if (!valid || (causal && j > i)) continue;
      const float p = expf(s - Ls[qq]);
      const float ds = p * (dp_ - Ds[qq]);
#pragma unroll
      for (int c = 0; c < DPT; ++c)
        if (c < dp) {
          dv[c] = fmaf(p, dOs[qq][t * dp + c], dv[c]);
          dk[c] = fmaf(ds, Qs[qq][t * dp + c], dk[c]);  // Qs already carries the scale
        }
    }
  }
  if (!valid) return;
#pragma unroll
  for (int c = 0; c < DPT; ++c)
    if (c < dp) {
      st_elem(dqkv, (row0 + j) * g.ld + g.H + h * g.d + t * dp + c, dk[c]);
      st_elem(dqkv, (row0 + j) * g.ld + 2 * g.H + h * g.d + t * dp + c, dv[c]);
    }
}

bool simt_ok(const AttnArgs& a) {
  return a.head_dim > 0 && a.head_dim <= DMAX && a.head_dim % TPR == 0;
}

}  // namespace

cudaError_t attention_fwd_simt(const AttnArgs& a, cudaStream_t st) {
  if (!simt_ok(a)) return cudaErrorNotSupported;
  if (a.batch == 0 || a.seq == 0) return cudaSuccess;
  Geo g{a.seq, a.hidden, a.head_dim, a.heads, 3 * (int64_t)a.hidden};
  const int M = a.batch * a.seq;
  dim3 grid((a.seq + ROWS - 1) / ROWS, a.heads, a.batch);
  const float scale = 1.f / sqrtf((float)a.head_dim);
  if (a.t == DType::F32)
    return launch_pdl(attn_fwd_kernel<float>, grid, dim3(NT), 0, st, (const float*)a.qkv,
                      (float*)a.o, a.lse, g, M, a.causal, scale);
  return launch_pdl(attn_fwd_kernel<__nv_bfloat16>, grid, dim3(NT), 0, st,
                    (const __nv_bfloat16*)a.qkv, (__nv_bfloat16*)a.o, a.lse, g, M, a.causal,
                    scale);
}

cudaError_t attention_delta(const AttnArgs& a, cudaStream_t st) {
  const int M = a.batch * a.seq;
  if (M == 0) return cudaSuccess;
  if (a.t == DType::BF16 && a.head_dim == 128 && a.hidden % 8 == 0 &&
      (((uintptr_t)a.o | (uintptr_t)a.d_o) & 15) == 0) {
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t blocks = ((int64_t)M * a.heads + 15) / 16;
    const int grid = (int)std::min<int64_t>(blocks, (int64_t)std::max(sms, 1) * 8);
    return launch_pdl(attn_delta_bf16_d128_kernel, dim3(grid), dim3(256), 0, st,
                      (const __nv_bfloat16*)a.o, (const __nv_bfloat16*)a.d_o, a.delta, M, a.hidden,
                      a.heads);
  }
  const int warps = M * a.heads;
  const int grid = (warps + 7) / 8;
  if (a.t == DType::F32)
    return launch_pdl(attn_delta_kernel<float>, dim3(grid), dim3(256), 0, st, (const float*)a.o,
                      (const float*)a.d_o, a.delta, M, a.hidden, a.head_dim, a.heads);
  return launch_pdl(attn_delta_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, st,
                    (const __nv_bfloat16*)a.o, (const __nv_bfloat16*)a.d_o, a.delta, M, a.hidden,
                    a.head_dim, a.heads);
}

cudaError_t attention_bwd_simt(const AttnArgs& a, cudaStream_t st) {
  if (!simt_ok(a)) return cudaErrorNotSupported;
  if (a.batch == 0 || a.seq == 0) return cudaSuccess;
  cudaError_t e = attention_delta(a, st);
  if (e != cudaSuccess) return e;
  Geo g{a.seq, a.hidden, a.head_dim, a.heads, 3 * (int64_t)a.hidden};
  const int M = a.batch * a.seq;
  dim3 grid((a.seq + ROWS - 1) / ROWS, a.heads, a.batch);
  const float scale = 1.f / sqrtf((float)a.head_dim);
  if (a.t == DType::F32) {
    e = launch_pdl(attn_bwd_dq_kernel<float>, grid, dim3(NT), 0, st, (const float*)a.qkv,
                   (const float*)a.d_o, (const float*)a.lse, (const float*)a.delta,
                   (float*)a.dqkv, g, M, a.causal, scale);
    if (e != cudaSuccess) return e;
    return launch_pdl(attn_bwd_dkv_kernel<float>, grid, dim3(NT), 0, st, (const float*)a.qkv,
                      (const float*)a.d_o, (const float*)a.lse, (const float*)a.delta,
                      (float*)a.dqkv, g, M, a.causal, scale);
  }
  e = launch_pdl(attn_bwd_dq_kernel<__nv_bfloat16>, grid, dim3(NT), 0, st,
                 (const __nv_bfloat16*)a.qkv, (const __nv_bfloat16*)a.d_o, (const float*)a.lse,
                 (const float*)a.delta, (__nv_bfloat16*)a.dqkv, g, M, a.causal, scale);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_bwd_dkv_kernel<__nv_bfloat16>, grid, dim3(NT), 0, st,
                    (const __nv_bfloat16*)a.qkv, (const __nv_bfloat16*)a.d_o,
                    (const float*)a.lse, (const float*)a.delta, (__nv_bfloat16*)a.dqkv, g, M,
                    a.causal, scale);
}

}  // namespace oases

namespace oases {

cudaError_t attention_fwd(const AttnArgs& a, cudaStream_t st) {
  if (attention_tc_supported(a)) return attention_fwd_tc(a, st);
  return attention_fwd_simt(a, st);
}
cudaError_t attention_bwd(const AttnArgs& a, cudaStream_t st) {
  if (attention_tc_supported(a) && !(((uintptr_t)a.d_o | (uintptr_t)a.dqkv) & 15))
    return attention_bwd_tc(a, st);
  return attention_bwd_simt(a, st);
}

}  // namespace oases
