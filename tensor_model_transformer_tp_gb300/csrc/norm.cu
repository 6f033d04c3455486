// LayerNorm forward / backward and deterministic column reductions.
//
// All of these are HBM-bound.  Row statistics are taken by one warp per row
// with 16-byte loads (bf16 rows whose width is a multiple of 256 are held in
// registers, so the row is read once).  Column sums (dgamma, dbeta, bias
// gradients) are taken in two fixed-order stages: a CTA owns a block of
// ROWS_PER_PART rows and a strip of columns, reads them coalesced (adjacent
// threads, adjacent columns) and writes one partial row; a second kernel adds
// the partial rows in order.  No atomics, so results are bit-reproducible.
#include <algorithm>

#include <functional>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace oases {

// Set by a norm kernel whose bounded wait gave up; read by oases_check_device.
__device__ int g_norm_error;

namespace {

constexpr int ROWS_PER_PART = 8;  // rows per partial row of the LayerNorm backward's column sums
constexpr int COLSUM_ROWS = 32;   // rows per partial row of a bias-gradient column sum
constexpr int WARPS = 8;
constexpr int COLS_PER_THREAD = 2;
constexpr int COL_THREADS = 256;
constexpr int COLS_PER_CTA = COL_THREADS * COLS_PER_THREAD;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void bf16x8_to_f32(const uint4& u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
// The same unpacking as opaque instructions, so that the compiler converts the
// packed row again in each pass instead of keeping every element live as fp32
// (which needs twice the registers and halves the resident warps).
__device__ __forceinline__ void bf16x8_to_f32_each_pass(const uint4& u, float* f) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t lo, hi;
    asm volatile("shl.b32 %0, %1, 16;" : "=r"(lo) : "r"(w[i]));
    asm volatile("and.b32 %0, %1, 0xffff0000;" : "=r"(hi) : "r"(w[i]));
    f[2 * i] = __uint_as_float(lo);
    f[2 * i + 1] = __uint_as_float(hi);
  }
}
__device__ __forceinline__ uint4 f32_to_bf16x8(const float* f) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  return u;
}

// ---- LayerNorm forward -------------------------------------------------------
// bf16, H = 256 * NV: lane j holds 16-byte vectors j, j+32, ... of its row.
template <int NV>
__global__ void __launch_bounds__(WARPS * 32, NV <= 8 ? 4 : (NV <= 12 ? 3 : 2))
ln_fwd_bf16_reg(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ gamma,
                const __nv_bfloat16* __restrict__ beta, __nv_bfloat16* __restrict__ u,
                float* __restrict__ mean, float* __restrict__ rstd, int M, int H, float eps) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x * WARPS + threadIdx.x / 32, lane = threadIdx.x % 32;
  if (row >= M) return;
  const uint4* xr = reinterpret_cast<const uint4*>(x + (int64_t)row * H);
  uint4 v[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) v[j] = __ldg(xr + lane + 32 * j);
  // sums in eight independent chains (one per element of a vector), then a tree
  float s8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    float f[8];
    bf16x8_to_f32_each_pass(v[j], f);
#pragma unroll
    for (int i = 0; i < 8; ++i) s8[i] += f[i];
  }
  const float s = ((s8[0] + s8[1]) + (s8[2] + s8[3])) + ((s8[4] + s8[5]) + (s8[6] + s8[7]));
  const float mu = warp_sum(s) / H;
  float q8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    float f[8];
    bf16x8_to_f32_each_pass(v[j], f);
#pragma unroll
    for (int i = 0; i < 8; ++i) q8[i] = fmaf(f[i] - mu, f[i] - mu, q8[i]);
  }
  const float q = ((q8[0] + q8[1]) + (q8[2] + q8[3])) + ((q8[4] + q8[5]) + (q8[6] + q8[7]));
  const float rs = rsqrtf(warp_sum(q) / H + eps);
  const uint4* gr = reinterpret_cast<const uint4*>(gamma);
  const uint4* br = reinterpret_cast<const uint4*>(beta);
  uint4* ur = reinterpret_cast<uint4*>(u + (int64_t)row * H);
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    float f[8], g[8], b[8];
    bf16x8_to_f32_each_pass(v[j], f);
    bf16x8_to_f32(__ldg(gr + lane + 32 * j), g);
    bf16x8_to_f32(__ldg(br + lane + 32 * j), b);
#pragma unroll
    for (int i = 0; i < 8; ++i) f[i] = (f[i] - mu) * rs * g[i] + b[i];
    ur[lane + 32 * j] = f32_to_bf16x8(f);
  }
  if (lane == 0) {
    mean[row] = mu;
    rstd[row] = rs;
  }
}

// Any type, any width: three passes over the row (the later two hit L1).
template <typename T>
__global__ void __launch_bounds__(WARPS * 32)
ln_fwd_kernel(const T* __restrict__ x, const T* __restrict__ gamma, const T* __restrict__ beta,
              T* __restrict__ u, float* __restrict__ mean, float* __restrict__ rstd, int M, int H,
              float eps) {
  pdl_wait();
  pdl_trigger();
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

// ---- LayerNorm backward --------------------------------------------------------
// Row pass: m1 = mean(du * gamma), m2 = mean(du * gamma * xhat), one warp per row.
template <typename T>
__global__ void __launch_bounds__(WARPS * 32)
ln_bwd_rowstat(const float* __restrict__ du, const T* __restrict__ x,
               const float* __restrict__ mean, const float* __restrict__ rstd,
               const T* __restrict__ gamma, float2* __restrict__ stat, int M, int H) {
  pdl_wait();
  pdl_trigger();
  const int row = blockIdx.x * WARPS + threadIdx.x / 32, lane = threadIdx.x % 32;
  if (row >= M) return;
  const float* dur = du + (int64_t)row * H;
  const T* xr = x + (int64_t)row * H;
  const float mu = mean[row], rs = rstd[row];
  float s1 = 0.f, s2 = 0.f;
  if (sizeof(T) == 2 && H % 8 == 0) {
    const float4* d4 = reinterpret_cast<const float4*>(dur);
    const uint4* x8 = reinterpret_cast<const uint4*>(xr);
    const uint4* g8 = reinterpret_cast<const uint4*>(gamma);
    for (int j = lane; j < H / 8; j += 32) {
      float xf[8], gf[8];
      bf16x8_to_f32(__ldg(x8 + j), xf);
      bf16x8_to_f32(__ldg(g8 + j), gf);
      const float4 a = __ldg(d4 + 2 * j), b = __ldg(d4 + 2 * j + 1);
      const float df[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const float gg = df[i] * gf[i];
        s1 += gg;
        s2 = fmaf(gg, (xf[i] - mu) * rs, s2);
      }
    }
  } else {
    for (int c = lane; c < H; c += 32) {
      const float gg = dur[c] * ld_elem(gamma, c);
      s1 += gg;
      s2 = fmaf(gg, (ld_elem(xr, c) - mu) * rs, s2);
    }
  }
  s1 = warp_sum(s1);
  s2 = warp_sum(s2);
  if (lane == 0) stat[row] = make_float2(s1 / H, s2 / H);
}

// Column pass over ROWS_PER_PART rows x COLS_PER_CTA columns:
//   dx = rstd * (du * gamma - m1 - xhat * m2) (+ dres), and the partial sums
//   pg = sum du * xhat, pb = sum du of this row block.
template <typename T>
__global__ void __launch_bounds__(COL_THREADS)
ln_bwd_colpass(const float* __restrict__ du, const T* __restrict__ x,
               const float* __restrict__ mean, const float* __restrict__ rstd,
               const float2* __restrict__ stat, const T* __restrict__ gamma,
               const T* __restrict__ dres, T* __restrict__ dx, float* __restrict__ pg,
               float* __restrict__ pb, int M, int H) {
  pdl_wait();
  pdl_trigger();
  const int c0 = (blockIdx.x * COL_THREADS + threadIdx.x) * COLS_PER_THREAD;
  const int m0 = blockIdx.y * ROWS_PER_PART, m1 = min(M, m0 + ROWS_PER_PART);
  if (c0 >= H) return;
  float ag[COLS_PER_THREAD] = {}, ab[COLS_PER_THREAD] = {};
  float g[COLS_PER_THREAD];
#pragma unroll
  for (int i = 0; i < COLS_PER_THREAD; ++i) g[i] = c0 + i < H ? ld_elem(gamma, c0 + i) : 0.f;
#pragma unroll 4
  for (int m = m0; m < m1; ++m) {
    const float mu = mean[m], rs = rstd[m];
    const float2 st = stat[m];
    const int64_t base = (int64_t)m * H + c0;
#pragma unroll
    for (int i = 0; i < COLS_PER_THREAD; ++i) {
      if (c0 + i >= H) continue;
      const float d = du[base + i];
      const float xh = (ld_elem(x, base + i) - mu) * rs;
      float v = rs * (d * g[i] - st.x - xh * st.y);
      if (dres) v += ld_elem(dres, base + i);
      st_elem(dx, base + i, v);
      ag[i] = fmaf(d, xh, ag[i]);
      ab[i] += d;
    }
  }
#pragma unroll
  for (int i = 0; i < COLS_PER_THREAD; ++i)
    if (c0 + i < H) {
      pg[(int64_t)blockIdx.y * H + c0 + i] = ag[i];
      pb[(int64_t)blockIdx.y * H + c0 + i] = ab[i];
    }
}

// 4 consecutive elements as fp32 (16-byte fp32 or 8-byte bf16 access).
__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }
__device__ __forceinline__ float4 ld4(const __nv_bfloat16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
__device__ __forceinline__ void st4(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
__device__ __forceinline__ void st4(__nv_bfloat16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

// LayerNorm backward for one block of ROWS_PER_PART rows (H % 4 == 0):
//   phase 1, warp w: m1 = mean(du * gamma), m2 = mean(du * gamma * xhat) of row w;
//   phase 2, threads over 4-column groups, rows in order:
//     dx = rstd * (du * gamma - m1 - xhat * m2) (+ dres), and the block's
//     partial column sums pg = sum du * xhat, pb = sum du.
template <typename T>
__global__ void __launch_bounds__(ROWS_PER_PART * 32)
ln_bwd_fused(const float* __restrict__ du, const T* __restrict__ x, const float* __restrict__ mean,
             const float* __restrict__ rstd, const T* __restrict__ gamma,
             const T* __restrict__ dres, T* __restrict__ dx, float* __restrict__ pg,
             float* __restrict__ pb, int M, int H) {
  pdl_wait();
  pdl_trigger();
  __shared__ float m1s[ROWS_PER_PART], m2s[ROWS_PER_PART];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int m0 = blockIdx.x * ROWS_PER_PART;
  {
    const int row = m0 + warp;
    float s1 = 0.f, s2 = 0.f;
    if (row < M) {
      const float mu = mean[row], rs = rstd[row];
      const float* dr = du + (int64_t)row * H;
      const T* xr = x + (int64_t)row * H;
#pragma unroll 4
      for (int c = lane * 4; c < H; c += 128) {
        const float4 d = ld4(dr + c), xv = ld4(xr + c), gv = ld4(gamma + c);
        const float g0 = d.x * gv.x, g1 = d.y * gv.y, g2 = d.z * gv.z, g3 = d.w * gv.w;
        s1 += (g0 + g1) + (g2 + g3);
        s2 = fmaf(g0, (xv.x - mu) * rs, s2);
        s2 = fmaf(g1, (xv.y - mu) * rs, s2);
        s2 = fmaf(g2, (xv.z - mu) * rs, s2);
        s2 = fmaf(g3, (xv.w - mu) * rs, s2);
      }
    }
    s1 = warp_sum(s1);
    s2 = warp_sum(s2);
    if (lane == 0) {
      m1s[warp] = s1 / H;
      m2s[warp] = s2 / H;
    }
  }
  __syncthreads();
  const int rows = min(ROWS_PER_PART, M - m0);
  for (int c = tid * 4; c < H; c += ROWS_PER_PART * 32 * 4) {
    const float4 gv = ld4(gamma + c);
    float4 ag = make_float4(0.f, 0.f, 0.f, 0.f), ab = ag;
#pragma unroll 8
    for (int r = 0; r < rows; ++r) {
      const int row = m0 + r;
      const float mu = mean[row], rs = rstd[row], a1 = m1s[r], a2 = m2s[r];
      const int64_t o = (int64_t)row * H + c;
      const float4 d = ld4(du + o), xv = ld4(x + o);
      float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
      if (dres) res = ld4(dres + o);
      const float h0 = (xv.x - mu) * rs, h1 = (xv.y - mu) * rs, h2 = (xv.z - mu) * rs,
                  h3 = (xv.w - mu) * rs;
      st4(dx + o, make_float4(fmaf(rs, d.x * gv.x - a1 - h0 * a2, res.x),
                              fmaf(rs, d.y * gv.y - a1 - h1 * a2, res.y),
                              fmaf(rs, d.z * gv.z - a1 - h2 * a2, res.z),
                              fmaf(rs, d.w * gv.w - a1 - h3 * a2, res.w)));
      ag.x = fmaf(d.x, h0, ag.x);
      ag.y = fmaf(d.y, h1, ag.y);
      ag.z = fmaf(d.z, h2, ag.z);
      ag.w = fmaf(d.w, h3, ag.w);
      ab.x += d.x;
      ab.y += d.y;
      ab.z += d.z;
      ab.w += d.w;
    }
    st4(pg + (int64_t)blockIdx.x * H + c, ag);
    st4(pb + (int64_t)blockIdx.x * H + c, ab);
  }
}

// LayerNorm backward for one block of ROWS_PER_PART rows, H % 4 == 0 and
// H <= 4096, reading every input once.  Each row is spread over the CTA's 256
// threads: thread t owns the 4-column chunks t, t + 256, ... (NCH of them).
// RB rows are loaded at a time (RB * NCH <= 4 chunks in flight per thread,
// which keeps two CTAs per SM within 128 registers a thread);
// their two row means m1 = mean(du * gamma), m2 = mean(du * gamma * xhat) are
// summed within each warp, then over the 8 warps in a fixed order through
// shared memory, so the result does not depend on timing.  Then
//   dx = rstd * (du * gamma - m1 - xhat * m2) (+ dres)
// and the block's partial column sums pg = sum du * xhat, pb = sum du, added
// over the rows in order, are written as one partial row.
constexpr int LNB_THREADS = 256;
// 4 elements of T as loaded (bf16: 8 bytes, kept packed until used)
template <typename T> struct Raw4 { using type = float4; };
template <> struct Raw4<__nv_bfloat16> { using type = uint2; };
__device__ __forceinline__ float4 raw_ld(const float* p) { return ld4(p); }
__device__ __forceinline__ uint2 raw_ld(const __nv_bfloat16* p) {
  return *reinterpret_cast<const uint2*>(p);
}
__device__ __forceinline__ float4 raw_f4(float4 v) { return v; }
__device__ __forceinline__ float4 raw_f4(uint2 u) {
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
// Four fp32 values as a T store would keep them.
template <typename T> __device__ __forceinline__ float4 round4(float4 v);
template <> __device__ __forceinline__ float4 round4<float>(float4 v) { return v; }
template <> __device__ __forceinline__ float4 round4<__nv_bfloat16>(float4 v) {
  return make_float4(__bfloat162float(__float2bfloat16(v.x)), __bfloat162float(__float2bfloat16(v.y)),
                     __bfloat162float(__float2bfloat16(v.z)), __bfloat162float(__float2bfloat16(v.w)));
}
template <typename R> __device__ __forceinline__ R raw_zero();
template <> __device__ __forceinline__ float4 raw_zero<float4>() { return make_float4(0.f, 0.f, 0.f, 0.f); }
template <> __device__ __forceinline__ uint2 raw_zero<uint2>() { return make_uint2(0u, 0u); }

template <typename T, int NCH, int RB>
__global__ void __launch_bounds__(LNB_THREADS, 2)
ln_bwd_rows(const float* __restrict__ du, const T* __restrict__ x, const float* __restrict__ mean,
            const float* __restrict__ rstd, const T* __restrict__ gamma,
            const T* __restrict__ dres, T* __restrict__ dx, float* __restrict__ pg,
            float* __restrict__ pb, int M, int H) {
  static_assert(ROWS_PER_PART % RB == 0, "whole row groups per block");
  constexpr int NW = LNB_THREADS / 32;
  pdl_wait();
  pdl_trigger();
  __shared__ float red[2][NW][2 * RB];
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int m0 = blockIdx.x * ROWS_PER_PART;
  float4 gv[NCH], ag[NCH], ab[NCH];
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int c = (tid + LNB_THREADS * j) * 4;
    gv[j] = c < H ? ld4(gamma + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    ag[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    ab[j] = ag[j];
  }
  using R = typename Raw4<T>::type;
  // the row group's inputs; the next group's loads are issued before this
  // group's block-wide reduction, so they are in flight while it waits (not
  // with four chunks per thread: the second set would not fit in registers)
  constexpr bool PF = NCH < 4;
  float4 d[RB][NCH], nd[RB][NCH];
  R xv[RB][NCH], rv[RB][NCH], nxv[RB][NCH], nrv[RB][NCH];
  float mu[RB], rs[RB], nmu[RB], nrs[RB];
  auto load_group = [&](int it, float4 (&dd)[RB][NCH], R (&xx)[RB][NCH], R (&rr)[RB][NCH],
                        float (&mm)[RB], float (&ss)[RB]) {
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      const int row = m0 + it * RB + i;
      const bool ok = row < M;
      mm[i] = ok ? mean[row] : 0.f;
      ss[i] = ok ? rstd[row] : 0.f;
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int c = (tid + LNB_THREADS * j) * 4;
        const int64_t o = (int64_t)row * H + c;
        const bool in = ok && c < H;
        dd[i][j] = in ? ld4(du + o) : make_float4(0.f, 0.f, 0.f, 0.f);
        xx[i][j] = in ? raw_ld(x + o) : raw_zero<R>();
        rr[i][j] = (in && dres) ? raw_ld(dres + o) : raw_zero<R>();
      }
    }
  };
  load_group(0, d, xv, rv, mu, rs);
#pragma unroll 1
  for (int it = 0; it < ROWS_PER_PART / RB; ++it) {
    const int par = it & 1;
    float s1[RB], s2[RB];
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const float4 dd = d[i][j], xx = raw_f4(xv[i][j]), g = gv[j];
        const float g0 = dd.x * g.x, g1 = dd.y * g.y, g2 = dd.z * g.z, g3 = dd.w * g.w;
        a += (g0 + g1) + (g2 + g3);
        b = fmaf(g0, (xx.x - mu[i]) * rs[i], b);
        b = fmaf(g1, (xx.y - mu[i]) * rs[i], b);
        b = fmaf(g2, (xx.z - mu[i]) * rs[i], b);
        b = fmaf(g3, (xx.w - mu[i]) * rs[i], b);
      }
      s1[i] = warp_sum(a);
      s2[i] = warp_sum(b);
    }
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        red[par][warp][2 * i] = s1[i];
        red[par][warp][2 * i + 1] = s2[i];
      }
    }
    if (PF && it + 1 < ROWS_PER_PART / RB) load_group(it + 1, nd, nxv, nrv, nmu, nrs);
    __syncthreads();  // (the other parity's slots are free: every thread has passed it)
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      float a = 0.f, b = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        a += red[par][w][2 * i];
        b += red[par][w][2 * i + 1];
      }
      const float a1 = a / H, a2 = b / H;
      const int row = m0 + it * RB + i;
      if (row >= M) continue;
#pragma unroll
      for (int j = 0; j < NCH; ++j) {
        const int c = (tid + LNB_THREADS * j) * 4;
        if (c >= H) continue;
        const float4 dd = d[i][j], xx = raw_f4(xv[i][j]), rr = raw_f4(rv[i][j]), g = gv[j];
        const float h0 = (xx.x - mu[i]) * rs[i], h1 = (xx.y - mu[i]) * rs[i],
                    h2 = (xx.z - mu[i]) * rs[i], h3 = (xx.w - mu[i]) * rs[i];
        st4(dx + (int64_t)row * H + c,
            make_float4(fmaf(rs[i], dd.x * g.x - a1 - h0 * a2, rr.x),
                        fmaf(rs[i], dd.y * g.y - a1 - h1 * a2, rr.y),
                        fmaf(rs[i], dd.z * g.z - a1 - h2 * a2, rr.z),
                        fmaf(rs[i], dd.w * g.w - a1 - h3 * a2, rr.w)));
        ag[j].x = fmaf(dd.x, h0, ag[j].x);
        ag[j].y = fmaf(dd.y, h1, ag[j].y);
        ag[j].z = fmaf(dd.z, h2, ag[j].z);
        ag[j].w = fmaf(dd.w, h3, ag[j].w);
        ab[j].x += dd.x;
        ab[j].y += dd.y;
        ab[j].z += dd.z;
        ab[j].w += dd.w;
      }
    }
    if constexpr (PF) {
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        mu[i] = nmu[i];
        rs[i] = nrs[i];
#pragma unroll
        for (int j = 0; j < NCH; ++j) {
          d[i][j] = nd[i][j];
          xv[i][j] = nxv[i][j];
          rv[i][j] = nrv[i][j];
        }
      }
    } else if (it + 1 < ROWS_PER_PART / RB) {
      load_group(it + 1, d, xv, rv, mu, rs);
    }
  }
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int c = (tid + LNB_THREADS * j) * 4;
    if (c < H) {
      st4(pg + (int64_t)blockIdx.x * H + c, ag[j]);
      st4(pb + (int64_t)blockIdx.x * H + c, ab[j]);
    }
  }
}

// The same computation with each row's inputs (du, x, dres) staged through a
// ring of LNS_STAGES shared-memory buffers by bulk copies (cp.async.bulk, one
// per row and tensor, completion on the stage's mbarrier), so that several
// rows per CTA are in flight without holding them in registers.  A
// persistent grid: CTA b takes the row blocks b, b + gridDim.x, ... and their
// rows in order, and writes one partial row of dgamma, dbeta sums over all of
// them: gridDim.x partial rows (at most two per SM), which one launch of
// part_reduce_kernel adds in a fixed order.
// Thread 0 refills stage s with row k + LNS_STAGES after the block barrier of
// row k + 1, which every thread passes only when done with row k.  A wait that
// gives up (about 0.25 s) sets g_norm_error and ends the CTA's loop; all
// threads of the CTA leave together.
constexpr int LNS_STAGES = 3;
constexpr uint64_t LNS_WAIT = 1ull << 29;

template <typename T, int NCH>
__global__ void __launch_bounds__(LNB_THREADS, NCH <= 3 ? 3 : 2)
ln_bwd_staged(const float* __restrict__ du, const T* __restrict__ x, const float* __restrict__ mean,
              const float* __restrict__ rstd, const T* __restrict__ gamma,
              const T* __restrict__ dres, T* __restrict__ dx, float* __restrict__ pg,
              float* __restrict__ pb, float* __restrict__ px, int M, int H) {
  extern __shared__ __align__(128) uint8_t lns_smem[];
  constexpr int NW = LNB_THREADS / 32;
  __shared__ float red[2][NW][2];
  __shared__ __align__(8) uint64_t full[LNS_STAGES];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int nb = (M + ROWS_PER_PART - 1) / ROWS_PER_PART, G = gridDim.x, b = blockIdx.x;
  const int nblk = b < nb ? (nb - 1 - b) / G + 1 : 0;
  const int last = b + (nblk - 1) * G;  // only the grid's last block can be short
  const int nrows = nblk == 0 ? 0 : (nblk - 1) * ROWS_PER_PART + min(ROWS_PER_PART, M - last * ROWS_PER_PART);
  const uint32_t dbytes = (uint32_t)H * 4u, xbytes = (uint32_t)H * (uint32_t)sizeof(T);
  const uint32_t stage = dbytes + (dres ? 2u : 1u) * xbytes;
  const uint32_t sbase = ptx::smem_u32(lns_smem);
  auto row_of = [&](int k) { return (b + (k / ROWS_PER_PART) * G) * ROWS_PER_PART + k % ROWS_PER_PART; };
  auto bar = [&](int s) { return ptx::smem_u32(&full[s]); };
  auto issue = [&](int k) {
    const int s = k % LNS_STAGES;
    const int64_t o = (int64_t)row_of(k) * H;
    const uint32_t dst = sbase + (uint32_t)s * stage;
    ptx::mbar_arrive_expect_tx(bar(s), stage);
    ptx::bulk_load(dst, du + o, dbytes, bar(s));
    ptx::bulk_load(dst + dbytes, x + o, xbytes, bar(s));
    if (dres) ptx::bulk_load(dst + dbytes + xbytes, dres + o, xbytes, bar(s));
  };
  if (tid == 0) {
    for (int s = 0; s < LNS_STAGES; ++s) ptx::mbar_init(bar(s), 1);
    ptx::fence_mbar_init();
    for (int k = 0; k < LNS_STAGES && k < nrows; ++k) issue(k);
  }
  __syncthreads();
  float4 gv[NCH], ag[NCH], ab[NCH], ax[NCH];
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int c = (tid + LNB_THREADS * j) * 4;
    gv[j] = c < H ? ld4(gamma + c) : make_float4(0.f, 0.f, 0.f, 0.f);
    ag[j] = make_float4(0.f, 0.f, 0.f, 0.f);
    ab[j] = ag[j];
    ax[j] = ag[j];
  }
  using R = typename Raw4<T>::type;
  // the row statistics are read one row ahead
  float mu_n = nrows > 0 ? mean[row_of(0)] : 0.f, rs_n = nrows > 0 ? rstd[row_of(0)] : 0.f;
  int k = 0;
  for (; k < nrows; ++k) {
    const int s = k % LNS_STAGES, par = k & 1, row = row_of(k);
    const float mu = mu_n, rs = rs_n;
    if (k + 1 < nrows) {
      mu_n = mean[row_of(k + 1)];
      rs_n = rstd[row_of(k + 1)];
    }
    const bool ok = ptx::mbar_wait(bar(s), (uint32_t)(k / LNS_STAGES) & 1u, LNS_WAIT);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) atomicExch(&g_norm_error, 1);
      break;
    }
    const uint8_t* st = lns_smem + (size_t)s * stage;
    const float* sd = reinterpret_cast<const float*>(st);
    const T* sx = reinterpret_cast<const T*>(st + dbytes);
    const T* sr = reinterpret_cast<const T*>(st + dbytes + xbytes);
    float a = 0.f, bsum = 0.f;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int c = (tid + LNB_THREADS * j) * 4;
      if (c < H) {
        const float4 dd = *reinterpret_cast<const float4*>(sd + c);
        const float4 xx = raw_f4(*reinterpret_cast<const R*>(sx + c)), g = gv[j];
        const float g0 = dd.x * g.x, g1 = dd.y * g.y, g2 = dd.z * g.z, g3 = dd.w * g.w;
        a += (g0 + g1) + (g2 + g3);
        bsum = fmaf(g0, (xx.x - mu) * rs, bsum);
        bsum = fmaf(g1, (xx.y - mu) * rs, bsum);
        bsum = fmaf(g2, (xx.z - mu) * rs, bsum);
        bsum = fmaf(g3, (xx.w - mu) * rs, bsum);
      }
    }
    a = warp_sum(a);
    bsum = warp_sum(bsum);
    if (lane == 0) {
      red[par][warp][0] = a;
      red[par][warp][1] = bsum;
    }
    __syncthreads();  // (every thread is done with row k - 1: its stage may be refilled)
    if (tid == 0 && k >= 1 && k - 1 + LNS_STAGES < nrows) {
      ptx::fence_async_smem();
      issue(k - 1 + LNS_STAGES);
    }
    float sa = 0.f, sb = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      sa += red[par][w][0];
      sb += red[par][w][1];
    }
    const float a1 = sa / H, a2 = sb / H;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int c = (tid + LNB_THREADS * j) * 4;
      if (c >= H) continue;
      const float4 dd = *reinterpret_cast<const float4*>(sd + c);
      const float4 xx = raw_f4(*reinterpret_cast<const R*>(sx + c)), g = gv[j];
      const float4 rr = dres ? raw_f4(*reinterpret_cast<const R*>(sr + c)) : make_float4(0.f, 0.f, 0.f, 0.f);
      const float h0 = (xx.x - mu) * rs, h1 = (xx.y - mu) * rs, h2 = (xx.z - mu) * rs, h3 = (xx.w - mu) * rs;
      const float4 o = make_float4(fmaf(rs, dd.x * g.x - a1 - h0 * a2, rr.x), fmaf(rs, dd.y * g.y - a1 - h1 * a2, rr.y),
                                   fmaf(rs, dd.z * g.z - a1 - h2 * a2, rr.z), fmaf(rs, dd.w * g.w - a1 - h3 * a2, rr.w));
      st4(dx + (int64_t)row * H + c, o);
      if (px) {  // the column sums of dx as stored (rounded to T)
        const float4 q = round4<T>(o);
        ax[j].x += q.x;
        ax[j].y += q.y;
        ax[j].z += q.z;
        ax[j].w += q.w;
      }
      ag[j].x = fmaf(dd.x, h0, ag[j].x);
      ag[j].y = fmaf(dd.y, h1, ag[j].y);
      ag[j].z = fmaf(dd.z, h2, ag[j].z);
      ag[j].w = fmaf(dd.w, h3, ag[j].w);
      ab[j].x += dd.x;
      ab[j].y += dd.y;
      ab[j].z += dd.z;
      ab[j].w += dd.w;
    }
  }
  // the CTA's partial column sums over all of its rows, one partial row per CTA
#pragma unroll
  for (int j = 0; j < NCH; ++j) {
    const int c = (tid + LNB_THREADS * j) * 4;
    if (c < H) {
      st4(pg + (int64_t)b * H + c, ag[j]);
      st4(pb + (int64_t)b * H + c, ab[j]);
      if (px) st4(px + (int64_t)b * H + c, ax[j]);
    }
  }
  // every copy issued has landed before the CTA may exit (the waits above
  // consumed rows 0 .. k - 1; the issued ones are rows up to min(nrows, ...))
  if (tid == 0) {
    const int issued = min(nrows, k >= 1 ? k - 1 + LNS_STAGES : LNS_STAGES);
    bool dr = true;
    for (int q = k; q < issued; ++q)
      dr = ptx::mbar_wait(bar(q % LNS_STAGES), (uint32_t)(q / LNS_STAGES) & 1u, LNS_WAIT) && dr;
    if (!dr) atomicExch(&g_norm_error, 2);
  }
}

template <typename T, int NCH>
cudaError_t ln_bwd_staged_launch_n(const float* du, const T* x, const float* mean, const float* rstd,
                                   const T* gamma, const T* dres, T* dx, float* pg, float* pb,
                                   float*& px, int px_cap, int M, int H, cudaStream_t st, int* parts) {
  static DeviceOnce attr;
  const cudaError_t ea = attr.run([] {
    return cudaFuncSetAttribute(ln_bwd_staged<T, NCH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                LNS_STAGES * 4096 * (4 + 2 * (int)sizeof(T)));
  });
  if (ea != cudaSuccess) return ea;
  const int smem = LNS_STAGES * H * (4 + (dres ? 2 : 1) * (int)sizeof(T));
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ln_bwd_staged<T, NCH>, LNB_THREADS, smem);
  if (e != cudaSuccess) return e;
  const int nb = (M + ROWS_PER_PART - 1) / ROWS_PER_PART;
  const int grid = std::max(1, std::min(nb, sms * std::max(per_sm, 1)));
  *parts = grid;
  if (grid > px_cap) px = nullptr;  // no room for the dx partial rows: not taken
  return launch_pdl(ln_bwd_staged<T, NCH>, dim3(grid), dim3(LNB_THREADS), smem, st, du, x, mean, rstd,
                    gamma, dres, dx, pg, pb, px, M, H);
}

// Rows staged through shared memory by bulk copies: every row's start and
// length 16-byte aligned.
template <typename T>
bool ln_bwd_staged_ok(const float* du, const void* x, const void* dres, int H) {
  return H % (16 / (int)sizeof(T)) == 0 && H <= 4096 &&
         (((uintptr_t)du | (uintptr_t)x | (uintptr_t)dres) & 15) == 0;
}

// Launches ln_bwd_staged; *parts = the partial rows it writes.
template <typename T>
cudaError_t ln_bwd_staged_launch(const float* du, const void* x, const float* mean, const float* rstd,
                                 const void* gamma, const void* dres, void* dx, float* pg, float* pb,
                                 float*& px, int px_cap, int M, int H, cudaStream_t st, int* parts) {
  const T *xt = (const T*)x, *gt = (const T*)gamma, *rt = (const T*)dres;
  T* dt = (T*)dx;
  switch ((H / 4 + LNB_THREADS - 1) / LNB_THREADS) {
    case 1: return ln_bwd_staged_launch_n<T, 1>(du, xt, mean, rstd, gt, rt, dt, pg, pb, px, px_cap, M, H, st, parts);
    case 2: return ln_bwd_staged_launch_n<T, 2>(du, xt, mean, rstd, gt, rt, dt, pg, pb, px, px_cap, M, H, st, parts);
    case 3: return ln_bwd_staged_launch_n<T, 3>(du, xt, mean, rstd, gt, rt, dt, pg, pb, px, px_cap, M, H, st, parts);
    default: return ln_bwd_staged_launch_n<T, 4>(du, xt, mean, rstd, gt, rt, dt, pg, pb, px, px_cap, M, H, st, parts);
  }
}

template <typename T>
cudaError_t ln_bwd_rows_launch(const float* du, const void* x, const float* mean, const float* rstd,
                               const void* gamma, const void* dres, void* dx, float* pg,
                               float* pb, int M, int H, cudaStream_t st) {
  const int nb = (M + ROWS_PER_PART - 1) / ROWS_PER_PART;
  const int nch = (H / 4 + LNB_THREADS - 1) / LNB_THREADS;  // 1 .. 4
  const T *xt = (const T*)x, *gt = (const T*)gamma, *rt = (const T*)dres;
  T* dt = (T*)dx;
  switch (nch) {
    case 1:
      return launch_pdl(ln_bwd_rows<T, 1, 4>, dim3(nb), dim3(LNB_THREADS), 0, st, du, xt, mean,
                        rstd, gt, rt, dt, pg, pb, M, H);
    case 2:
      return launch_pdl(ln_bwd_rows<T, 2, 2>, dim3(nb), dim3(LNB_THREADS), 0, st, du, xt, mean,
                        rstd, gt, rt, dt, pg, pb, M, H);
    case 3:
      return launch_pdl(ln_bwd_rows<T, 3, 1>, dim3(nb), dim3(LNB_THREADS), 0, st, du, xt, mean,
                        rstd, gt, rt, dt, pg, pb, M, H);
    default:
      return launch_pdl(ln_bwd_rows<T, 4, 1>, dim3(nb), dim3(LNB_THREADS), 0, st, du, xt, mean,
                        rstd, gt, rt, dt, pg, pb, M, H);
  }
}

// Column sums of a block of COLSUM_ROWS rows: each thread takes the 16 bytes
// of 16 / sizeof(T) columns (N a multiple of that) and adds the block's rows in
// order; partial row p covers rows COLSUM_ROWS p .. + COLSUM_ROWS - 1.
template <typename T>
__global__ void __launch_bounds__(COL_THREADS)
colsum_vec_kernel(const T* __restrict__ in, int64_t ld, int M, int N, float* __restrict__ part) {
  pdl_wait();
  pdl_trigger();
  constexpr int V = 16 / sizeof(T);
  const int c = (blockIdx.x * COL_THREADS + threadIdx.x) * V;
  if (c >= N) return;
  // CTA row y takes the partial rows y, y + gridDim.y, ...
  const int nb = (M + COLSUM_ROWS - 1) / COLSUM_ROWS;
  for (int p = blockIdx.y; p < nb; p += gridDim.y) {
    const int m0 = p * COLSUM_ROWS, m1 = min(M, m0 + COLSUM_ROWS);
    float a[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
    for (int m = m0; m < m1; ++m) {
      const uint4 w = __ldg(reinterpret_cast<const uint4*>(in + (int64_t)m * ld + c));
      if constexpr (sizeof(T) == 2) {
        float f[8];
        bf16x8_to_f32(w, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) a[i] += f[i];
      } else {
        a[0] += __uint_as_float(w.x);
        a[1] += __uint_as_float(w.y);
        a[2] += __uint_as_float(w.z);
        a[3] += __uint_as_float(w.w);
      }
    }
    float* o = part + (int64_t)p * N + c;
    st4(o, make_float4(a[0], a[1], a[2], a[3]));
    if constexpr (V == 8) st4(o + 4, make_float4(a[4], a[5], a[6], a[7]));
  }
}

template <typename T>
__global__ void __launch_bounds__(COL_THREADS)
colsum_part_kernel(const T* __restrict__ in, int64_t ld, int M, int N, float* __restrict__ part) {
  pdl_wait();
  pdl_trigger();
  const int c0 = (blockIdx.x * COL_THREADS + threadIdx.x) * COLS_PER_THREAD;
  if (c0 >= N) return;
  const int nb = (M + COLSUM_ROWS - 1) / COLSUM_ROWS;
  for (int p = blockIdx.y; p < nb; p += gridDim.y) {
    const int m0 = p * COLSUM_ROWS, m1 = min(M, m0 + COLSUM_ROWS);
    float s[COLS_PER_THREAD] = {};
#pragma unroll 8
    for (int m = m0; m < m1; ++m) {
#pragma unroll
      for (int i = 0; i < COLS_PER_THREAD; ++i)
        if (c0 + i < N) s[i] += ld_elem(in, (int64_t)m * ld + c0 + i);
    }
#pragma unroll
    for (int i = 0; i < COLS_PER_THREAD; ++i)
      if (c0 + i < N) part[(int64_t)p * N + c0 + i] = s[i];
  }
}

// out[n] += sum_b part[b, n] over b = 0 .. nb-1 in a fixed order: thread group g
// (of 8) sums b = g, g+8, ... and the eight group sums are added in order 0..7.
// A second (part2, out2) pair is reduced by the same launch when given.
constexpr int RED_COLS = 32, RED_GROUPS = 8;
__global__ void __launch_bounds__(RED_COLS * RED_GROUPS)
part_reduce_kernel(const float* __restrict__ part, float* __restrict__ out,
                   const float* __restrict__ part2, float* __restrict__ out2, int nb, int N) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sh[2][RED_GROUPS][RED_COLS];
  const int cl = threadIdx.x % RED_COLS, g = threadIdx.x / RED_COLS;
  const int n = blockIdx.x * RED_COLS + cl;
  float s = 0.f, s2 = 0.f;
  if (n < N) {
    // eight rows' loads in flight before they are added, in the same order
    constexpr int U = 8;
    int b = g;
    for (; b + (U - 1) * RED_GROUPS < nb; b += U * RED_GROUPS) {
      float v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = part[(int64_t)(b + u * RED_GROUPS) * N + n];
#pragma unroll
      for (int u = 0; u < U; ++u) s += v[u];
      if (part2) {
#pragma unroll
        for (int u = 0; u < U; ++u) v[u] = part2[(int64_t)(b + u * RED_GROUPS) * N + n];
#pragma unroll
        for (int u = 0; u < U; ++u) s2 += v[u];
      }
    }
    for (; b < nb; b += RED_GROUPS) {
      s += part[(int64_t)b * N + n];
      if (part2) s2 += part2[(int64_t)b * N + n];
    }
  }
  sh[0][g][cl] = s;
  sh[1][g][cl] = s2;
  __syncthreads();
  if (g == 0 && n < N) {
    float t = 0.f, t2 = 0.f;
#pragma unroll
    for (int k = 0; k < RED_GROUPS; ++k) {
      t += sh[0][k][cl];
      t2 += sh[1][k][cl];
    }
    out[n] += t;
    if (part2) out2[n] += t2;
  }
}

// Two-level fixed-order column sum of nb partial rows [nb, N] (and optionally
// a second array).  Level 1: CTA (x, g) sums rows 16g .. 16g+15 of each column
// (four independent accumulators, combined in a fixed order) and writes the
// result over row 16g — every row of the group is read before that write by
// the same thread, so the update is in place.  Level 2 adds rows 0, 16, 32, ...
// into out in a fixed order (part_reduce_l2).
constexpr int RED_ROWS = 16;
__global__ void __launch_bounds__(256)
part_reduce_l1(float* __restrict__ part, float* __restrict__ part2, int nb, int N) {
  pdl_wait();
  pdl_trigger();
  const int n = blockIdx.x * 256 + threadIdx.x;
  if (n >= N) return;
  const int ngroups = (nb + RED_ROWS - 1) / RED_ROWS;
  for (int grp = blockIdx.y; grp < ngroups; grp += gridDim.y) {
    const int r0 = grp * RED_ROWS, r1 = min(nb, r0 + RED_ROWS);
    for (int a = 0; a < (part2 ? 2 : 1); ++a) {
      float* p = a == 0 ? part : part2;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
      int r = r0;
      for (; r + 4 <= r1; r += 4) {
        s0 += p[(int64_t)r * N + n];
        s1 += p[(int64_t)(r + 1) * N + n];
        s2 += p[(int64_t)(r + 2) * N + n];
        s3 += p[(int64_t)(r + 3) * N + n];
      }
      for (; r < r1; ++r) s0 += p[(int64_t)r * N + n];
      p[(int64_t)r0 * N + n] = (s0 + s1) + (s2 + s3);
    }
  }
}
// Level 2: out[n] += the level-1 rows 0, 16, 32, ... of column n.  A CTA
// takes 32 columns with 8 thread groups; group g adds the rows 16 (g + 8 i)
// in order of i, then group sums are added in order 0..7: a fixed order, so
// the result does not depend on timing.
__global__ void __launch_bounds__(RED_COLS * RED_GROUPS)
part_reduce_l2(const float* __restrict__ part, float* __restrict__ out,
               const float* __restrict__ part2, float* __restrict__ out2, int nb, int N) {
  pdl_wait();
  pdl_trigger();
  __shared__ float sh[2][RED_GROUPS][RED_COLS];
  const int cl = threadIdx.x % RED_COLS, g = threadIdx.x / RED_COLS;
  const int n = blockIdx.x * RED_COLS + cl;
  float s = 0.f, s2 = 0.f;
  if (n < N) {
    for (int r = g * RED_ROWS; r < nb; r += RED_GROUPS * RED_ROWS) {
      s += part[(int64_t)r * N + n];
      if (part2) s2 += part2[(int64_t)r * N + n];
    }
  }
  sh[0][g][cl] = s;
  sh[1][g][cl] = s2;
  __syncthreads();
  if (g == 0 && n < N) {
    float t = 0.f, t2 = 0.f;
#pragma unroll
    for (int k = 0; k < RED_GROUPS; ++k) {
      t += sh[0][k][cl];
      t2 += sh[1][k][cl];
    }
    out[n] += t;
    if (part2) out2[n] += t2;
  }
}

// The same with 16-byte loads, for N % 4 == 0 and 16-byte aligned rows: a CTA
// takes 16 columns (four float4 quads) with 64 row groups; group g adds rows
// g, g + 64, ... in order (four loads in flight), then each column's 64 group
// sums are added in a fixed two-stage order (groups 4k .. 4k + 3, then k =
// 0 .. 15), so the result does not depend on timing.  Twice the CTAs of the
// scalar kernel and four times the bytes per load keep enough reads in flight
// for a few MB of partial rows.
constexpr int RV_COLS = 16, RV_GROUPS = 64;
__global__ void __launch_bounds__(256)
part_reduce_v4_kernel(const float* __restrict__ part, float* __restrict__ out,
                      const float* __restrict__ part2, float* __restrict__ out2,
                      const float* __restrict__ part3, float* __restrict__ out3, int nb, int N) {
  pdl_wait();
  pdl_trigger();
  __shared__ float4 sh[3][RV_GROUPS][RV_COLS / 4];
  __shared__ float sh2[3][16][RV_COLS];
  const int q = threadIdx.x & 3, g = threadIdx.x >> 2;
  const int n = blockIdx.x * RV_COLS + q * 4;
  float4 s = make_float4(0.f, 0.f, 0.f, 0.f), s2 = s, s3 = s;
  auto add4 = [](float4& a, const float4 b) {
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
  };
  if (n < N) {
    constexpr int U = 4;
    int b = g;
    for (; b + (U - 1) * RV_GROUPS < nb; b += U * RV_GROUPS) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = *reinterpret_cast<const float4*>(part + (int64_t)(b + u * RV_GROUPS) * N + n);
#pragma unroll
      for (int u = 0; u < U; ++u) add4(s, v[u]);
      if (part2) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          v[u] = *reinterpret_cast<const float4*>(part2 + (int64_t)(b + u * RV_GROUPS) * N + n);
#pragma unroll
        for (int u = 0; u < U; ++u) add4(s2, v[u]);
      }
      if (part3) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          v[u] = *reinterpret_cast<const float4*>(part3 + (int64_t)(b + u * RV_GROUPS) * N + n);
#pragma unroll
        for (int u = 0; u < U; ++u) add4(s3, v[u]);
      }
    }
    for (; b < nb; b += RV_GROUPS) {
      add4(s, *reinterpret_cast<const float4*>(part + (int64_t)b * N + n));
      if (part2) add4(s2, *reinterpret_cast<const float4*>(part2 + (int64_t)b * N + n));
      if (part3) add4(s3, *reinterpret_cast<const float4*>(part3 + (int64_t)b * N + n));
    }
  }
  sh[0][g][q] = s;
  sh[1][g][q] = s2;
  sh[2][g][q] = s3;
  __syncthreads();
  {  // stage 1: thread (k, c) adds groups 4k .. 4k + 3 of column c
    const int c = threadIdx.x & (RV_COLS - 1), k = threadIdx.x >> 4;
#pragma unroll
    for (int a = 0; a < 3; ++a) {
      float t = 0.f;
#pragma unroll
      for (int u = 0; u < 4; ++u) t += reinterpret_cast<const float*>(&sh[a][4 * k + u][c >> 2])[c & 3];
      sh2[a][k][c] = t;
    }
  }
  __syncthreads();
  if (threadIdx.x < RV_COLS) {  // stage 2: k = 0 .. 15 in order
    const int c = threadIdx.x, col = blockIdx.x * RV_COLS + c;
    float t = 0.f, t2 = 0.f, t3 = 0.f;
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      t += sh2[0][k][c];
      t2 += sh2[1][k][c];
      t3 += sh2[2][k][c];
    }
    if (col < N) {
      out[col] += t;
      if (part2) out2[col] += t2;
      if (part3) out3[col] += t3;
    }
  }
}

cudaError_t reduce_parts(float* part, float* out, float* part2, float* out2, int nb, int N,
                         cudaStream_t st) {
  if (nb <= 64 * RED_GROUPS && N % 4 == 0 &&
      (((uintptr_t)part | (uintptr_t)(part2 ? part2 : part)) & 15) == 0)
    return launch_pdl(part_reduce_v4_kernel, dim3((N + RV_COLS - 1) / RV_COLS), dim3(256), 0, st,
                      (const float*)part, out, (const float*)part2, out2, (const float*)nullptr,
                      (float*)nullptr, nb, N);
  // up to 512 partial rows (the bias gradients of 8192 rows, the LayerNorm
  // backward's per-CTA rows): one launch, each of the eight thread groups
  // adding at most 64 rows
  if (nb <= 64 * RED_GROUPS)
    return launch_pdl(part_reduce_kernel, dim3((N + RED_COLS - 1) / RED_COLS),
                      dim3(RED_COLS * RED_GROUPS), 0, st, (const float*)part, out,
                      (const float*)part2, out2, nb, N);
  const int gx = (N + 255) / 256;
  const int gy = std::min((nb + RED_ROWS - 1) / RED_ROWS, 65535);
  cudaError_t e = launch_pdl(part_reduce_l1, dim3(gx, gy), dim3(256),
                             0, st, part, part2, nb, N);
  if (e != cudaSuccess) return e;
  return launch_pdl(part_reduce_l2, dim3((N + RED_COLS - 1) / RED_COLS), dim3(RED_COLS * RED_GROUPS),
                    0, st, (const float*)part, out, (const float*)part2, out2, nb, N);
}

template <typename T>
__global__ void add_into_kernel(const T* __restrict__ a, const float* __restrict__ b,
                                T* __restrict__ out, int64_t n) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    float v = b[i];
    if (a) v += ld_elem(a, i);
    st_elem(out, i, v);
  }
}

template <int NV>
cudaError_t ln_fwd_reg_launch(const void* x, const void* gamma, const void* beta, void* u,
                              float* mean, float* rstd, int M, int H, float eps, cudaStream_t st) {
  return launch_pdl(ln_fwd_bf16_reg<NV>, dim3((M + WARPS - 1) / WARPS), dim3(WARPS * 32), 0, st,
                    (const __nv_bfloat16*)x, (const __nv_bfloat16*)gamma,
                    (const __nv_bfloat16*)beta, (__nv_bfloat16*)u, mean, rstd, M, H, eps);
}

template <typename T>
cudaError_t ln_bwd_t(const float* du, const void* x, const float* mean, const float* rstd,
                     const void* gamma, const void* dres, void* dx, float* part_g, float* part_b,
                     float2* stat, float* dgamma, float* dbeta, int M, int H, cudaStream_t st) {
  const int nb = (M + ROWS_PER_PART - 1) / ROWS_PER_PART;
  cudaError_t e = launch_pdl(ln_bwd_rowstat<T>, dim3((M + WARPS - 1) / WARPS), dim3(WARPS * 32),
                             0, st, du, (const T*)x, mean, rstd, (const T*)gamma, stat, M, H);
  if (e != cudaSuccess) return e;
  e = launch_pdl(ln_bwd_colpass<T>, dim3((H + COLS_PER_CTA - 1) / COLS_PER_CTA, nb),
                 dim3(COL_THREADS), 0, st, du, (const T*)x, mean, rstd, (const float2*)stat,
                 (const T*)gamma, (const T*)dres, (T*)dx, part_g, part_b, M, H);
  if (e != cudaSuccess) return e;
  return launch_pdl(part_reduce_kernel, dim3((H + RED_COLS - 1) / RED_COLS),
                    dim3(RED_COLS * RED_GROUPS), 0, st, (const float*)part_g, dgamma,
                    (const float*)part_b, dbeta, nb, H);
}

// out[m, n] = sum_{k < w} part[k][m, n] (+ bias[n]) (+ resid[m, n]): the shard
// sum of the separate-reduction mode, k in order 0, 1, ...; part fp32 with
// pstride floats between shards and row pitch N; VEC = 4 or 1 columns per thread.
template <typename TO, typename TI, int VEC>
__global__ void __launch_bounds__(256)
shard_sum_kernel(const float* __restrict__ part, int64_t pstride, int w,
                 const TI* __restrict__ bias, const TI* __restrict__ resid, TO* __restrict__ out,
                 int64_t n_vec, int N) {
  pdl_wait();
  pdl_trigger();
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n_vec;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t e = i * VEC;
    const int c = (int)(e % N);
    if (VEC == 4) {
      float4 a = ld4(part + e);
      for (int k = 1; k < w; ++k) {
        const float4 b = ld4(part + k * pstride + e);
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      if (bias) {
        const float4 b = ld4(bias + c);
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      if (resid) {
        const float4 b = ld4(resid + e);
        a.x += b.x;
        a.y += b.y;
        a.z += b.z;
        a.w += b.w;
      }
      st4(out + e, a);
    } else {
      float a = part[e];
      for (int k = 1; k < w; ++k) a += part[k * pstride + e];
      if (bias) a += ld_elem(bias, c);
      if (resid) a += ld_elem(resid, e);
      st_elem(out, e, a);
    }
  }
}

template <typename TO, typename TI>
cudaError_t shard_sum_t(const float* part, int64_t pstride, int w, const void* bias,
                        const void* resid, void* out, int M, int N, cudaStream_t st) {
  const int64_t n = (int64_t)M * N;
  const bool vec = N % 4 == 0 && pstride % 4 == 0 &&
                   (((uintptr_t)part | (uintptr_t)out | (uintptr_t)bias | (uintptr_t)resid) % 16) == 0;
  if (vec) {
    const int64_t nv = n / 4;
    const int grid = (int)std::min<int64_t>((nv + 255) / 256, 152 * 8);
    return launch_pdl(shard_sum_kernel<TO, TI, 4>, dim3(grid), dim3(256), 0, st, part, pstride, w,
                      (const TI*)bias, (const TI*)resid, (TO*)out, nv, N);
  }
  const int grid = (int)std::min<int64_t>((n + 255) / 256, 152 * 8);
  return launch_pdl(shard_sum_kernel<TO, TI, 1>, dim3(grid), dim3(256), 0, st, part, pstride, w,
                    (const TI*)bias, (const TI*)resid, (TO*)out, n, N);
}

}  // namespace

cudaError_t shard_sum(const float* part, int64_t pstride, int w, const void* bias,
                      const void* resid, void* out, DType out_t, DType in_t, int M, int N,
                      cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  if (out_t == DType::F32)
    return in_t == DType::F32 ? shard_sum_t<float, float>(part, pstride, w, bias, resid, out, M, N, st)
                              : shard_sum_t<float, __nv_bfloat16>(part, pstride, w, bias, resid, out, M, N, st);
  return in_t == DType::F32 ? shard_sum_t<__nv_bfloat16, float>(part, pstride, w, bias, resid, out, M, N, st)
                            : shard_sum_t<__nv_bfloat16, __nv_bfloat16>(part, pstride, w, bias, resid, out, M, N, st);
}

// Three pairs of partial rows (the same count nb) reduced into their outputs:
// one launch where the 16-byte kernel applies, else one pair at a time.
cudaError_t reduce_parts3(float* p1, float* o1, float* p2, float* o2, float* p3, float* o3, int nb,
                          int N, cudaStream_t st) {
  if (nb <= 64 * RED_GROUPS && N % 4 == 0 && (((uintptr_t)p1 | (uintptr_t)p2 | (uintptr_t)p3) & 15) == 0)
    return launch_pdl(part_reduce_v4_kernel, dim3((N + RV_COLS - 1) / RV_COLS), dim3(256), 0, st,
                      (const float*)p1, o1, (const float*)p2, o2, (const float*)p3, o3, nb, N);
  cudaError_t e = reduce_parts(p1, o1, p2, o2, nb, N, st);
  if (e != cudaSuccess) return e;
  return reduce_parts(p3, o3, nullptr, nullptr, nb, N, st);
}

// out[n] += the sum of the nparts partial rows part[r][n], in a fixed order.
cudaError_t reduce_partial_rows(float* part, float* out, int nparts, int N, cudaStream_t st) {
  if (nparts <= 0 || N <= 0) return cudaSuccess;
  return reduce_parts(part, out, nullptr, nullptr, nparts, N, st);
}

int norm_read_and_clear_error() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_norm_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_norm_error, &z, sizeof(int));
  return v;
}

int ln_bwd_blocks(int M) { return (M + ROWS_PER_PART - 1) / ROWS_PER_PART; }
int colsum_blocks(int M) { return (M + COLSUM_ROWS - 1) / COLSUM_ROWS; }

cudaError_t layer_norm_fwd(const void* x, const void* gamma, const void* beta, void* u,
                           float* mean, float* rstd, int M, int H, float eps, DType t,
                           cudaStream_t st) {
  if (M == 0) return cudaSuccess;
  const dim3 grid((M + WARPS - 1) / WARPS), block(WARPS * 32);
  if (t == DType::BF16 && H % 256 == 0 && H / 256 <= 16) {
    switch (H / 256) {
#define OASES_LN_CASE(n) \
  case n: return ln_fwd_reg_launch<n>(x, gamma, beta, u, mean, rstd, M, H, eps, st);
      OASES_LN_CASE(1) OASES_LN_CASE(2) OASES_LN_CASE(3) OASES_LN_CASE(4) OASES_LN_CASE(5)
      OASES_LN_CASE(6) OASES_LN_CASE(7) OASES_LN_CASE(8) OASES_LN_CASE(9) OASES_LN_CASE(10)
      OASES_LN_CASE(11) OASES_LN_CASE(12) OASES_LN_CASE(13) OASES_LN_CASE(14) OASES_LN_CASE(15)
      OASES_LN_CASE(16)
#undef OASES_LN_CASE
    }
  }
  if (t == DType::F32)
    return launch_pdl(ln_fwd_kernel<float>, grid, block, 0, st, (const float*)x,
                      (const float*)gamma, (const float*)beta, (float*)u, mean, rstd, M, H, eps);
  return launch_pdl(ln_fwd_kernel<__nv_bfloat16>, grid, block, 0, st, (const __nv_bfloat16*)x,
                    (const __nv_bfloat16*)gamma, (const __nv_bfloat16*)beta, (__nv_bfloat16*)u,
                    mean, rstd, M, H, eps);
}

cudaError_t layer_norm_bwd_dx_colsum(const float* du, const void* x, const float* mean,
                                     const float* rstd, const void* gamma, const void* dres, void* dx,
                                     float* part_g, float* part_b, float2* stat, float* dgamma,
                                     float* dbeta, int M, int H, DType t, cudaStream_t st,
                                     float* part_x, int part_x_cap, int* n_part_x, float* out_x,
                                     const std::function<void(bool)>* before_reduce);

cudaError_t layer_norm_bwd(const float* du, const void* x, const float* mean, const float* rstd,
                           const void* gamma, const void* dres, void* dx, float* part_g,
                           float* part_b, float2* stat, float* dgamma, float* dbeta, int M, int H,
                           DType t, cudaStream_t st) {
  return layer_norm_bwd_dx_colsum(du, x, mean, rstd, gamma, dres, dx, part_g, part_b, stat, dgamma,
                                  dbeta, M, H, t, st, nullptr, 0, nullptr, nullptr, nullptr);
}

// The same, and where the staged kernel runs and at most part_x_cap partial
// rows are needed, also the column sums of dx as stored: *n_part_x partial
// rows of H floats in part_x (16-byte aligned), for a fixed-order reduction by
// the caller, or, with out_x given, added into out_x by the same reduction
// launch as dgamma and dbeta (*n_part_x = -1).  Otherwise *n_part_x = 0 and
// part_x is not written.  before_reduce (optional) runs on the host right
// before the dgamma / dbeta reduction is enqueued, with true when out_x is
// reduced by it too: the caller's stream waits for accumulation order go there.
cudaError_t layer_norm_bwd_dx_colsum(const float* du, const void* x, const float* mean,
                                     const float* rstd, const void* gamma, const void* dres, void* dx,
                                     float* part_g, float* part_b, float2* stat, float* dgamma,
                                     float* dbeta, int M, int H, DType t, cudaStream_t st,
                                     float* part_x, int part_x_cap, int* n_part_x, float* out_x,
                                     const std::function<void(bool)>* before_reduce) {
  auto hook = [&](bool with_x) {
    if (before_reduce) (*before_reduce)(with_x);
  };
  if (n_part_x) *n_part_x = 0;
  if ((uintptr_t)part_x & 15) part_x = nullptr;
  if (M == 0) return cudaSuccess;
  // du is fp32 (16-byte vector loads); x, gamma, dres, dx 8-byte (bf16) or
  // 16-byte (fp32) vectors of 4 elements
  const bool vec = H % 4 == 0 && ((uintptr_t)du & 15) == 0 &&
                   (((uintptr_t)x | (uintptr_t)gamma | (uintptr_t)dres | (uintptr_t)dx) &
                    (t == DType::BF16 ? 7 : 15)) == 0 &&
                   ((uintptr_t)part_g & 15) == 0 && ((uintptr_t)part_b & 15) == 0;
  if (H <= 4 * LNB_THREADS * 4 && ((uintptr_t)part_g & 15) == 0 && ((uintptr_t)part_b & 15) == 0 &&
      (t == DType::F32 ? ln_bwd_staged_ok<float>(du, x, dres, H)
                       : ln_bwd_staged_ok<__nv_bfloat16>(du, x, dres, H))) {
    int parts = 0;
    float* px = part_x;
    cudaError_t e = t == DType::F32
                        ? ln_bwd_staged_launch<float>(du, x, mean, rstd, gamma, dres, dx, part_g,
                                                      part_b, px, part_x_cap, M, H, st, &parts)
                        : ln_bwd_staged_launch<__nv_bfloat16>(du, x, mean, rstd, gamma, dres, dx,
                                                              part_g, part_b, px, part_x_cap, M, H, st,
                                                              &parts);
    if (e != cudaSuccess) return e;
    if (px && out_x) {
      hook(true);
      if (n_part_x) *n_part_x = -1;
      return reduce_parts3(part_g, dgamma, part_b, dbeta, px, out_x, parts, H, st);
    }
    if (n_part_x) *n_part_x = px ? parts : 0;
    hook(false);
    return reduce_parts(part_g, dgamma, part_b, dbeta, parts, H, st);
  }
  if (vec && H <= 4 * LNB_THREADS * 4) {
    const int nb = ln_bwd_blocks(M);
    cudaError_t e = t == DType::F32
                        ? ln_bwd_rows_launch<float>(du, x, mean, rstd, gamma, dres, dx, part_g,
                                                    part_b, M, H, st)
                        : ln_bwd_rows_launch<__nv_bfloat16>(du, x, mean, rstd, gamma, dres, dx,
                                                            part_g, part_b, M, H, st);
    if (e != cudaSuccess) return e;
    hook(false);
    return reduce_parts(part_g, dgamma, part_b, dbeta, nb, H, st);
  }
  if (vec) {
    const int nb = ln_bwd_blocks(M);
    cudaError_t e;
    if (t == DType::F32)
      e = launch_pdl(ln_bwd_fused<float>, dim3(nb), dim3(ROWS_PER_PART * 32), 0, st, du,
                     (const float*)x, mean, rstd, (const float*)gamma, (const float*)dres,
                     (float*)dx, part_g, part_b, M, H);
    else
      e = launch_pdl(ln_bwd_fused<__nv_bfloat16>, dim3(nb), dim3(ROWS_PER_PART * 32), 0, st, du,
                     (const __nv_bfloat16*)x, mean, rstd, (const __nv_bfloat16*)gamma,
                     (const __nv_bfloat16*)dres, (__nv_bfloat16*)dx, part_g, part_b, M, H);
    if (e != cudaSuccess) return e;
    hook(false);
    return reduce_parts(part_g, dgamma, part_b, dbeta, nb, H, st);
  }
  hook(false);  // (its reductions are inside ln_bwd_t)
  if (t == DType::F32)
    return ln_bwd_t<float>(du, x, mean, rstd, gamma, dres, dx, part_g, part_b, stat, dgamma,
                           dbeta, M, H, st);
  return ln_bwd_t<__nv_bfloat16>(du, x, mean, rstd, gamma, dres, dx, part_g, part_b, stat,
                                 dgamma, dbeta, M, H, st);
}

cudaError_t colsum_accum(const void* in, int64_t ld, int M, int N, DType t, float* part,
                         float* out, cudaStream_t st) {
  if (M == 0 || N == 0) return cudaSuccess;
  const int nb = colsum_blocks(M);
  // gridDim.y is limited to 65535: beyond that each CTA row takes several
  // partial rows (same partial sums, same order)
  const int gy = std::min(nb, 65535);
  const dim3 pgrid((N + COLS_PER_CTA - 1) / COLS_PER_CTA, gy);
  cudaError_t e;
  const size_t esz = t == DType::F32 ? 4 : 2;
  const int V = 16 / (int)esz;  // columns per thread of the vector kernel
  if (N % V == 0 && ld % V == 0 && ((uintptr_t)in % 16) == 0) {
    const dim3 vgrid((N + V * COL_THREADS - 1) / (V * COL_THREADS), gy);
    if (t == DType::F32)
      e = launch_pdl(colsum_vec_kernel<float>, vgrid, dim3(COL_THREADS), 0, st, (const float*)in,
                     ld, M, N, part);
    else
      e = launch_pdl(colsum_vec_kernel<__nv_bfloat16>, vgrid, dim3(COL_THREADS), 0, st,
                     (const __nv_bfloat16*)in, ld, M, N, part);
  } else if (t == DType::F32)
    e = launch_pdl(colsum_part_kernel<float>, pgrid, dim3(COL_THREADS), 0, st, (const float*)in,
                   ld, M, N, part);
  else
    e = launch_pdl(colsum_part_kernel<__nv_bfloat16>, pgrid, dim3(COL_THREADS), 0, st,
                   (const __nv_bfloat16*)in, ld, M, N, part);
  if (e != cudaSuccess) return e;
  return reduce_parts(part, out, nullptr, nullptr, nb, N, st);
}

cudaError_t add_into(const void* a, const float* b, void* out, int64_t n, DType t,
                     cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int grid = (int)std::min<int64_t>((n + 255) / 256, 152 * 16);
  if (t == DType::F32)
    return launch_pdl(add_into_kernel<float>, dim3(grid), dim3(256), 0, st, (const float*)a, b,
                      (float*)out, n);
  return launch_pdl(add_into_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, st,
                    (const __nv_bfloat16*)a, b, (__nv_bfloat16*)out, n);
}

}  // namespace oases
