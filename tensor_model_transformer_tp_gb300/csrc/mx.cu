// Quantisers to the MX-FP8 operand layout of the block-scaled GEMM
// (OCP Microscaling Formats v1.0: E4M3 elements, one UE8M0 scale per 32
// consecutive elements along the contraction).
//
// For a block v of 32 values with m = max |v|:
//   X = 2^(floor(log2 m) - 8), 8 being the exponent of E4M3's largest power of
//   two (448 = 1.75 * 2^8), clamped to the UE8M0 range [2^-127, 2^127];
//   X = 1 for an all-zero block;
//   element code = E4M3(v / X), nearest value with ties to the even code and
//   magnitudes above 448 saturated to 448 (cvt.rn.satfinite).
// v / X is exact in fp32 (a power-of-two scaling that stays within range), so
// the codes depend only on v.  The scale byte is the biased exponent
// log2(X) + 127.
//
// Scale tiles: 512 bytes per 128 rows x 4 blocks (128 K elements); tile
// (row block rb, K group kg) at byte (rb * kgroups + kg) * 512, row r of the
// tile and block j of the group at byte (r % 32) * 16 + (r / 32) * 4 + j.
// That is the layout tcgen05.cp.32x128b.warpx4 places in tensor memory:
// row r in lane r % 32 of every lane quarter, column r / 32, byte j.  Rows and
// blocks past the matrix get the scale byte 127 (X = 1).
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"

namespace oases {
namespace {

constexpr int MXB = 32;  // elements per scale block

__device__ __forceinline__ float load_f(const float* p) { return *p; }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }

// floor(log2(m)) of a finite m > 0, subnormals included.
__device__ __forceinline__ int floor_log2(float m) {
  const uint32_t b = __float_as_uint(m);
  const int ex = (int)(b >> 23);
  if (ex > 0) return ex - 127;
  return (31 - __clz((int)(b & 0x7FFFFFu))) - 149;
}

// Scale exponent of a block with maximum magnitude amax (0 for amax = 0).
__device__ __forceinline__ int block_exponent(float amax) {
  if (!(amax > 0.f)) return 0;
  return max(-127, min(127, floor_log2(amax) - 8));
}

// 2^-xe as an fp32 (xe in [-127, 126]: always a normal number).
__device__ __forceinline__ float pow2_neg(int xe) { return __int_as_float((127 - xe) << 23); }

// Two E4M3 codes, a at the lower address.
__device__ __forceinline__ uint16_t e4m3x2(float a, float b) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(b), "f"(a));
  return d;
}

__device__ __forceinline__ int64_t sf_offset(int r, int j, int kgroups) {
  return ((int64_t)(r / 128) * kgroups + j / 4) * 512 + (r % 32) * 16 + ((r % 128) / 32) * 4 + (j % 4);
}

// Quantises 32 values (n of them real, the rest 0) into codes + scale byte.
__device__ __forceinline__ uint8_t quantize_block(const float (&v)[MXB], int n, uint8_t (&code)[MXB]) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < MXB; ++i) amax = fmaxf(amax, i < n ? fabsf(v[i]) : 0.f);
  const int xe = block_exponent(amax);
  const float mul = pow2_neg(xe);
#pragma unroll
  for (int i = 0; i < MXB; i += 2) {
    const uint16_t d = e4m3x2(v[i] * mul, v[i + 1] * mul);
    code[i] = (uint8_t)(d & 0xFF);
    code[i + 1] = (uint8_t)(d >> 8);
  }
  return (uint8_t)(xe + 127);
}

// Item i of the padded (row, block) domain: rows_p x blocks_p, block fastest.
template <typename T>
__global__ void __launch_bounds__(256)
mx_rows_kernel(const T* __restrict__ x, int64_t ld, int R, int K, uint8_t* __restrict__ q,
               int64_t ldq, uint8_t* __restrict__ sf, int blocks_p, int64_t items, int vec) {
  pdl_wait();
  pdl_trigger();
  const int kgroups = blocks_p / 4;
  const int nblk = (K + MXB - 1) / MXB;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < items;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int r = (int)(i / blocks_p), j = (int)(i % blocks_p);
    uint8_t s = 127;
    if (r < R && j < nblk) {
      const int k0 = j * MXB, n = min(MXB, K - k0);
      const T* src = x + (int64_t)r * ld + k0;
      float v[MXB];
      if (vec && n == MXB) {
        if constexpr (sizeof(T) == 2) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 w = *reinterpret_cast<const uint4*>(src + 8 * u);
            const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = __bfloat1622float2(h[e]);
              v[8 * u + 2 * e] = f.x;
              v[8 * u + 2 * e + 1] = f.y;
            }
          }
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float4 w = *reinterpret_cast<const float4*>(src + 4 * u);
            v[4 * u] = w.x;
            v[4 * u + 1] = w.y;
            v[4 * u + 2] = w.z;
            v[4 * u + 3] = w.w;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < MXB; ++e) v[e] = e < n ? load_f(src + e) : 0.f;
      }
      uint8_t code[MXB];
      s = quantize_block(v, n, code);
      uint8_t* dst = q + (int64_t)r * ldq + k0;
      if (vec && n == MXB) {
        uint4 w[2];
        uint8_t* wb = reinterpret_cast<uint8_t*>(w);
#pragma unroll
        for (int e = 0; e < MXB; ++e) wb[e] = code[e];
        reinterpret_cast<uint4*>(dst)[0] = w[0];
        reinterpret_cast<uint4*>(dst)[1] = w[1];
      } else {
        for (int e = 0; e < n; ++e) dst[e] = code[e];
      }
    }
    sf[sf_offset(r, j, kgroups)] = s;
  }
}

// The transpose: x [Rx, Cx] (leading dim ld); the quantised matrix is
// x^T [Cx, Rx] with blocks of 32 along Rx.  Item i: output row c (fastest,
// so a warp reads 32 consecutive columns of each input row) and block j.
template <typename T>
__global__ void __launch_bounds__(256)
mx_cols_kernel(const T* __restrict__ x, int64_t ld, int Rx, int Cx, uint8_t* __restrict__ q,
               int64_t ldq, uint8_t* __restrict__ sf, int rows_p, int blocks_p, int64_t items,
               int vec) {
  pdl_wait();
  pdl_trigger();
  const int kgroups = blocks_p / 4;
  const int nblk = (Rx + MXB - 1) / MXB;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < items;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int c = (int)(i % rows_p), j = (int)(i / rows_p);
    uint8_t s = 127;
    if (c < Cx && j < nblk) {
      const int k0 = j * MXB, n = min(MXB, Rx - k0);
      float v[MXB];
#pragma unroll
      for (int e = 0; e < MXB; ++e) v[e] = e < n ? load_f(x + (int64_t)(k0 + e) * ld + c) : 0.f;
      uint8_t code[MXB];
      s = quantize_block(v, n, code);
      uint8_t* dst = q + (int64_t)c * ldq + k0;
      if (vec && n == MXB) {
        uint4 w[2];
        uint8_t* wb = reinterpret_cast<uint8_t*>(w);
#pragma unroll
        for (int e = 0; e < MXB; ++e) wb[e] = code[e];
        reinterpret_cast<uint4*>(dst)[0] = w[0];
        reinterpret_cast<uint4*>(dst)[1] = w[1];
      } else {
        for (int e = 0; e < n; ++e) dst[e] = code[e];
      }
    }
    sf[sf_offset(c, j, kgroups)] = s;
  }
}

int grid_for(int64_t items) {
  return (int)std::min<int64_t>((items + 255) / 256, 152 * 16);
}

}  // namespace

cudaError_t mx_quantize_rows(const void* x, int64_t ld, int R, int K, DType t, uint8_t* q,
                             int64_t ldq, uint8_t* sf, cudaStream_t st) {
  if (R <= 0 || K <= 0) return cudaSuccess;
  const int rows_p = (R + 127) / 128 * 128, blocks_p = (K + 127) / 128 * 4;
  const int64_t items = (int64_t)rows_p * blocks_p;
  const size_t esz = dtype_size(t);
  // 16-byte loads of a 32-element block and 16-byte code stores
  const int vec = ((uintptr_t)x % 16 == 0) && ((ld * esz) % 16 == 0) && ((uintptr_t)q % 16 == 0) &&
                  (ldq % 16 == 0);
  if (t == DType::F32)
    return launch_pdl(mx_rows_kernel<float>, dim3(grid_for(items)), dim3(256), 0, st,
                      (const float*)x, ld, R, K, q, ldq, sf, blocks_p, items, vec);
  if (t == DType::BF16)
    return launch_pdl(mx_rows_kernel<__nv_bfloat16>, dim3(grid_for(items)), dim3(256), 0, st,
                      (const __nv_bfloat16*)x, ld, R, K, q, ldq, sf, blocks_p, items, vec);
  return cudaErrorInvalidValue;
}

cudaError_t mx_quantize_cols(const void* x, int64_t ld, int R, int C, DType t, uint8_t* q,
                             int64_t ldq, uint8_t* sf, cudaStream_t st) {
  if (R <= 0 || C <= 0) return cudaSuccess;
  const int rows_p = (C + 127) / 128 * 128, blocks_p = (R + 127) / 128 * 4;
  const int64_t items = (int64_t)rows_p * blocks_p;
  const int vec = ((uintptr_t)q % 16 == 0) && (ldq % 16 == 0);
  if (t == DType::F32)
    return launch_pdl(mx_cols_kernel<float>, dim3(grid_for(items)), dim3(256), 0, st,
                      (const float*)x, ld, R, C, q, ldq, sf, rows_p, blocks_p, items, vec);
  if (t == DType::BF16)
    return launch_pdl(mx_cols_kernel<__nv_bfloat16>, dim3(grid_for(items)), dim3(256), 0, st,
                      (const __nv_bfloat16*)x, ld, R, C, q, ldq, sf, rows_p, blocks_p, items, vec);
  return cudaErrorInvalidValue;
}

}  // namespace oases

// ---- C ABI -------------------------------------------------------------------
#include "oases_mx.h"

namespace oases {
void api_begin();
void api_set_error(const char* what);
oases_status api_end(cudaError_t e);
}  // namespace oases

extern "C" size_t oases_mx_scale_bytes(int rows, int K) {
  if (rows < 0 || K < 0) return 0;
  return (size_t)oases::mx_sf_bytes(rows, K);
}

extern "C" oases_status oases_mx_quantize(const void* x, int64_t ld, int rows, int K, int dtype,
                                          int transpose, uint8_t* q, int64_t ldq, uint8_t* scales,
                                          void* stream) {
  using namespace oases;
  api_begin();
  if (rows < 0 || K < 0 || (dtype != OASES_F32 && dtype != OASES_BF16) ||
      (transpose != 0 && transpose != 1))
    return OASES_ERR_INVALID_ARG;
  if (rows == 0 || K == 0) return OASES_OK;
  if (!x || !q || !scales || ldq < K || ldq % 16 != 0 || ((uintptr_t)q & 15) ||
      ((uintptr_t)scales & 15) || ld < (transpose ? rows : K))
    return OASES_ERR_INVALID_ARG;
  const DType t = static_cast<DType>(dtype);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t e = transpose ? mx_quantize_cols(x, ld, K, rows, t, q, ldq, scales, st)
                                  : mx_quantize_rows(x, ld, rows, K, t, q, ldq, scales, st);
  return api_end(e);
}

extern "C" oases_status oases_mx_gemm(int M, int N, int K, const uint8_t* a, int64_t lda,
                                      const uint8_t* a_scales, const uint8_t* b, int64_t ldb,
                                      const uint8_t* b_scales, int epilogue, void* C, int64_t ldc,
                                      int c_dtype, void* C2, const void* bias, const void* aux,
                                      int64_t ld_aux, void* stream) {
  using namespace oases;
  api_begin();
  if (M < 0 || N < 0 || K < 0 || epilogue < 0 || epilogue > 5 ||
      (c_dtype != OASES_F32 && c_dtype != OASES_BF16))
    return OASES_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return OASES_OK;
  if (K == 0 || !a || !b || !a_scales || !b_scales || !C || ldc < N) return OASES_ERR_INVALID_ARG;
  const Epi epi = static_cast<Epi>(epilogue);
  if ((epi == Epi::Bias || epi == Epi::BiasGelu || epi == Epi::BiasResid) && !bias)
    return OASES_ERR_INVALID_ARG;
  if ((epi == Epi::BiasResid || epi == Epi::Mul) && (!aux || ld_aux < N))
    return OASES_ERR_INVALID_ARG;
  if (epi == Epi::Accum && c_dtype != OASES_F32) return OASES_ERR_INVALID_ARG;
  for (const void* p : {(const void*)C, (const void*)C2, bias, aux})
    if ((uintptr_t)p & 15) return OASES_ERR_UNSUPPORTED;
  GemmArgs g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.in_t = DType::E4M3;
  g.A = a;
  g.lda = lda;
  g.B = b;
  g.ldb = ldb;
  g.a_sf = a_scales;
  g.b_sf = b_scales;
  g.epi = epi;
  g.C = C;
  g.ldc = ldc;
  g.c_t = static_cast<DType>(c_dtype);
  g.C2 = C2;
  g.bias = bias;
  g.aux = aux;
  g.ld_aux = ld_aux;
  g.aux_t = DType::BF16;
  if (!gemm_mx_supported(g)) return OASES_ERR_UNSUPPORTED;
  return api_end(gemm_mx(g, static_cast<cudaStream_t>(stream)));
}
