// Shared device helpers of the Oases GB300 library: element types, GeLU, and
// the launch descriptors every kernel family takes.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

namespace oases {

// ---- host: per-device state for a process that drives several GPUs -------
inline int current_device() {
  int d = 0;
  return cudaGetDevice(&d) == cudaSuccess ? d : 0;
}
// Unique id of the calling thread's current CUDA context (the driver's
// context id, never reused within the process), 0 if there is none yet.
// Host caches of per-device state (events, streams, kernel attributes, device
// addresses) keep the id they were made under and are remade when it changes,
// so state of a context that was destroyed (cudaDeviceReset) is never reused.
uint64_t current_ctx_id();

// Runs a per-device setup step (a kernel attribute, say) once per device and
// context: run(f) calls f until it succeeds on the current device, then skips
// it there while the context stays the same.  Safe from several threads (f may
// run more than once concurrently, so it must be idempotent).  Device ordinals
// >= 64 run f on every call.
struct DeviceOnce {
  std::atomic<uint64_t> ctx[64] = {};
  template <typename F>
  cudaError_t run(F&& f) {
    const int dev = current_device();
    const uint64_t id = current_ctx_id();
    if (dev < 64 && id != 0 && ctx[dev].load(std::memory_order_acquire) == id) return cudaSuccess;
    const cudaError_t e = f();
    if (e == cudaSuccess && dev < 64) ctx[dev].store(current_ctx_id(), std::memory_order_release);
    return e;
  }
};

// E4M3 (FP8, 1-4-3, bias 7) occurs only as a GEMM operand of the MX path,
// with UE8M0 block scales beside it.
enum class DType : int { F32 = 0, BF16 = 1, E4M3 = 2 };

// Kernel launches issued by this host thread (read and reset by the scheduler).
extern thread_local int g_launch_count;
#define OASES_COUNT_LAUNCH() (++::oases::g_launch_count)

inline size_t dtype_size(DType t) { return t == DType::F32 ? 4 : t == DType::BF16 ? 2 : 1; }

// Programmatic dependent launch.  Every kernel of the library is launched with
// programmatic stream serialization, so it may start while its predecessor on
// the stream is finishing; it must call pdl_wait() before its first global
// memory access (read or write), which returns once the predecessor grid has
// completed and its writes are visible.  pdl_trigger() lets the next kernel on
// the stream be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  ++g_launch_count;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Element load / store in fp32 registers.
__device__ __forceinline__ float ld_elem(const float* p, int64_t i) { return p[i]; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* p, int64_t i) {
  return __bfloat162float(p[i]);
}
__device__ __forceinline__ void st_elem(float* p, int64_t i, float v) { p[i] = v; }
__device__ __forceinline__ void st_elem(__nv_bfloat16* p, int64_t i, float v) {
  p[i] = __float2bfloat16_rn(v);
}
__device__ __forceinline__ float load_any(const void* p, DType t, int64_t i) {
  return t == DType::F32 ? static_cast<const float*>(p)[i]
                         : __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}
__device__ __forceinline__ void store_any(void* p, DType t, int64_t i, float v) {
  if (t == DType::F32)
    static_cast<float*>(p)[i] = v;
  else
    static_cast<__nv_bfloat16*>(p)[i] = __float2bfloat16_rn(v);
}

// GeLU in its exact form a * Phi(a), Phi the standard normal CDF, and its
// derivative Phi(a) + a * phi(a), phi the standard normal density.
//
// Phi is evaluated through erf with formula 7.1.26 of Abramowitz & Stegun,
// Handbook of Mathematical Functions: for x >= 0,
//   erf(x) = 1 - t (a1 + t (a2 + t (a3 + t (a4 + t a5)))) exp(-x^2) + e(x),
//   t = 1 / (1 + p x),  |e(x)| <= 1.5e-7,
//   p = 0.3275911, a1..a5 = 0.254829592, -0.284496736, 1.421413741,
//   -1.453152027, 1.061405429,
// and erf(-x) = -erf(x).  With x = |a| / sqrt(2), exp(-x^2) = exp(-a^2 / 2) is
// also the Gaussian density's exponential, so GeLU' costs one more FMA.  One
// reciprocal, one exp2 and a handful of FMAs, no branch.
__device__ __forceinline__ void gelu_cdf_pdf(float a, float& cdf, float& pdf) {
  const float x = fabsf(a) * 0.70710678118654752f;
  float t, e;
  // hardware reciprocal and base-2 exponential (relative error ~2^-22; an
  // exponential that underflows is flushed to 0, i.e. erf = 1 exactly)
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(fmaf(0.3275911f, x, 1.0f)));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(-x * x * 1.4426950408889634f));  // exp(-a^2/2)
  const float poly =
      t * fmaf(t, fmaf(t, fmaf(t, fmaf(t, 1.061405429f, -1.453152027f), 1.421413741f),
                       -0.284496736f),
               0.254829592f);
  const float erf_abs = fmaf(-poly, e, 1.0f);
  cdf = 0.5f + 0.5f * copysignf(erf_abs, a);
  pdf = 0.39894228040143268f * e;
}
__device__ __forceinline__ float gelu_f(float a) {
  float cdf, pdf;
  gelu_cdf_pdf(a, cdf, pdf);
  return a * cdf;
}
__device__ __forceinline__ float gelu_grad_f(float a) {
  float cdf, pdf;
  gelu_cdf_pdf(a, cdf, pdf);
  return fmaf(a, pdf, cdf);
}

// ---- two values at a time: packed fp32x2 arithmetic (sm_100 family) --------
// Each lane of a packed fma / mul / add rounds exactly like the scalar
// operation, so the pair forms below return the same bits as gelu_f,
// gelu_grad_f and scalar adds while issuing about half the instructions.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  return (uint64_t)__float_as_uint(a) | ((uint64_t)__float_as_uint(b) << 32);
}
__device__ __forceinline__ float f2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_mul(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2_splat(float a) { return f2_pack(a, a); }
// (a0, a1) += (b0, b1)
__device__ __forceinline__ void add2_inplace(float& a0, float& a1, float b0, float b1) {
  const uint64_t r = f2_add(f2_pack(a0, a1), f2_pack(b0, b1));
  a0 = f2_lo(r);
  a1 = f2_hi(r);
}
// Phi and phi of a pair, the operations of gelu_cdf_pdf in the same order.
__device__ __forceinline__ void gelu_cdf_pdf2(uint64_t a, uint64_t& cdf, uint64_t& pdf) {
  constexpr uint64_t ABS = 0x7fffffff7fffffffull, SIGN = 0x8000000080000000ull;
  const uint64_t x = f2_mul(a & ABS, f2_splat(0.70710678118654752f));
  const uint64_t den = f2_fma(f2_splat(0.3275911f), x, f2_splat(1.0f));
  const uint64_t arg = f2_mul(f2_mul(x, x), f2_splat(-1.4426950408889634f));
  float t0, t1, e0, e1;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t0) : "f"(f2_lo(den)));
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(t1) : "f"(f2_hi(den)));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e0) : "f"(f2_lo(arg)));
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e1) : "f"(f2_hi(arg)));
  const uint64_t t = f2_pack(t0, t1), e = f2_pack(e0, e1);
  uint64_t poly = f2_fma(t, f2_splat(1.061405429f), f2_splat(-1.453152027f));
  poly = f2_fma(t, poly, f2_splat(1.421413741f));
  poly = f2_fma(t, poly, f2_splat(-0.284496736f));
  poly = f2_fma(t, poly, f2_splat(0.254829592f));
  poly = f2_mul(t, poly);
  const uint64_t erf_abs = f2_fma(poly ^ SIGN, e, f2_splat(1.0f));
  const uint64_t erf_s = (erf_abs & ABS) | (a & SIGN);  // copysign(erf_abs, a)
  cdf = f2_fma(f2_splat(0.5f), erf_s, f2_splat(0.5f));
  pdf = f2_mul(f2_splat(0.39894228040143268f), e);
}
// (a0, a1) = (gelu(a0), gelu(a1))
__device__ __forceinline__ void gelu2_inplace(float& a0, float& a1) {
  const uint64_t a = f2_pack(a0, a1);
  uint64_t cdf, pdf;
  gelu_cdf_pdf2(a, cdf, pdf);
  const uint64_t r = f2_mul(a, cdf);
  a0 = f2_lo(r);
  a1 = f2_hi(r);
}
// (a0, a1) = (gelu(a0), gelu(a1)) and (d0, d1) = (gelu'(a0), gelu'(a1))
__device__ __forceinline__ void gelu_and_grad2(float& a0, float& a1, float& d0, float& d1) {
  const uint64_t a = f2_pack(a0, a1);
  uint64_t cdf, pdf;
  gelu_cdf_pdf2(a, cdf, pdf);
  const uint64_t g = f2_mul(a, cdf), d = f2_fma(a, pdf, cdf);
  a0 = f2_lo(g);
  a1 = f2_hi(g);
  d0 = f2_lo(d);
  d1 = f2_hi(d);
}

// ---------------------------------------------------------------------------
// GEMM description shared by the SIMT and the tensor-core kernels.
//   D[m, n] = sum_k A(m, k) * B(n, k), m < M, n < N, k < K.
//   A(m, k) = a_kmajor ? A[m * lda + k] : A[k * lda + m]
//   B(n, k) = b_kmajor ? B[n * ldb + k] : B[k * ldb + n]
// followed by an epilogue on the fp32 accumulator.
// ---------------------------------------------------------------------------
enum class Epi : int {
  Store = 0,      // C = acc
  Bias = 1,       // C = acc + bias[n]
  BiasGelu = 2,   // C = gelu(acc + bias[n]); C2 (if given) = gelu'(acc + bias[n])
  BiasResid = 3,  // C = acc + bias[n] + aux[m, n]
  Mul = 4,        // C = acc * aux[m, n] (the GeLU backward with aux = the stored gelu')
  Accum = 5,      // C (fp32) += acc
};

struct GemmArgs {
  int M = 0, N = 0, K = 0;
  DType in_t = DType::BF16;
  const void* A = nullptr;
  int64_t lda = 0;
  bool a_kmajor = true;
  const void* B = nullptr;
  int64_t ldb = 0;
  bool b_kmajor = true;
  Epi epi = Epi::Store;
  void* C = nullptr;
  int64_t ldc = 0;
  DType c_t = DType::BF16;
  void* C2 = nullptr;  // BiasGelu derivative output gelu'(acc + bias), type c_t, leading dim ldc
  const void* bias = nullptr;  // [N], type in_t
  const void* aux = nullptr;   // [M, N] with leading dim ld_aux, type aux_t
  int64_t ld_aux = 0;
  DType aux_t = DType::BF16;
  int tma_store = 0;  // set by the tensor-core path: outputs leave through TMA stores
  // Split contraction (tensor-core path only, Epi::Store): `splits` independent
  // products in one launch.  Product s contracts over kpieces ranges of K
  // coordinates, piece p covering [p * kpiece_stride + s * K / kpieces, + K / kpieces)
  // of A's and B's K axis (k_extent wide), and writes rows [s * c_split_rows, + M)
  // of C.  splits = 1, kpieces = 1 is the plain GEMM.
  int splits = 1, kpieces = 1;
  int64_t kpiece_stride = 0, k_extent = 0, c_split_rows = 0;
  // 1 when another stream's work runs beside this GEMM (the two sub-batch
  // streams): SMs that 256-wide tiles leave idle are then filled by the other
  // stream, so the dispatcher always takes the faster 256-wide pair tiles.
  int concurrent = 0;
  // MX path (in_t == E4M3, both operands K-major): UE8M0 scales of A's and B's
  // 32-element K blocks, in 512-byte tiles of 128 rows x 4 blocks; tile
  // (row block rb, K group kg) at byte (rb * ceil(K / 128) + kg) * 512, row r
  // of the tile, block j at byte (r % 32) * 16 + (r / 32) * 4 + j.  Bias and
  // aux stay bf16.
  const uint8_t* a_sf = nullptr;
  const uint8_t* b_sf = nullptr;
  // Optional (bf16 C through the TMA-store epilogue, no split slabs): the
  // column sums of C as stored, one partial row of N floats per 32-row slab
  // of C (ceil(M / 32) rows, every element written), for a fixed-order
  // reduction by the caller.  The launch sets *colsum_rows to that count when
  // it takes them, and leaves it alone (and colsum_part unwritten) otherwise.
  float* colsum_part = nullptr;
  int* colsum_rows = nullptr;
  // Optional (bf16 C through the TMA-store epilogue with 256-wide tiles, N a
  // multiple of 128): for each row m and each group of 128 columns from n0,
  // rowdot_out[(n0 / 128) * rowdot_ld + m] = the sum over the group of C[m][n]
  // as stored times rowdot_aux[m][n] (bf16, leading dim rowdot_lda) -- the
  // attention backward's delta = rowsum(dO * O) per head when C = dO.  The
  // launch sets *rowdot_done = 1 when it takes it.
  const void* rowdot_aux = nullptr;
  int64_t rowdot_lda = 0;
  float* rowdot_out = nullptr;
  int64_t rowdot_ld = 0;
  int* rowdot_done = nullptr;
};

// Returns cudaSuccess or the launch error.  Picks the tensor-core kernel when
// the operands allow it and the SIMT kernel otherwise.
cudaError_t gemm(const GemmArgs& g, cudaStream_t st);
cudaError_t gemm_simt(const GemmArgs& g, cudaStream_t st);
// Tensor-core path (tcgen05 + TMA); returns cudaErrorNotSupported when the
// operands do not meet its alignment rules.
cudaError_t gemm_tc(const GemmArgs& g, cudaStream_t st);
bool gemm_tc_supported(const GemmArgs& g);
// MX-FP8 path: E4M3 operands with block-32 UE8M0 scales (kind::mxf8f6f4).
bool gemm_mx_supported(const GemmArgs& g);
cudaError_t gemm_mx(const GemmArgs& g, cudaStream_t st);
// Quantisers to the MX layout (E4M3 codes + scale tiles above).
//   rows: q[r, k] = E4M3(x[r, k] / X[r, k / 32]) for x [R, K] (leading dim ld)
//   cols: the same for the transpose x^T [C, R] of x [R, C]: q[c, r] with blocks
//         of 32 along r (q has leading dim ldq, at least R)
// X = 2^(floor(log2(max |block|)) - 8), clamped to the UE8M0 range; 1 for an
// all-zero block.  Every byte of every scale tile is written (127 = 2^0 for
// rows and blocks beyond the matrix).
cudaError_t mx_quantize_rows(const void* x, int64_t ld, int R, int K, DType t, uint8_t* q,
                             int64_t ldq, uint8_t* sf, cudaStream_t st);
cudaError_t mx_quantize_cols(const void* x, int64_t ld, int R, int C, DType t, uint8_t* q,
                             int64_t ldq, uint8_t* sf, cudaStream_t st);
inline int64_t mx_sf_bytes(int rows, int K) {
  return (int64_t)((rows + 127) / 128) * ((K + 127) / 128) * 512;
}

// ---------------------------------------------------------------------------
// Row-wise LayerNorm and column reductions (norm.cu).
// ---------------------------------------------------------------------------
// u = (x - mean) * rstd * gamma + beta over each row of [M, H]; writes mean,
// rstd (fp32, [M]).
cudaError_t layer_norm_fwd(const void* x, const void* gamma, const void* beta, void* u,
                           float* mean, float* rstd, int M, int H, float eps, DType t,
                           cudaStream_t st);
// dx = rstd * (g - mean(g) - xhat * mean(g * xhat)) (+ dres), g = du * gamma;
// du fp32 [M, H]; x, dres, dx in t.  Per-row-block partial sums of du * xhat
// and du go to part_g / part_b ([ln_bwd_blocks(M), H] fp32) and the two row
// means to stat ([M] float2); a last pass adds the partials' column sums to
// dgamma / dbeta in a fixed order.
int ln_bwd_blocks(int M);
cudaError_t layer_norm_bwd(const float* du, const void* x, const float* mean, const float* rstd,
                           const void* gamma, const void* dres, void* dx, float* part_g,
                           float* part_b, float2* stat, float* dgamma, float* dbeta, int M, int H,
                           DType t, cudaStream_t st);
// out[n] += sum_m in[m, n] for in [M, N] (type t, leading dim ld); partials in
// part ([colsum_blocks(M), N] fp32).  Deterministic: fixed summation order.
int colsum_blocks(int M);
cudaError_t colsum_accum(const void* in, int64_t ld, int M, int N, DType t, float* part,
                         float* out, cudaStream_t st);
// Shard sum of the separate-reduction mode: out[m, n] = sum_{k<w} part[k][m, n]
// (+ bias[n]) (+ resid[m, n]); part fp32 with pstride floats between shards;
// bias / resid of type in_t, out of type out_t.  Fixed order k = 0, 1, ...
cudaError_t shard_sum(const float* part, int64_t pstride, int w, const void* bias,
                      const void* resid, void* out, DType out_t, DType in_t, int M, int N,
                      cudaStream_t st);
// y = x + a elementwise (n elements, type t); used for the residual gradient
// when there is no LayerNorm.
cudaError_t add_into(const void* a, const float* b, void* out, int64_t n, DType t,
                     cudaStream_t st);

// ---------------------------------------------------------------------------
// Causal softmax attention over heads (attn.cu).
//   qkv [M, 3H] (rows of one sequence contiguous; Q at column h*d, K at
//   H + h*d, V at 2H + h*d), o [M, H], lse [heads, M] fp32.
// ---------------------------------------------------------------------------
struct AttnArgs {
  int batch = 0, seq = 0, heads = 0, head_dim = 0, hidden = 0;
  bool causal = true;
  DType t = DType::BF16;
  const void* qkv = nullptr;
  void* o = nullptr;
  float* lse = nullptr;
  // backward
  const void* d_o = nullptr;  // [M, H]
  float* delta = nullptr;     // [heads, M]: rowsum(dO * O)
  void* dqkv = nullptr;       // [M, 3H]
  bool delta_ready = false;   // delta already holds rowsum(dO * O) (the dO GEMM's epilogue)
};
cudaError_t attention_fwd(const AttnArgs& a, cudaStream_t st);
cudaError_t attention_bwd(const AttnArgs& a, cudaStream_t st);
cudaError_t attention_fwd_simt(const AttnArgs& a, cudaStream_t st);
// Tensor-core forward (bf16, head dimension 128); see attn_tc.cu.
bool attention_tc_supported(const AttnArgs& a);
cudaError_t attention_fwd_tc(const AttnArgs& a, cudaStream_t st);
cudaError_t attention_bwd_tc(const AttnArgs& a, cudaStream_t st);
int attention_read_and_clear_error();
// Debugging aid: host-mapped int[768] that the attention kernels' thread 0
// fills with progress markers (nullptr switches them off).
cudaError_t attention_set_progress(int* p);
cudaError_t attention_set_timeline(unsigned long long* p);
cudaError_t attention_bwd_simt(const AttnArgs& a, cudaStream_t st);

// Reads and clears the error word the tensor-core kernels set when a bounded
// wait expires (0 = none, -1 = could not read).
int gemm_read_and_clear_error();

}  // namespace oases
