// Causal softmax attention forward on the 5th-generation tensor cores
// (tcgen05 + TMEM + TMA), head dimension 128, bf16 in, fp32 softmax.
//
// One CTA (128 threads) owns 128 queries of one (sequence, head).  Thread r is
// query row r: TMEM lane r holds its scores.  Per block of 128 keys j:
//   S_j  = Q K_j^T          tcgen05.mma, A = Q (smem), B = K_j (smem) -> TMEM
//   P_j  = exp(S_j - m_j)   the thread's row, online max m and sum l (fp32),
//                           written as bf16 into shared memory in the
//                           128-byte-swizzled K-major layout the MMA reads
//   O   += P_j V_j          tcgen05.mma, A = P_j (smem), B = V_j (smem,
//                           MN-major) -> a TMEM buffer the thread adds into its
//                           register accumulator O = O * exp(m_{j-1} - m_j) + PV
// S_{j+1} is issued before the softmax of block j and PV_j is added one block
// later, so the tensor core overlaps the exponentials.  K/V blocks are loaded
// by TMA two blocks ahead.  Key blocks past the diagonal are skipped; keys
// past the diagonal inside the diagonal block (and past the sequence end) get
// weight 0.  LSE = m + log(l) is stored per (head, row) for the backward.
//
// Every mbarrier wait is bounded (ptx::mbar_wait); on expiry the CTA records
// g_attn_error, stops issuing work and drains what is in flight.
#include <cuda.h>

#include <math.h>

#include <mutex>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace oases {

__device__ int g_attn_error;

namespace {

constexpr int D = 128;                 // head dimension
constexpr int BQ = 128, BKV = 128;     // query rows per CTA, keys per block
constexpr int BOX = 128 * 64 * 2;      // one TMA box: 128 rows x 64 bf16 (16 KB)
constexpr int TILE = 2 * BOX;          // 128 rows x 128 bf16 (32 KB)
constexpr int KV_STAGES = 2;
// shared-memory map (offsets from a 1024-aligned base)
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE;                  // KV_STAGES tiles
constexpr int OFF_V = OFF_K + KV_STAGES * TILE;      // KV_STAGES tiles
constexpr int OFF_P = OFF_V + KV_STAGES * TILE;      // 2 tiles (double-buffered P)
constexpr int OFF_BAR = OFF_P + 2 * TILE;
constexpr int NBAR = 1 + 2 * KV_STAGES + 2 + 2 + 1;  // q, K full, V full, s, pv, drain
constexpr int FWD_SMEM = OFF_BAR + 8 * NBAR + 16 + 1024;
constexpr int NT = 128;

// S = Q K^T: M = 128 queries, N = 128 keys, both operands K-major (over d).
constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(BQ, BKV, false, false);
// O = P V: M = 128 queries, N = 128 dims; P K-major (over keys), V MN-major.
constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(BQ, D, false, true);

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// Descriptor of a K-major operand tile [128 rows][128 cols] stored as two
// 128-byte-swizzled 64-column boxes, for k-step kk (16 columns) of 8.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
  return ptx::smem_desc_sw128(tile + (kk >> 2) * BOX + (kk & 3) * 32, 16, 1024);
}
// Descriptor of an MN-major operand [128 k-rows][128 n-cols] stored as two
// boxes of 64 n-columns, for k-step kk (16 k-rows) of 8.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
  return ptx::smem_desc_sw128(tile + kk * 2048, BOX, 1024);
}

struct FwdArgs {
  __nv_bfloat16* o;
  float* lse;
  int S, H, heads, M;  // sequence length, hidden, heads, rows of this call
  int causal;
  float scale_log2;    // log2(e) / sqrt(d)
};

__global__ void __launch_bounds__(NT, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm, const FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + OFF_BAR;
  const uint32_t bar_q = bars;
  auto bar_k = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_v = [&](int s) { return bars + 8u * (1 + KV_STAGES + s); };
  auto bar_s = [&](int i) { return bars + 8u * (1 + 2 * KV_STAGES + i); };
  auto bar_pv = [&](int i) { return bars + 8u * (3 + 2 * KV_STAGES + i); };
  const uint32_t bar_drain = bars + 8u * (5 + 2 * KV_STAGES);
  const uint32_t tslot = bars + 8u * NBAR;

  const int tid = threadIdx.x, warp = tid / 32;
  const int tile = gridDim.x - 1 - blockIdx.x;  // heavy (late) query tiles first
  const int h = blockIdx.y, b = blockIdx.z;
  const int q0 = tile * BQ;
  const int row0 = b * a.S;
  const int nkv_all = (a.S + BKV - 1) / BKV;
  const int nkv = a.causal ? min(tile + 1, nkv_all) : nkv_all;
  const int col_q = h * D, col_k = a.H + h * D, col_v = 2 * a.H + h * D;

  if (tid == 0) {
    ptx::mbar_init(bar_q, 1);
    for (int s = 0; s < KV_STAGES; ++s) {
      ptx::mbar_init(bar_k(s), 1);
      ptx::mbar_init(bar_v(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(bar_s(i), 1);
      ptx::mbar_init(bar_pv(i), 1);
    }
    ptx::mbar_init(bar_drain, 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tm);
  }
  if (warp == 0) {
    ptx::tmem_alloc(tslot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + (tslot - base));
  const uint32_t t_s[2] = {tmem, tmem + 128};
  const uint32_t t_pv[2] = {tmem + 256, tmem + 384};
  pdl_wait();
  pdl_trigger();

  // Thread 0 issues every TMA load and MMA.  Loads in flight per stage are
  // tracked (bit s of k_issued / v_issued, parity in k_par / v_par) so that a
  // CTA that stops early can wait for them before it exits.
  bool ok = true;
  uint32_t k_issued = 0, k_par = 0, v_issued = 0, v_par = 0;
  auto load_k = [&](int j) {
    const int s = j % KV_STAGES;
    ptx::mbar_arrive_expect_tx(bar_k(s), TILE);
    const uint32_t kt = base + OFF_K + s * TILE;
    ptx::tma_load_2d(kt, &tm, bar_k(s), col_k, row0 + j * BKV);
    ptx::tma_load_2d(kt + BOX, &tm, bar_k(s), col_k + 64, row0 + j * BKV);
    k_issued |= 1u << s;
    k_par = (k_par & ~(1u << s)) | ((uint32_t)((j / KV_STAGES) & 1) << s);
  };
  auto load_v = [&](int j) {
    const int s = j % KV_STAGES;
    ptx::mbar_arrive_expect_tx(bar_v(s), TILE);
    const uint32_t vt = base + OFF_V + s * TILE;
    ptx::tma_load_2d(vt, &tm, bar_v(s), col_v, row0 + j * BKV);
    ptx::tma_load_2d(vt + BOX, &tm, bar_v(s), col_v + 64, row0 + j * BKV);
    v_issued |= 1u << s;
    v_par = (v_par & ~(1u << s)) | ((uint32_t)((j / KV_STAGES) & 1) << s);
  };
  auto issue_s = [&](int j) {  // K_j must have landed
    const uint32_t qt = base + OFF_Q, kt = base + OFF_K + (j % KV_STAGES) * TILE;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      ptx::mma_bf16(t_s[j & 1], kmajor_desc(qt, kk), kmajor_desc(kt, kk), IDESC_S, kk > 0);
    ptx::mma_commit(bar_s(j & 1));
  };

  if (tid == 0) {
    ptx::mbar_arrive_expect_tx(bar_q, TILE);
    ptx::tma_load_2d(base + OFF_Q, &tm, bar_q, col_q, row0 + q0);
    ptx::tma_load_2d(base + OFF_Q + BOX, &tm, bar_q, col_q + 64, row0 + q0);
    for (int j = 0; j < KV_STAGES && j < nkv; ++j) {
      load_k(j);
      load_v(j);
    }
    ok = ptx::mbar_wait(bar_q, 0) && ptx::mbar_wait(bar_k(0), 0);
    if (ok) {
      ptx::tc_fence_after();
      issue_s(0);
    }
  }

  const int qi = q0 + tid;  // this thread's query position
  float O[D];
#pragma unroll
  for (int c = 0; c < D; ++c) O[c] = 0.f;
  float m2 = -INFINITY, l = 0.f, corr_prev = 1.f;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  bool done_all = true;

  for (int j = 0; j < nkv; ++j) {
    // (1) S_{j+1} overlaps this block's softmax
    if (tid == 0 && ok && j + 1 < nkv) {
      ok = ptx::mbar_wait(bar_k((j + 1) % KV_STAGES), ((j + 1) / KV_STAGES) & 1);
      if (ok) {
        ptx::tc_fence_after();
        issue_s(j + 1);
      }
    }
    // (2) row max of S_j; afterwards K stage j % 2 is free for K_{j+2}
    if (!ptx::mbar_wait(bar_s(j & 1), (j >> 1) & 1)) ok = false;
    ptx::tc_fence_after();
    if (tid == 0 && ok && j + 2 < nkv) load_k(j + 2);
    const int kbase = j * BKV;
    float mx = -INFINITY;
#pragma unroll 1
    for (int c0 = 0; c0 < BKV; c0 += 32) {
      float v[32];
      ptx::tmem_ld32(t_s[j & 1] + lane_off + c0, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int key = kbase + c0 + i;
        const bool valid = key < a.S && (!a.causal || key <= qi);
        if (valid) mx = fmaxf(mx, v[i] * a.scale_log2);
      }
    }
    const float m_new = fmaxf(m2, mx);
    const float corr = (m_new == -INFINITY) ? 1.f : exp2f(m2 - m_new);
    // (3) PV_{j-1} complete: fold it into O; its V stage takes V_{j+1}
    if (j >= 1) {
      if (!ptx::mbar_wait(bar_pv((j - 1) & 1), ((j - 1) >> 1) & 1)) ok = false;
      ptx::tc_fence_after();
      if (tid == 0 && ok && j + 1 < nkv) load_v(j + 1);
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float v[32];
        ptx::tmem_ld32(t_pv[(j - 1) & 1] + lane_off + c0, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) O[c0 + i] = fmaf(O[c0 + i], corr_prev, v[i]);
      }
    }
    // (4) P_j = exp2(s - m_new) as bf16 into the swizzled P buffer (j & 1)
    float rs = 0.f;
    const uint32_t pbuf = OFF_P + (j & 1) * TILE;
#pragma unroll 1
    for (int c0 = 0; c0 < BKV; c0 += 32) {
      float v[32];
      ptx::tmem_ld32(t_s[j & 1] + lane_off + c0, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int key = kbase + c0 + i;
        const bool valid = key < a.S && (!a.causal || key <= qi) && m_new != -INFINITY;
        const float p = valid ? exp2f(v[i] * a.scale_log2 - m_new) : 0.f;
        v[i] = p;
        rs += p;
      }
      // 32 keys = 4 16-byte units of this row in chunk c0 / 64
      uint8_t* rowp = gbase + pbuf + (c0 >> 6) * BOX + tid * 128;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int unit = ((c0 & 63) >> 3) + u;
        const uint4 w = make_uint4(pack2(v[8 * u], v[8 * u + 1]), pack2(v[8 * u + 2], v[8 * u + 3]),
                                   pack2(v[8 * u + 4], v[8 * u + 5]),
                                   pack2(v[8 * u + 6], v[8 * u + 7]));
        *reinterpret_cast<uint4*>(rowp + ((unit ^ (tid & 7)) << 4)) = w;
      }
    }
    l = l * corr + rs;
    m2 = m_new;
    corr_prev = corr;
    // (5) make P visible to the tensor core; all threads decide together
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    ptx::tc_fence_before();
    if (__syncthreads_or(!ok)) {
      done_all = false;
      break;
    }
    if (tid == 0) {
      ok = ptx::mbar_wait(bar_v(j % KV_STAGES), (j / KV_STAGES) & 1);
      if (ok) {
        ptx::tc_fence_after();
        const uint32_t pt = base + pbuf, vt = base + OFF_V + (j % KV_STAGES) * TILE;
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          ptx::mma_bf16(t_pv[j & 1], kmajor_desc(pt, kk), mnmajor_desc(vt, kk), IDESC_PV, kk > 0);
        ptx::mma_commit(bar_pv(j & 1));
      }
    }
  }
  if (done_all && nkv >= 1) {  // fold the last PV
    const int j = nkv - 1;
    if (!ptx::mbar_wait(bar_pv(j & 1), (j >> 1) & 1)) ok = false;
    ptx::tc_fence_after();
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      float v[32];
      ptx::tmem_ld32(t_pv[j & 1] + lane_off + c0, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) O[c0 + i] = fmaf(O[c0 + i], corr_prev, v[i]);
    }
  }
  if (done_all && ok && qi < a.S) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint4* orow = reinterpret_cast<uint4*>(a.o + (int64_t)(row0 + qi) * a.H + h * D);
#pragma unroll
    for (int u = 0; u < D / 8; ++u)
      orow[u] = make_uint4(pack2(O[8 * u] * inv, O[8 * u + 1] * inv),
                           pack2(O[8 * u + 2] * inv, O[8 * u + 3] * inv),
                           pack2(O[8 * u + 4] * inv, O[8 * u + 5] * inv),
                           pack2(O[8 * u + 6] * inv, O[8 * u + 7] * inv));
    a.lse[(int64_t)h * a.M + row0 + qi] = (m2 + log2f(l)) * 0.69314718055994531f;
  }
  if (!(done_all && ok)) atomicExch(&g_attn_error, 1);
  if (tid == 0) {
    // drain: issued MMAs complete and issued loads land before the CTA exits
    ptx::mma_commit(bar_drain);
    bool dr = ptx::mbar_wait(bar_drain, 0);
    for (int s = 0; s < KV_STAGES; ++s) {
      if ((k_issued >> s) & 1u) dr = ptx::mbar_wait(bar_k(s), (k_par >> s) & 1u) && dr;
      if ((v_issued >> s) & 1u) dr = ptx::mbar_wait(bar_v(s), (v_par >> s) & 1u) && dr;
    }
    dr = ptx::mbar_wait(bar_q, 0) && dr;
    if (!dr) atomicExch(&g_attn_error, 2);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// Tensor map over qkv [M, 3H] bf16, box 128 rows x 64 columns, 128-byte swizzle.
bool qkv_map(CUtensorMap* m, const void* qkv, int M, int H) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)3 * H, (cuuint64_t)M};
  const cuuint64_t strides[1] = {(cuuint64_t)3 * H * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(qkv), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

bool attention_tc_supported(const AttnArgs& a) {
  return a.t == DType::BF16 && a.head_dim == D && a.hidden % 8 == 0 &&
         (((uintptr_t)a.qkv | (uintptr_t)a.o) & 15) == 0 && encode_fn() != nullptr;
}

cudaError_t attention_fwd_tc(const AttnArgs& a, cudaStream_t st) {
  if (!attention_tc_supported(a)) return cudaErrorNotSupported;
  if (a.batch == 0 || a.seq == 0) return cudaSuccess;
  CUtensorMap m;
  const int M = a.batch * a.seq;
  if (!qkv_map(&m, a.qkv, M, a.hidden)) return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_fwd_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, FWD_SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  FwdArgs fa;
  fa.o = static_cast<__nv_bfloat16*>(a.o);
  fa.lse = a.lse;
  fa.S = a.seq;
  fa.H = a.hidden;
  fa.heads = a.heads;
  fa.M = M;
  fa.causal = a.causal ? 1 : 0;
  fa.scale_log2 = 1.4426950408889634f / sqrtf((float)a.head_dim);
  const dim3 grid((a.seq + BQ - 1) / BQ, a.heads, a.batch);
  return launch_pdl(attn_fwd_tc_kernel, grid, dim3(NT), FWD_SMEM, st, m, fa);
}

int attention_read_and_clear_error() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_attn_error, &z, sizeof(int));
  return v;
}

}  // namespace oases
