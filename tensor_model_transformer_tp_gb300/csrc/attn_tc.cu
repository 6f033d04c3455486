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
// Optional progress markers (debugging aid, off when null): thread 0 of CTA c
// of kernel k writes its current stage to g_attn_progress[k * 256 + c].
__device__ int* g_attn_progress;

namespace {

constexpr int D = 128;                 // head dimension
constexpr int BQ = 128, BKV = 128;     // query rows per CTA, keys per block
constexpr int BOX = 128 * 64 * 2;      // one TMA box: 128 rows x 64 bf16 (16 KB)
constexpr int TILE = 2 * BOX;          // 128 rows x 128 bf16 (32 KB)
constexpr int KV_STAGES = 2;
constexpr int NT = 128;

// S = Q K^T: M = 128 queries, N = 128 keys, both operands K-major (over d).
constexpr uint32_t IDESC_S = ptx::idesc_bf16_f32(BQ, BKV, false, false);
// O = P V: M = 128 queries, N = 128 dims; P K-major (over keys), V MN-major.
constexpr uint32_t IDESC_PV = ptx::idesc_bf16_f32(BQ, D, false, true);

// 2^x on the hardware unit (relative error ~2^-22); results below the
// normal range, including 2^-inf for masked keys, are flushed to 0.
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

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

__device__ __forceinline__ void progress(int kid, int code) {
  int* p = g_attn_progress;
  if (p != nullptr && threadIdx.x == 0) {
    const int cta = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
    if (cta < 256) {
      *reinterpret_cast<volatile int*>(p + kid * 256 + cta) = code;
      __threadfence_system();
    }
  }
}
// Records the first failed wait site (kernel * 100 + site) in g_attn_error.
__device__ __forceinline__ void wait_failed(int code) { atomicCAS(&g_attn_error, 0, code); }

struct FwdArgs {
  __nv_bfloat16* o;
  float* lse;
  int S, H, heads, M;  // sequence length, hidden, heads, rows of this call
  int causal;
  float scale_log2;    // log2(e) / sqrt(d)
};

// Forward shared-memory map: Q, two K stages, three V stages, one P tile.
constexpr int F_KST = 2, F_VST = 3;
constexpr int F_OFF_Q = 0, F_OFF_K = TILE, F_OFF_V = F_OFF_K + F_KST * TILE;
constexpr int F_OFF_P = F_OFF_V + F_VST * TILE, F_OFF_BAR = F_OFF_P + TILE;
constexpr int F_NBAR = 1 + F_KST + F_VST + 2 + 2 + 1;  // q, K, V, s, pv, drain
constexpr int FWD_SMEM = F_OFF_BAR + 8 * F_NBAR + 16 + 1024;
// A row's reference maximum (log2 units) is raised only when the running
// maximum exceeds it by more than this: P = exp2(s - m_ref) <= 256 stays exact
// in fp32 and representable in bf16, and O (accumulated in TMEM) is rescaled
// only on those rare occasions.
constexpr float RESCALE_LOG2 = 8.f;

__global__ void __launch_bounds__(NT, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm, const FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + F_OFF_BAR;
  const uint32_t bar_q = bars;
  auto bar_k = [&](int s) { return bars + 8u * (1 + s); };
  auto bar_v = [&](int s) { return bars + 8u * (1 + F_KST + s); };
  auto bar_s = [&](int i) { return bars + 8u * (1 + F_KST + F_VST + i); };
  auto bar_pv = [&](int i) { return bars + 8u * (3 + F_KST + F_VST + i); };
  const uint32_t bar_drain = bars + 8u * (5 + F_KST + F_VST);
  const uint32_t tslot = bars + 8u * F_NBAR;

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
    for (int s = 0; s < F_KST; ++s) ptx::mbar_init(bar_k(s), 1);
    for (int s = 0; s < F_VST; ++s) ptx::mbar_init(bar_v(s), 1);
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
  const uint32_t t_o = tmem + 256;
  progress(0, 2);
  pdl_wait();
  pdl_trigger();
  progress(0, 3);

  // Thread 0 issues every TMA load and MMA; loads in flight per stage are
  // tracked (issued bit, parity) so that a CTA that stops early waits for them.
  bool ok = true;
  uint32_t k_issued = 0, k_par = 0, v_issued = 0, v_par = 0;
  auto load_k = [&](int j) {
    const int s = j % F_KST;
    ptx::mbar_arrive_expect_tx(bar_k(s), TILE);
    const uint32_t kt = base + F_OFF_K + s * TILE;
    ptx::tma_load_2d(kt, &tm, bar_k(s), col_k, row0 + j * BKV);
    ptx::tma_load_2d(kt + BOX, &tm, bar_k(s), col_k + 64, row0 + j * BKV);
    k_issued |= 1u << s;
    k_par = (k_par & ~(1u << s)) | ((uint32_t)((j / F_KST) & 1) << s);
  };
  auto load_v = [&](int j) {
    const int s = j % F_VST;
    ptx::mbar_arrive_expect_tx(bar_v(s), TILE);
    const uint32_t vt = base + F_OFF_V + s * TILE;
    ptx::tma_load_2d(vt, &tm, bar_v(s), col_v, row0 + j * BKV);
    ptx::tma_load_2d(vt + BOX, &tm, bar_v(s), col_v + 64, row0 + j * BKV);
    v_issued |= 1u << s;
    v_par = (v_par & ~(1u << s)) | ((uint32_t)((j / F_VST) & 1) << s);
  };
  auto issue_s = [&](int j) {  // K_j must have landed
    const uint32_t qt = base + F_OFF_Q, kt = base + F_OFF_K + (j % F_KST) * TILE;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      ptx::mma_bf16(t_s[j & 1], kmajor_desc(qt, kk), kmajor_desc(kt, kk), IDESC_S, kk > 0);
    ptx::mma_commit(bar_s(j & 1));
  };

  if (tid == 0) {
    ptx::mbar_arrive_expect_tx(bar_q, TILE);
    ptx::tma_load_2d(base + F_OFF_Q, &tm, bar_q, col_q, row0 + q0);
    ptx::tma_load_2d(base + F_OFF_Q + BOX, &tm, bar_q, col_q + 64, row0 + q0);
    for (int j = 0; j < F_KST && j < nkv; ++j) load_k(j);
    for (int j = 0; j < F_VST && j < nkv; ++j) load_v(j);
    ok = ptx::mbar_wait(bar_q, 0) && ptx::mbar_wait(bar_k(0), 0);
    if (ok) {
      ptx::tc_fence_after();
      issue_s(0);
    }
  }

  const int qi = q0 + tid;  // this thread's query position
  float m_ref = -INFINITY, l = 0.f;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  bool done_all = true;

  for (int j = 0; j < nkv; ++j) {
    // (1) S_{j+1} overlaps this block's softmax
    if (tid == 0 && ok && j + 1 < nkv) {
      ok = ptx::mbar_wait(bar_k((j + 1) % F_KST), ((j + 1) / F_KST) & 1);
      if (ok) {
        ptx::tc_fence_after();
        issue_s(j + 1);
      }
    }
    // (2) S_j ready.  In issue order S_j follows PV_{j-2}, so PV_{j-2} is done:
    //     K stage j % 2 (S_j) and V stage (j-2) % 3 (PV_{j-2}) are free.
    if (!ptx::mbar_wait(bar_s(j & 1), (j >> 1) & 1)) ok = false;
    ptx::tc_fence_after();
    if (tid == 0 && ok) {
      if (j + 2 < nkv) load_k(j + 2);
      if (j + 1 < nkv && j + 1 >= F_VST) load_v(j + 1);
    }
    const int kbase = j * BKV;
    float sv[BKV];
#pragma unroll
    for (int c0 = 0; c0 < BKV; c0 += 32)
      ptx::tmem_ld32(t_s[j & 1] + lane_off + c0, *reinterpret_cast<float(*)[32]>(sv + c0));
    float mx = -INFINITY;
#pragma unroll
    for (int i = 0; i < BKV; ++i) {
      const int key = kbase + i;
      const bool valid = key < a.S && (!a.causal || key <= qi);
      sv[i] = valid ? sv[i] * a.scale_log2 : -INFINITY;
      mx = fmaxf(mx, sv[i]);
    }
    const float m_new = fmaxf(m_ref, mx);
    // (3) reference maximum
    if (j == 0) {
      m_ref = m_new;
    } else {
      const bool need = m_new > m_ref + RESCALE_LOG2;
      if (__any_sync(0xffffffffu, need)) {  // warp-uniform: tcgen05.ld/st are collective
        if (!ptx::mbar_wait(bar_pv((j - 1) & 1), ((j - 1) >> 1) & 1)) ok = false;
        ptx::tc_fence_after();
        const float f = need ? exp2f(m_ref - m_new) : 1.f;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float v[32];
          ptx::tmem_ld32(t_o + lane_off + c0, v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= f;
          ptx::tmem_st32(t_o + lane_off + c0, v);
        }
        if (need) {
          l *= f;
          m_ref = m_new;
        }
      }
    }
    // (4) P_j = exp2(s - m_ref) into the P buffer, free once PV_{j-1} is done
    if (j >= 1 && !ptx::mbar_wait(bar_pv((j - 1) & 1), ((j - 1) >> 1) & 1)) ok = false;
    float rs = 0.f;
    const bool live = m_ref != -INFINITY;
#pragma unroll
    for (int c0 = 0; c0 < BKV; c0 += 32) {
      float v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float p = live ? fast_exp2(sv[c0 + i] - m_ref) : 0.f;  // masked keys: exp2(-inf) = 0
        v[i] = p;
        rs += p;
      }
      uint8_t* rowp = gbase + F_OFF_P + (c0 >> 6) * BOX + tid * 128;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int unit = ((c0 & 63) >> 3) + u;
        const uint4 w = make_uint4(pack2(v[8 * u], v[8 * u + 1]), pack2(v[8 * u + 2], v[8 * u + 3]),
                                   pack2(v[8 * u + 4], v[8 * u + 5]),
                                   pack2(v[8 * u + 6], v[8 * u + 7]));
        *reinterpret_cast<uint4*>(rowp + ((unit ^ (tid & 7)) << 4)) = w;
      }
    }
    l += rs;
    // (5) make P (and any rescaled O) visible to the tensor core; all threads decide together
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    ptx::tc_fence_before();
    if (__syncthreads_or(!ok)) {
      done_all = false;
      break;
    }
    if (tid == 0) {
      ok = ptx::mbar_wait(bar_v(j % F_VST), (j / F_VST) & 1);
      if (ok) {
        ptx::tc_fence_after();
        const uint32_t pt = base + F_OFF_P, vt = base + F_OFF_V + (j % F_VST) * TILE;
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          ptx::mma_bf16(t_o, kmajor_desc(pt, kk), mnmajor_desc(vt, kk), IDESC_PV,
                        (j > 0 || kk > 0) ? 1u : 0u);
        ptx::mma_commit(bar_pv(j & 1));
      }
    }
  }
  if (done_all && nkv >= 1) {
    const int j = nkv - 1;
    if (!ptx::mbar_wait(bar_pv(j & 1), (j >> 1) & 1)) ok = false;
    ptx::tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const bool store = ok && qi < a.S;
    uint4* orow = reinterpret_cast<uint4*>(a.o + (int64_t)(row0 + qi) * a.H + h * D);
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      float v[32];
      ptx::tmem_ld32(t_o + lane_off + c0, v);  // every lane: warp-collective
      if (store) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          orow[c0 / 8 + u] = make_uint4(pack2(v[8 * u] * inv, v[8 * u + 1] * inv),
                                        pack2(v[8 * u + 2] * inv, v[8 * u + 3] * inv),
                                        pack2(v[8 * u + 4] * inv, v[8 * u + 5] * inv),
                                        pack2(v[8 * u + 6] * inv, v[8 * u + 7] * inv));
      }
    }
    if (store) a.lse[(int64_t)h * a.M + row0 + qi] = (m_ref + log2f(l)) * 0.69314718055994531f;
  }
  if (!(done_all && ok)) atomicExch(&g_attn_error, 1);
  if (tid == 0) {
    // drain: issued MMAs complete and issued loads land before the CTA exits
    ptx::mma_commit(bar_drain);
    bool dr = ptx::mbar_wait(bar_drain, 0);
    for (int s = 0; s < F_KST; ++s)
      if ((k_issued >> s) & 1u) dr = ptx::mbar_wait(bar_k(s), (k_par >> s) & 1u) && dr;
    for (int s = 0; s < F_VST; ++s)
      if ((v_issued >> s) & 1u) dr = ptx::mbar_wait(bar_v(s), (v_par >> s) & 1u) && dr;
    dr = ptx::mbar_wait(bar_q, 0) && dr;
    if (!dr) atomicExch(&g_attn_error, 2);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  progress(0, 999);
}

// ---------------------------------------------------------------------------
// Backward.  With s = Q K^T / sqrt(d), P = exp(s - LSE), delta = rowsum(dO * O):
//   dP = dO V^T,  dS = P * (dP - delta),
//   dQ = dS K / sqrt(d),  dK = dS^T Q / sqrt(d),  dV = P^T dO.
// Two kernels own disjoint outputs, so there are no atomics:
//   dq kernel   one CTA per 128 queries, loops over key blocks (thread = query)
//   dkv kernel  one CTA per 128 keys, loops over 64-query blocks (thread = key)
// ---------------------------------------------------------------------------
struct BwdArgs {
  const float* lse;
  const float* delta;
  __nv_bfloat16* dqkv;
  int S, H, heads, M, causal;
  float scale_log2;  // log2(e) / sqrt(d)
  float scale;       // 1 / sqrt(d)
};

// dq kernel shared-memory map
constexpr int DQ_OFF_Q = 0, DQ_OFF_DO = TILE, DQ_OFF_K = 2 * TILE;
constexpr int DQ_OFF_V = DQ_OFF_K + KV_STAGES * TILE, DQ_OFF_DS = DQ_OFF_V + KV_STAGES * TILE;
constexpr int DQ_OFF_BAR = DQ_OFF_DS + TILE;
constexpr int DQ_NBAR = 1 + KV_STAGES + 1 + 1 + 1;  // q+dO, kv, s+dP, final, drain
constexpr int DQ_SMEM = DQ_OFF_BAR + 8 * DQ_NBAR + 16 + 1024;

__global__ void __launch_bounds__(NT, 1)
attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tdo,
                      const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + DQ_OFF_BAR;
  const uint32_t bar_qdo = bars;
  auto bar_kv = [&](int s) { return bars + 8u * (1 + s); };
  const uint32_t bar_sdp = bars + 8u * (1 + KV_STAGES);
  const uint32_t bar_fin = bars + 8u * (2 + KV_STAGES);
  const uint32_t bar_drain = bars + 8u * (3 + KV_STAGES);
  const uint32_t tslot = bars + 8u * DQ_NBAR;

  const int tid = threadIdx.x, warp = tid / 32;
  const int tile = gridDim.x - 1 - blockIdx.x;
  const int h = blockIdx.y, b = blockIdx.z;
  const int q0 = tile * BQ, row0 = b * a.S;
  const int nkv_all = (a.S + BKV - 1) / BKV;
  const int n = a.causal ? min(tile + 1, nkv_all) : nkv_all;
  const int col_q = h * D, col_k = a.H + h * D, col_v = 2 * a.H + h * D;

  if (tid == 0) {
    ptx::mbar_init(bar_qdo, 1);
    for (int s2 = 0; s2 < KV_STAGES; ++s2) ptx::mbar_init(bar_kv(s2), 1);
    ptx::mbar_init(bar_sdp, 1);
    ptx::mbar_init(bar_fin, 1);
    ptx::mbar_init(bar_drain, 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tq);
    ptx::prefetch_tmap(&tdo);
  }
  if (warp == 0) {
    ptx::tmem_alloc(tslot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + (tslot - base));
  const uint32_t t_s = tmem, t_dp = tmem + 128, t_dq = tmem + 256;
  progress(1, 2);
  pdl_wait();
  pdl_trigger();
  progress(1, 3);

  bool ok = true;
  uint32_t kv_issued = 0, kv_par = 0;
  auto load_kv = [&](int j) {
    const int st = j % KV_STAGES;
    ptx::mbar_arrive_expect_tx(bar_kv(st), 2 * TILE);
    const uint32_t kt = base + DQ_OFF_K + st * TILE, vt = base + DQ_OFF_V + st * TILE;
    const int r = row0 + j * BKV;
    ptx::tma_load_2d(kt, &tq, bar_kv(st), col_k, r);
    ptx::tma_load_2d(kt + BOX, &tq, bar_kv(st), col_k + 64, r);
    ptx::tma_load_2d(vt, &tq, bar_kv(st), col_v, r);
    ptx::tma_load_2d(vt + BOX, &tq, bar_kv(st), col_v + 64, r);
    kv_issued |= 1u << st;
    kv_par = (kv_par & ~(1u << st)) | ((uint32_t)((j / KV_STAGES) & 1) << st);
  };
  auto issue_sdp = [&](int j) {  // S = Q K_j^T, dP = dO V_j^T
    const uint32_t kt = base + DQ_OFF_K + (j % KV_STAGES) * TILE;
    const uint32_t vt = base + DQ_OFF_V + (j % KV_STAGES) * TILE;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      ptx::mma_bf16(t_s, kmajor_desc(base + DQ_OFF_Q, kk), kmajor_desc(kt, kk), IDESC_S, kk > 0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      ptx::mma_bf16(t_dp, kmajor_desc(base + DQ_OFF_DO, kk), kmajor_desc(vt, kk), IDESC_S, kk > 0);
    ptx::mma_commit(bar_sdp);
  };

  if (tid == 0) {
    ptx::mbar_arrive_expect_tx(bar_qdo, 2 * TILE);
    ptx::tma_load_2d(base + DQ_OFF_Q, &tq, bar_qdo, col_q, row0 + q0);
    ptx::tma_load_2d(base + DQ_OFF_Q + BOX, &tq, bar_qdo, col_q + 64, row0 + q0);
    ptx::tma_load_2d(base + DQ_OFF_DO, &tdo, bar_qdo, h * D, row0 + q0);
    ptx::tma_load_2d(base + DQ_OFF_DO + BOX, &tdo, bar_qdo, h * D + 64, row0 + q0);
    for (int j = 0; j < KV_STAGES && j < n; ++j) load_kv(j);
    progress(1, 4);
    ok = ptx::mbar_wait(bar_qdo, 0);
    if (!ok) wait_failed(101);
    ok = ok && ptx::mbar_wait(bar_kv(0), 0);
    if (!ok) wait_failed(102);
    if (ok) {
      ptx::tc_fence_after();
      issue_sdp(0);
    }
    progress(1, 5);
  }

  const int qi = q0 + tid;
  const bool valid_q = qi < a.S;
  const float lse2 = valid_q ? a.lse[(int64_t)h * a.M + row0 + qi] * 1.4426950408889634f : 0.f;
  const float dlt = valid_q ? a.delta[(int64_t)h * a.M + row0 + qi] : 0.f;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  bool done_all = true;

  for (int j = 0; j < n; ++j) {
    // (a) S_j, dP_j ready; dQ_{j-1} (issued before them) is complete too, so
    //     the dS buffer and K/V stage (j-1) % 2 are free
    progress(1, 10 + 10 * j);
    if (!ptx::mbar_wait(bar_sdp, j & 1)) {
      ok = false;
      wait_failed(103);
    }
    ptx::tc_fence_after();
    progress(1, 11 + 10 * j);
    if (tid == 0 && ok && j + 1 < n && j + 1 >= KV_STAGES) load_kv(j + 1);
    // (b) dS = P * (dP - delta) into the swizzled dS buffer
    const int kbase = j * BKV;
#pragma unroll 1
    for (int c0 = 0; c0 < BKV; c0 += 32) {
      float v[32], w[32];
      ptx::tmem_ld32(t_s + lane_off + c0, v);
      ptx::tmem_ld32(t_dp + lane_off + c0, w);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int key = kbase + c0 + i;
        const bool valid = valid_q && key < a.S && (!a.causal || key <= qi);
        const float p = valid ? fast_exp2(v[i] * a.scale_log2 - lse2) : 0.f;
        v[i] = p * (w[i] - dlt);
      }
      uint8_t* rowp = gbase + DQ_OFF_DS + (c0 >> 6) * BOX + tid * 128;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int unit = ((c0 & 63) >> 3) + u;
        *reinterpret_cast<uint4*>(rowp + ((unit ^ (tid & 7)) << 4)) =
            make_uint4(pack2(v[8 * u], v[8 * u + 1]), pack2(v[8 * u + 2], v[8 * u + 3]),
                       pack2(v[8 * u + 4], v[8 * u + 5]), pack2(v[8 * u + 6], v[8 * u + 7]));
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    ptx::tc_fence_before();
    if (__syncthreads_or(!ok)) {
      done_all = false;
      break;
    }
    // (d) dQ += dS K_j; then S_{j+1}, dP_{j+1}
    progress(1, 12 + 10 * j);
    if (tid == 0) {
      ptx::tc_fence_after();
      const uint32_t kt = base + DQ_OFF_K + (j % KV_STAGES) * TILE;
#pragma unroll
      for (int kk = 0; kk < BKV / 16; ++kk)
        ptx::mma_bf16(t_dq, kmajor_desc(base + DQ_OFF_DS, kk), mnmajor_desc(kt, kk), IDESC_PV,
                      (j > 0 || kk > 0) ? 1u : 0u);
      if (j + 1 < n) {
        ok = ptx::mbar_wait(bar_kv((j + 1) % KV_STAGES), ((j + 1) / KV_STAGES) & 1);
        if (!ok) wait_failed(104);
        if (ok) issue_sdp(j + 1);
      }
    }
  }
  progress(1, 900);
  if (tid == 0) ptx::mma_commit(bar_fin);
  if (!ptx::mbar_wait(bar_fin, 0)) {
    ok = false;
    wait_failed(105);
  }
  ptx::tc_fence_after();
  progress(1, 950);
  // tcgen05.ld is warp-collective: every thread loads, only valid rows store.
  if (done_all && n > 0) {
    const bool store = ok && valid_q;
    uint4* out = reinterpret_cast<uint4*>(a.dqkv + (int64_t)(row0 + qi) * 3 * a.H + h * D);
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      float v[32];
      ptx::tmem_ld32(t_dq + lane_off + c0, v);
      if (store) {
#pragma unroll
        for (int u = 0; u < 4; ++u)
          out[c0 / 8 + u] = make_uint4(
              pack2(v[8 * u] * a.scale, v[8 * u + 1] * a.scale),
              pack2(v[8 * u + 2] * a.scale, v[8 * u + 3] * a.scale),
              pack2(v[8 * u + 4] * a.scale, v[8 * u + 5] * a.scale),
              pack2(v[8 * u + 6] * a.scale, v[8 * u + 7] * a.scale));
      }
    }
  }
  if (!(done_all && ok)) atomicExch(&g_attn_error, 3);
  if (tid == 0) {
    ptx::mma_commit(bar_drain);
    bool dr = ptx::mbar_wait(bar_drain, 0);
    for (int s2 = 0; s2 < KV_STAGES; ++s2)
      if ((kv_issued >> s2) & 1u) dr = ptx::mbar_wait(bar_kv(s2), (kv_par >> s2) & 1u) && dr;
    dr = ptx::mbar_wait(bar_qdo, 0) && dr;
    if (!dr) wait_failed(106);
  }
  progress(1, 990);
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  progress(1, 999);
}

// dkv kernel: 64-query blocks stored as two 64x64 boxes.
constexpr int QB = 64;
constexpr int BOX64 = 64 * 64 * 2;   // 8 KB
constexpr int QTILE = 2 * BOX64;     // 64 rows x 128 dims
constexpr int KV_OFF_K = 0, KV_OFF_V = TILE, KV_OFF_ST = 2 * TILE;  // stages: Q then dO
constexpr int KV_STAGE = 2 * QTILE;
constexpr int KV_OFF_PT = KV_OFF_ST + KV_STAGES * KV_STAGE;
constexpr int KV_OFF_DST = KV_OFF_PT + 128 * QB * 2;
constexpr int KV_OFF_STAT = KV_OFF_DST + 128 * QB * 2;  // lse2 / delta, [2][2][QB] floats
constexpr int KV_OFF_BAR = KV_OFF_STAT + 4 * QB * 4;
constexpr int KV_NBAR = 1 + KV_STAGES + 1 + 1 + 1;  // K+V, q+dO stages, st+dpt, final, drain
constexpr int KV_SMEM = KV_OFF_BAR + 8 * KV_NBAR + 16 + 1024;
// S^T = K Q^T: M = 128 keys, N = 64 queries, both K-major (over d).
constexpr uint32_t IDESC_ST = ptx::idesc_bf16_f32(128, QB, false, false);
// dV = P^T dO, dK = dS^T Q: M = 128 keys, N = 128 dims; A K-major (over queries), B MN-major.
constexpr uint32_t IDESC_DKV = ptx::idesc_bf16_f32(128, D, false, true);

__device__ __forceinline__ uint64_t kmajor64_desc(uint32_t tile, int kk) {  // [64 rows][128 cols]
  return ptx::smem_desc_sw128(tile + (kk >> 2) * BOX64 + (kk & 3) * 32, 16, 1024);
}
__device__ __forceinline__ uint64_t mnmajor64_desc(uint32_t tile, int kk) {  // [64 k][128 n]
  return ptx::smem_desc_sw128(tile + kk * 2048, BOX64, 1024);
}

__global__ void __launch_bounds__(NT, 1)
attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tkv, const __grid_constant__ CUtensorMap tq64,
                       const __grid_constant__ CUtensorMap tdo64, const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + KV_OFF_BAR;
  const uint32_t bar_kv = bars;
  auto bar_qd = [&](int s) { return bars + 8u * (1 + s); };
  const uint32_t bar_st = bars + 8u * (1 + KV_STAGES);
  const uint32_t bar_fin = bars + 8u * (2 + KV_STAGES);
  const uint32_t bar_drain = bars + 8u * (3 + KV_STAGES);
  const uint32_t tslot = bars + 8u * KV_NBAR;
  float* stat = reinterpret_cast<float*>(gbase + KV_OFF_STAT);  // [buf][lse2 | delta][QB]

  const int tid = threadIdx.x, warp = tid / 32;
  const int ktile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int k0 = ktile * 128, row0 = b * a.S;
  const int nq_all = (a.S + QB - 1) / QB;
  const int i0 = a.causal ? k0 / QB : 0;
  const int n = nq_all - i0;
  const int col_q = h * D, col_k = a.H + h * D, col_v = 2 * a.H + h * D;

  if (tid == 0) {
    ptx::mbar_init(bar_kv, 1);
    for (int s2 = 0; s2 < KV_STAGES; ++s2) ptx::mbar_init(bar_qd(s2), 1);
    ptx::mbar_init(bar_st, 1);
    ptx::mbar_init(bar_fin, 1);
    ptx::mbar_init(bar_drain, 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tkv);
    ptx::prefetch_tmap(&tq64);
    ptx::prefetch_tmap(&tdo64);
  }
  if (warp == 0) {
    ptx::tmem_alloc(tslot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + (tslot - base));
  const uint32_t t_st = tmem, t_dpt = tmem + 64, t_dv = tmem + 128, t_dk = tmem + 256;
  progress(2, 2);
  pdl_wait();
  pdl_trigger();
  progress(2, 3);

  bool ok = true;
  uint32_t qd_issued = 0, qd_par = 0;
  auto load_qd = [&](int ii) {  // query block i0 + ii into stage ii % 2
    const int st = ii % KV_STAGES;
    const uint32_t qt = base + KV_OFF_ST + st * KV_STAGE, dt = qt + QTILE;
    const int r = row0 + (i0 + ii) * QB;
    ptx::mbar_arrive_expect_tx(bar_qd(st), KV_STAGE);
    ptx::tma_load_2d(qt, &tq64, bar_qd(st), col_q, r);
    ptx::tma_load_2d(qt + BOX64, &tq64, bar_qd(st), col_q + 64, r);
    ptx::tma_load_2d(dt, &tdo64, bar_qd(st), h * D, r);
    ptx::tma_load_2d(dt + BOX64, &tdo64, bar_qd(st), h * D + 64, r);
    qd_issued |= 1u << st;
    qd_par = (qd_par & ~(1u << st)) | ((uint32_t)((ii / KV_STAGES) & 1) << st);
  };
  auto issue_st = [&](int ii) {  // S^T = K Q_i^T, dP^T = V dO_i^T
    const uint32_t qt = base + KV_OFF_ST + (ii % KV_STAGES) * KV_STAGE, dt = qt + QTILE;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      ptx::mma_bf16(t_st, kmajor_desc(base + KV_OFF_K, kk), kmajor64_desc(qt, kk), IDESC_ST, kk > 0);
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk)
      ptx::mma_bf16(t_dpt, kmajor_desc(base + KV_OFF_V, kk), kmajor64_desc(dt, kk), IDESC_ST, kk > 0);
    ptx::mma_commit(bar_st);
  };

  if (tid == 0) {
    ptx::mbar_arrive_expect_tx(bar_kv, 2 * TILE);
    ptx::tma_load_2d(base + KV_OFF_K, &tkv, bar_kv, col_k, row0 + k0);
    ptx::tma_load_2d(base + KV_OFF_K + BOX, &tkv, bar_kv, col_k + 64, row0 + k0);
    ptx::tma_load_2d(base + KV_OFF_V, &tkv, bar_kv, col_v, row0 + k0);
    ptx::tma_load_2d(base + KV_OFF_V + BOX, &tkv, bar_kv, col_v + 64, row0 + k0);
    for (int ii = 0; ii < KV_STAGES && ii < n; ++ii) load_qd(ii);
    progress(2, 4);
    ok = ptx::mbar_wait(bar_kv, 0);
    if (!ok) wait_failed(201);
    ok = ok && (n <= 0 || ptx::mbar_wait(bar_qd(0), 0));
    if (!ok) wait_failed(202);
    if (ok && n > 0) {
      ptx::tc_fence_after();
      issue_st(0);
    }
    progress(2, 5);
  }

  const int kj = k0 + tid;
  const bool valid_k = kj < a.S;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  bool done_all = true;

  for (int ii = 0; ii < n; ++ii) {
    const int i = i0 + ii;
    float* lse_s = stat + (ii & 1) * 2 * QB;
    float* dl_s = lse_s + QB;
    if (tid < QB) {
      const int q = i * QB + tid;
      lse_s[tid] = q < a.S ? a.lse[(int64_t)h * a.M + row0 + q] * 1.4426950408889634f : 0.f;
      dl_s[tid] = q < a.S ? a.delta[(int64_t)h * a.M + row0 + q] : 0.f;
    }
    __syncthreads();
    // (a) S^T, dP^T of block i ready; dK/dV MMAs of block i-1 are complete, so
    //     P^T / dS^T buffers and stage (ii-1) % 2 are free
    progress(2, 10 + 10 * ii);
    if (!ptx::mbar_wait(bar_st, ii & 1)) {
      ok = false;
      wait_failed(203);
    }
    ptx::tc_fence_after();
    progress(2, 11 + 10 * ii);
    if (tid == 0 && ok && ii + 1 < n && ii + 1 >= KV_STAGES) load_qd(ii + 1);
    // (b) P^T and dS^T rows of this key
#pragma unroll
    for (int c0 = 0; c0 < QB; c0 += 32) {
      float v[32], w[32];
      ptx::tmem_ld32(t_st + lane_off + c0, v);
      ptx::tmem_ld32(t_dpt + lane_off + c0, w);
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        const int q = i * QB + c0 + c;
        const bool valid = valid_k && q < a.S && (!a.causal || kj <= q);
        const float p = valid ? fast_exp2(v[c] * a.scale_log2 - lse_s[c0 + c]) : 0.f;
        v[c] = p;
        w[c] = p * (w[c] - dl_s[c0 + c]);
      }
      uint8_t* prow = gbase + KV_OFF_PT + tid * 128;
      uint8_t* drow = gbase + KV_OFF_DST + tid * 128;
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int unit = (c0 >> 3) + u;
        const int off = (unit ^ (tid & 7)) << 4;
        *reinterpret_cast<uint4*>(prow + off) =
            make_uint4(pack2(v[8 * u], v[8 * u + 1]), pack2(v[8 * u + 2], v[8 * u + 3]),
                       pack2(v[8 * u + 4], v[8 * u + 5]), pack2(v[8 * u + 6], v[8 * u + 7]));
        *reinterpret_cast<uint4*>(drow + off) =
            make_uint4(pack2(w[8 * u], w[8 * u + 1]), pack2(w[8 * u + 2], w[8 * u + 3]),
                       pack2(w[8 * u + 4], w[8 * u + 5]), pack2(w[8 * u + 6], w[8 * u + 7]));
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    ptx::tc_fence_before();
    if (__syncthreads_or(!ok)) {
      done_all = false;
      break;
    }
    // (d) dV += P^T dO_i, dK += dS^T Q_i; then the next block's S^T, dP^T
    progress(2, 12 + 10 * ii);
    if (tid == 0) {
      ptx::tc_fence_after();
      const uint32_t qt = base + KV_OFF_ST + (ii % KV_STAGES) * KV_STAGE, dt = qt + QTILE;
#pragma unroll
      for (int kk = 0; kk < QB / 16; ++kk) {
        const uint32_t acc = (ii > 0 || kk > 0) ? 1u : 0u;
        ptx::mma_bf16(t_dv, ptx::smem_desc_sw128(base + KV_OFF_PT + kk * 32, 16, 1024),
                      mnmajor64_desc(dt, kk), IDESC_DKV, acc);
        ptx::mma_bf16(t_dk, ptx::smem_desc_sw128(base + KV_OFF_DST + kk * 32, 16, 1024),
                      mnmajor64_desc(qt, kk), IDESC_DKV, acc);
      }
      if (ii + 1 < n) {
        ok = ptx::mbar_wait(bar_qd((ii + 1) % KV_STAGES), ((ii + 1) / KV_STAGES) & 1);
        if (!ok) wait_failed(204);
        if (ok) issue_st(ii + 1);
      }
    }
  }
  progress(2, 900);
  if (tid == 0) ptx::mma_commit(bar_fin);
  if (!ptx::mbar_wait(bar_fin, 0)) {
    ok = false;
    wait_failed(205);
  }
  ptx::tc_fence_after();
  progress(2, 950);
  // tcgen05.ld is warp-collective: every thread loads, only valid rows store.
  if (done_all) {
    const bool store = ok && valid_k;
    __nv_bfloat16* rowp = a.dqkv + (int64_t)(row0 + kj) * 3 * a.H;
    uint4* dk_out = reinterpret_cast<uint4*>(rowp + a.H + h * D);
    uint4* dv_out = reinterpret_cast<uint4*>(rowp + 2 * a.H + h * D);
#pragma unroll
    for (int c0 = 0; c0 < D; c0 += 32) {
      float v[32], w[32];
      ptx::tmem_ld32(t_dk + lane_off + c0, v);
      ptx::tmem_ld32(t_dv + lane_off + c0, w);
      if (store) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          dk_out[c0 / 8 + u] = make_uint4(pack2(v[8 * u] * a.scale, v[8 * u + 1] * a.scale),
                                          pack2(v[8 * u + 2] * a.scale, v[8 * u + 3] * a.scale),
                                          pack2(v[8 * u + 4] * a.scale, v[8 * u + 5] * a.scale),
                                          pack2(v[8 * u + 6] * a.scale, v[8 * u + 7] * a.scale));
          dv_out[c0 / 8 + u] = make_uint4(pack2(w[8 * u], w[8 * u + 1]), pack2(w[8 * u + 2], w[8 * u + 3]),
                                          pack2(w[8 * u + 4], w[8 * u + 5]), pack2(w[8 * u + 6], w[8 * u + 7]));
        }
      }
    }
  }
  if (!(done_all && ok)) atomicExch(&g_attn_error, 5);
  if (tid == 0) {
    ptx::mma_commit(bar_drain);
    bool dr = ptx::mbar_wait(bar_drain, 0);
    for (int s2 = 0; s2 < KV_STAGES; ++s2)
      if ((qd_issued >> s2) & 1u) dr = ptx::mbar_wait(bar_qd(s2), (qd_par >> s2) & 1u) && dr;
    dr = ptx::mbar_wait(bar_kv, 0) && dr;
    if (!dr) wait_failed(206);
  }
  progress(2, 990);
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  progress(2, 999);
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

// Tensor map over a row-major bf16 [rows, cols] matrix (leading dimension ld
// elements), box box_rows x 64 columns, 128-byte swizzle, zero fill outside.
bool map2d(CUtensorMap* m, const void* p, int cols, int rows, int64_t ld, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

bool qkv_map(CUtensorMap* m, const void* qkv, int M, int H) {
  return map2d(m, qkv, 3 * H, M, 3 * (int64_t)H, 128);
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

cudaError_t attention_delta(const AttnArgs& a, cudaStream_t st);

cudaError_t attention_bwd_tc(const AttnArgs& a, cudaStream_t st) {
  if (!attention_tc_supported(a) || ((uintptr_t)a.d_o | (uintptr_t)a.dqkv) & 15)
    return cudaErrorNotSupported;
  if (a.batch == 0 || a.seq == 0) return cudaSuccess;
  const int M = a.batch * a.seq;
  CUtensorMap tq128, tq64, tdo128, tdo64;
  if (!map2d(&tq128, a.qkv, 3 * a.hidden, M, 3 * (int64_t)a.hidden, 128) ||
      !map2d(&tq64, a.qkv, 3 * a.hidden, M, 3 * (int64_t)a.hidden, 64) ||
      !map2d(&tdo128, a.d_o, a.hidden, M, a.hidden, 128) ||
      !map2d(&tdo64, a.d_o, a.hidden, M, a.hidden, 64))
    return cudaErrorInvalidValue;
  static bool attr = false;
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, DQ_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(attn_bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             KV_SMEM);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  cudaError_t e = attention_delta(a, st);
  if (e != cudaSuccess) return e;
  BwdArgs ba;
  ba.lse = a.lse;
  ba.delta = a.delta;
  ba.dqkv = static_cast<__nv_bfloat16*>(a.dqkv);
  ba.S = a.seq;
  ba.H = a.hidden;
  ba.heads = a.heads;
  ba.M = M;
  ba.causal = a.causal ? 1 : 0;
  ba.scale = 1.f / sqrtf((float)a.head_dim);
  ba.scale_log2 = 1.4426950408889634f * ba.scale;
  const int tiles = (a.seq + 127) / 128;
  e = launch_pdl(attn_bwd_dq_tc_kernel, dim3(tiles, a.heads, a.batch), dim3(NT), DQ_SMEM, st,
                 tq128, tdo128, ba);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_bwd_dkv_tc_kernel, dim3(tiles, a.heads, a.batch), dim3(NT), KV_SMEM, st,
                    tq128, tq64, tdo64, ba);
}

cudaError_t attention_set_progress(int* p) {
  return cudaMemcpyToSymbol(g_attn_progress, &p, sizeof(p));
}

int attention_read_and_clear_error() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_attn_error, &z, sizeof(int));
  return v;
}

}  // namespace oases
