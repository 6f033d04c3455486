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
#include <queue>
#include <vector>

#include "common.cuh"
#include "sm100_ptx.cuh"

namespace oases {

__device__ int g_attn_error;
// Optional progress markers (debugging aid, off when null): thread 0 of CTA c
// of kernel k writes its current stage to g_attn_progress[k * 256 + c].
__device__ int* g_attn_progress;
// Optional timeline of the backward kernels (debugging aid, off when null),
// %globaltimer stamps: entry and exit of every CTA (dq kernel at
// [2 c], dK/dV kernel at [8192 + 2 c], c = linear CTA index < 4096), and per
// block j < 64 of CTA 0 (dq at 16384 + 4 j, dK/dV at 16640 + 4 j): [0] S, dP
// MMAs issued, [1] accumulation MMAs issued, [2] compute warp 2 saw S, dP,
// [3] compute warp 2 handed over its dS (and P) rows.
__device__ unsigned long long* g_attn_timeline;

namespace {

constexpr int D = 128;                 // head dimension
constexpr int BQ = 128, BKV = 128;     // query rows per CTA, keys per block
constexpr int BOX = 128 * 64 * 2;      // one TMA box: 128 rows x 64 bf16 (16 KB)
constexpr int TILE = 2 * BOX;          // 128 rows x 128 bf16 (32 KB)

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

// Shared-memory descriptors are formed once per tile and stepped per MMA: the
// start-address field (bits 0..13) holds the address in 16-byte units, and
// every shared address here is below 2^18, so adding byte offset d as d >> 4
// cannot carry out of the field.  (Forming each descriptor from scratch cost
// more issue time in the single MMA thread than the MMA itself takes.)
__device__ __forceinline__ uint64_t desc_step(uint64_t base_desc, uint32_t byte_off) {
  return base_desc + (uint64_t)(byte_off >> 4);
}
// Descriptor of a K-major operand tile [128 rows][128 cols] stored as two
// 128-byte-swizzled 64-column boxes, for k-step kk (16 columns) of 8.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t tile, int kk) {
  return desc_step(ptx::smem_desc_sw128(tile, 16, 1024), (kk >> 2) * BOX + (kk & 3) * 32);
}
// Descriptor of an MN-major operand [128 k-rows][128 n-cols] stored as two
// boxes of 64 n-columns, for k-step kk (16 k-rows) of 8.
__device__ __forceinline__ uint64_t mnmajor_desc(uint32_t tile, int kk) {
  return desc_step(ptx::smem_desc_sw128(tile, BOX, 1024), kk * 2048);
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
__device__ __forceinline__ int linear_cta() {
  return blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
}
// kid 1 = dq (c = work item of the persistent kernel; what 0 = its first
// MMAs issued, 1 = its dQ stored), 2 = dK/dV (c = CTA; 0 = entry, 1 = exit)
__device__ __forceinline__ void tl_unit(int kid, int c, int what) {
  unsigned long long* t = g_attn_timeline;
  if (t != nullptr && c < 4096) t[(kid - 1) * 8192 + 2 * c + what] = ptx::globaltimer();
}
__device__ __forceinline__ void tl_cta(int kid, int what) { tl_unit(kid, linear_cta(), what); }
__device__ __forceinline__ void tl_block(int kid, int j, int what) {
  unsigned long long* t = g_attn_timeline;
  if (t != nullptr && linear_cta() == 0 && j < 64)
    t[16384 + (kid - 1) * 256 + 4 * j + what] = ptx::globaltimer();
}
// Forward, CTA 0, tile t, key block j < 64: [0] S_t(j) issued, [1] the
// softmax warp of lane quarter 2 saw S_t(j), [2 + q] the warp of lane quarter
// q published P_t(j), [6] PV_t(j) issued, [7] PV_t(j) about to be issued (its
// P and V ready).
__device__ __forceinline__ void tl_fwd(int t, int j, int what) {
  unsigned long long* tb = g_attn_timeline;
  if (tb != nullptr && linear_cta() == 0 && j < 64) tb[16896 + 8 * (64 * t + j) + what] = ptx::globaltimer();
}
// Records the first failed wait site (kernel * 100 + site) in g_attn_error.
__device__ __forceinline__ void wait_failed(int code) { atomicCAS(&g_attn_error, 0, code); }

// A work-item schedule for the persistent forward, computed on the host
// (longest items first, each to the CTA with the least work so far): CTA c
// runs order[start[c]] .. order[start[c + 1] - 1] in that order.
constexpr int FWD_SCHED_ITEMS = 2048, FWD_SCHED_CTAS = 256;
struct FwdSched {
  uint16_t start[FWD_SCHED_CTAS + 1];
  uint16_t order[FWD_SCHED_ITEMS];
};

struct FwdArgs {
  __nv_bfloat16* o;
  float* lse;
  int S, H, heads, M;  // sequence length, hidden, heads, rows of this call
  int causal;
  float scale_log2;    // log2(e) / sqrt(d)
  int batch, pairs;    // sequences; pairs of 128-query tiles per sequence
  int items;           // batch * heads * pairs
  int use_sched;       // 1: sched holds the item order; 0: the snake order
  FwdSched sched;
};

// Forward: a persistent kernel, one CTA per SM.  A work item is 256 queries
// of one (sequence, head): two tiles of 128 queries that share every K/V
// block.  Items are numbered heaviest first (the causal pairs nearest the end
// of the sequence have the most key blocks); the host assigns them longest
// first, each to the CTA with the least work so far, and passes the order in
// the kernel's parameters (for more than 2048 items or 256 CTAs, CTA c of G
// takes items c, 2G - 1 - c, 2G + c, ...: a snake over rounds of G).  320
// threads:
//   warp 0      TMA loads, in the order the MMAs consume them: per item Q_0,
//               then K_j and V_j into two-stage rings that run on across
//               items, Q_1 after the first block; a tile's Q buffer is
//               refilled for the next item as soon as the tile's last S MMA
//               of this item has read it;
//   warp 1      TMEM allocation (512 columns, once); one thread issues the
//               MMAs;
//   warps 2..5  softmax of tile 0, warps 6..9 softmax of tile 1: thread r
//               (TMEM lane r of its warp's quarter) owns one query row.
// TMEM: S_t (then P_t) in columns 128 t .. +127, O_t in 256 + 128 t .. +127.
// Per tile t and key block j:
//   S_t = Q_t K_j^T                 tcgen05.mma, A and B from shared memory
//   P_t = exp2(s - m)               the softmax threads read S_t, keep the row
//                                   maximum m and sum l in registers, and write
//                                   P_t back over the first 64 columns of S_t
//                                   as packed bf16
//   O_t += P_t V_j                  tcgen05.mma, A = P_t from tensor memory,
//                                   B = V_j (MN-major) from shared memory
// The MMA thread issues, per block, PV_0(j), S_0(j+1), PV_1(j), S_1(j+1): while
// one tile's softmax threads turn S into P, the tensor core works on the other
// tile.  S_t(j+1) overwrites P_t(j); it is issued after PV_t(j), and MMAs of
// one thread run in issue order.  The completion of S_t(j) therefore also
// means PV_t(j-1) is complete, so the softmax threads may rescale their O row
// in place before publishing P_t(j).  A row's reference maximum is raised only
// when the running maximum exceeds it by more than 2^8 (RESCALE_LOG2), so P
// stays <= 256 and O is rescaled rarely.  Key blocks past the diagonal are
// skipped; keys past the diagonal inside it (and past the sequence end) get
// weight 0.  LSE = m + log(l) per (head, row) for the backward.
// Across items: once the round that issues tile t's last PV of an item is
// done, the MMA thread issues S_t(0) of the next item, so a tile whose item
// ends a block early (the lower tile of a causal pair) starts the next item
// while the other tile finishes its diagonal block, and its softmax warps
// store O of the finished item meanwhile.  The next item's first PV_t, which
// overwrites O_t, waits for P_t(0), which those warps publish only after
// they have read O_t out.
constexpr int F_NT = 320;
constexpr int F_KST = 2, F_VST = 2;
constexpr int F_OFF_Q = 0, F_OFF_K = 2 * TILE, F_OFF_V = F_OFF_K + F_KST * TILE;
constexpr int F_OFF_EPI = F_OFF_V + F_VST * TILE;  // O staging: 4 KB per softmax warp
constexpr int F_OFF_BAR = F_OFF_EPI + 8 * 4096;
// q_full[2], q_empty[2], k_full[2], k_empty[2], v_full[2], v_empty[2],
// s_full[2], p_full[2], o_full[2], drain
constexpr int F_NBAR = 4 + 2 * F_KST + 2 * F_VST + 6 + 1;
constexpr int FWD_SMEM = F_OFF_BAR + 8 * F_NBAR + 16 + 1024;
static_assert(FWD_SMEM <= 232448, "attention forward: more than 227 KB of shared memory");
constexpr float RESCALE_LOG2 = 8.f;

// Item k of CTA c (of G) in a persistent kernel whose items are numbered
// heaviest first: rounds of G items, in snake order.
__device__ __forceinline__ int persistent_item(int k, int c, int G) {
  return k * G + ((k & 1) ? G - 1 - c : c);
}
// Item k of CTA c (of G) of the forward: the host's schedule, else the snake.
__device__ __forceinline__ int fwd_item_at(const FwdArgs& a, int k, int c, int G) {
  if (!a.use_sched) return persistent_item(k, c, G);
  const int s0 = a.sched.start[c], s1 = a.sched.start[c + 1];
  return k < s1 - s0 ? (int)a.sched.order[s0 + k] : a.items;
}

struct FwdItem {
  int h, b, q0;  // head, sequence, first query of the pair
  int n0, n1;    // key blocks of each tile (0: the tile lies past the sequence end)
};
__device__ __forceinline__ FwdItem fwd_item(const FwdArgs& a, int i) {
  const int bh = a.heads * a.batch;
  FwdItem it;
  const int pair = a.pairs - 1 - i / bh, r = i % bh;
  it.h = r % a.heads;
  it.b = r / a.heads;
  it.q0 = pair * 2 * BQ;
  const int nkv_all = (a.S + BKV - 1) / BKV;
  const int q1 = it.q0 + BQ;
  it.n0 = a.causal ? min(it.q0 / BKV + 1, nkv_all) : nkv_all;  // q0 < S: the pair exists
  it.n1 = q1 >= a.S ? 0 : (a.causal ? min(q1 / BKV + 1, nkv_all) : nkv_all);
  return it;
}
// Forward, every item i < 4096 (256 queries of one sequence and head): eight
// stamps at [17920 + 8i]: [0] its CTA's entry, [1] its CTA set up, [2] Q_0 and
// K_0 of the item landed (MMA thread), [3] tile 0's softmax saw S_0(0), [4]
// tile 0's and [5] tile 1's last PV complete, [6] tile 1's O stored, [7] its
// CTA's exit.
__device__ __forceinline__ void tl_fitem(int i, int what) {
  unsigned long long* tb = g_attn_timeline;
  if (tb != nullptr && i < 4096) tb[17920 + 8 * i + what] = ptx::globaltimer();
}
__device__ __forceinline__ void tl_fitems(const FwdArgs& a, int c, int G, int what) {
  const int items = a.items;
  unsigned long long* tb = g_attn_timeline;
  if (tb == nullptr) return;
  const unsigned long long now = ptx::globaltimer();
  // CTA 0's globaltimer and SM clock at entry (what 0) and exit (what 7) at
  // [50688 + 0..3]: the two deltas give the SM clock rate over the launch
  if (c == 0 && (what == 0 || what == 7)) {
    tb[50688 + (what ? 2 : 0)] = now;
    tb[50689 + (what ? 2 : 0)] = (unsigned long long)clock64();
  }
  for (int k = 0;; ++k) {
    const int i = fwd_item_at(a, k, c, G);
    if (i >= items) break;
    if (i < 4096) tb[17920 + 8 * i + what] = now;
  }
}

__global__ void __launch_bounds__(F_NT, 1)
attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm, const __grid_constant__ FwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + F_OFF_BAR;
  auto q_full = [&](int t) { return bars + 8u * t; };
  auto q_empty = [&](int t) { return bars + 8u * (2 + t); };
  auto k_full = [&](int s) { return bars + 8u * (4 + s); };
  auto k_empty = [&](int s) { return bars + 8u * (4 + F_KST + s); };
  auto v_full = [&](int s) { return bars + 8u * (4 + 2 * F_KST + s); };
  auto v_empty = [&](int s) { return bars + 8u * (4 + 2 * F_KST + F_VST + s); };
  auto s_full = [&](int t) { return bars + 8u * (4 + 2 * F_KST + 2 * F_VST + t); };
  auto p_full = [&](int t) { return bars + 8u * (6 + 2 * F_KST + 2 * F_VST + t); };
  auto o_full = [&](int t) { return bars + 8u * (8 + 2 * F_KST + 2 * F_VST + t); };
  const uint32_t bar_drain = bars + 8u * (10 + 2 * F_KST + 2 * F_VST);
  const uint32_t tslot = bars + 8u * F_NBAR;

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int cta = blockIdx.x, G = gridDim.x;
  if (tid == 0) tl_fitems(a, cta, G, 0);

  if (tid == 0) {
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(q_full(t), 1);
      ptx::mbar_init(q_empty(t), 1);
    }
    for (int s = 0; s < F_KST; ++s) {
      ptx::mbar_init(k_full(s), 1);
      ptx::mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < F_VST; ++s) {
      ptx::mbar_init(v_full(s), 1);
      ptx::mbar_init(v_empty(s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(s_full(t), 1);
      ptx::mbar_init(p_full(t), 4);  // one arrival per softmax warp of the tile
      ptx::mbar_init(o_full(t), 1);
    }
    ptx::mbar_init(bar_drain, 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tm);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tslot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + (tslot - base));
  progress(0, 2);
  if (tid == 0) tl_fitems(a, cta, G, 1);
  pdl_wait();
  pdl_trigger();
  progress(0, 3);
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      // ring entries loaded so far (entry e sits in stage e % depth), Q loads per tile
      uint32_t ke = 0, ve = 0, qn[2] = {0u, 0u};
      auto load_q = [&](const FwdItem& it, int t) {
        if (qn[t] > 0 && !ptx::mbar_wait(q_empty(t), (qn[t] - 1) & 1)) {
          wait_failed(10);
          return false;
        }
        ptx::mbar_arrive_expect_tx(q_full(t), TILE);
        const uint32_t qt = base + F_OFF_Q + t * TILE;
        const int r = it.b * a.S + it.q0 + t * BQ;
        ptx::tma_load_2d(qt, &tm, q_full(t), it.h * D, r);
        ptx::tma_load_2d(qt + BOX, &tm, q_full(t), it.h * D + 64, r);
        ++qn[t];
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int i = fwd_item_at(a, k, cta, G);
        if (i >= a.items) break;
        const FwdItem it = fwd_item(a, i);
        const int nmax = max(it.n0, it.n1);
        const int col_k = a.H + it.h * D, col_v = 2 * a.H + it.h * D;
        ok = load_q(it, 0);
        for (int j = 0; j < nmax && ok; ++j) {
          const int r = it.b * a.S + j * BKV;
          const uint32_t s = ke % F_KST, u = ke / F_KST;
          if (u > 0 && !ptx::mbar_wait(k_empty(s), (u - 1) & 1)) {
            ok = false;
            wait_failed(11);
            break;
          }
          ptx::mbar_arrive_expect_tx(k_full(s), TILE);
          const uint32_t kt = base + F_OFF_K + s * TILE;
          ptx::tma_load_2d(kt, &tm, k_full(s), col_k, r);
          ptx::tma_load_2d(kt + BOX, &tm, k_full(s), col_k + 64, r);
          ++ke;
          const uint32_t sv = ve % F_VST, uv = ve / F_VST;
          if (uv > 0 && !ptx::mbar_wait(v_empty(sv), (uv - 1) & 1)) {
            ok = false;
            wait_failed(12);
            break;
          }
          ptx::mbar_arrive_expect_tx(v_full(sv), TILE);
          const uint32_t vt = base + F_OFF_V + sv * TILE;
          ptx::tma_load_2d(vt, &tm, v_full(sv), col_v, r);
          ptx::tma_load_2d(vt + BOX, &tm, v_full(sv), col_v + 64, r);
          ++ve;
          if (j == 0 && it.n1 > 0) ok = load_q(it, 1);
        }
      }
      // every load issued has landed before the CTA may exit: the last
      // entry of each stage, the last Q of each tile
      bool dr = true;
      for (uint32_t s = 0; s < F_KST; ++s)
        if (ke > s) {
          const uint32_t e = ke - 1 - (ke - 1 + F_KST - s) % F_KST;
          dr = ptx::mbar_wait(k_full(s), (e / F_KST) & 1) && dr;
        }
      for (uint32_t s = 0; s < F_VST; ++s)
        if (ve > s) {
          const uint32_t e = ve - 1 - (ve - 1 + F_VST - s) % F_VST;
          dr = ptx::mbar_wait(v_full(s), (e / F_VST) & 1) && dr;
        }
      for (int t = 0; t < 2; ++t)
        if (qn[t] > 0) dr = ptx::mbar_wait(q_full(t), (qn[t] - 1) & 1) && dr;
      if (!dr) wait_failed(13);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t qc0 = 0u, qc1 = 0u;  // Q loads consumed per tile
      uint32_t pc0 = 0u, pc1 = 0u;  // P_t hand-overs consumed per tile
      // K and V ring entries advance in step, one per key block of an item.
      // Tile 1 reads an entry after tile 0 does (within an item the rounds
      // issue tile 0 first; across items tile 1 never starts the next item
      // before tile 0), so an entry is released by tile 1's MMA, or by tile
      // 0's where tile 1 does not read it (last = true).
      auto issue_s = [&](int t, uint32_t e, bool last) {  // S_t = Q_t K_e^T
        const uint32_t s = e % F_KST;
        if (!ptx::mbar_wait(k_full(s), (e / F_KST) & 1)) {
          wait_failed(14);
          return false;
        }
        ptx::tc_fence_after();
        const uint32_t qt = base + F_OFF_Q + t * TILE, kt = base + F_OFF_K + s * TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_bf16(tmem + 128u * t, kmajor_desc(qt, kk), kmajor_desc(kt, kk), IDESC_S, kk > 0);
        ptx::mma_commit(s_full(t));
        if (last) ptx::mma_commit(k_empty(s));
        return true;
      };
      auto issue_pv = [&](int t, uint32_t e, int j, int k, bool last) {  // O_t += P_t V_e
        uint32_t& pc = t ? pc1 : pc0;
        if (!ptx::mbar_wait(p_full(t), pc & 1)) {
          wait_failed(16);
          return false;
        }
        ++pc;
        const uint32_t s = e % F_VST;
        if (!ptx::mbar_wait(v_full(s), (e / F_VST) & 1)) {
          wait_failed(15);
          return false;
        }
        ptx::tc_fence_after();
        if (k == 0) tl_fwd(t, j, 7);
        const uint32_t vt = base + F_OFF_V + s * TILE;
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          ptx::mma_bf16_ts(tmem + 256u + 128u * t, tmem + 128u * t + 8u * kk, mnmajor_desc(vt, kk),
                           IDESC_PV, (j > 0 || kk > 0) ? 1u : 0u);
        if (last) ptx::mma_commit(v_empty(s));
        return true;
      };
      // S_t(0) of item it (index i, k-th of this CTA), block 0 at ring entry e0
      auto start_tile = [&](const FwdItem& it, int i, int k, int t, uint32_t e0) {
        uint32_t& qc = t ? qc1 : qc0;
        if (!ptx::mbar_wait(q_full(t), qc & 1)) {
          wait_failed(17);
          return false;
        }
        ++qc;
        if (t == 0) {
          if (!ptx::mbar_wait(k_full(e0 % F_KST), (e0 / F_KST) & 1)) {
            wait_failed(14);
            return false;
          }
          tl_fitem(i, 2);
        }
        if (!issue_s(t, e0, t == 1 || it.n1 == 0)) return false;
        if (k == 0) tl_fwd(t, 0, 0);
        if ((t ? it.n1 : it.n0) == 1) ptx::mma_commit(q_empty(t));  // the tile's last S of the item
        return true;
      };
      int k = 0, i = fwd_item_at(a, 0, cta, G);
      uint32_t kb = 0;  // ring entry of the current item's block 0
      FwdItem it{};
      if (i < a.items) {
        it = fwd_item(a, i);
        ok = start_tile(it, i, 0, 0, 0u);
        if (ok && it.n1 > 0) ok = start_tile(it, i, 0, 1, 0u);
      }
      while (ok && i < a.items) {
        const int nmax = max(it.n0, it.n1);
        const int inext = fwd_item_at(a, k + 1, cta, G);
        const bool has_next = inext < a.items;
        FwdItem nx{};
        if (has_next) nx = fwd_item(a, inext);
        const uint32_t kb_next = kb + (uint32_t)nmax;
        for (int j = 0; j < nmax && ok; ++j) {
          bool done0 = false, done1 = false;  // the tile's last PV of the item issued in this round
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int n = t ? it.n1 : it.n0;
            if (!ok || j >= n) continue;
            ok = issue_pv(t, kb + j, j, k, t == 1 || it.n1 <= j);
            if (!ok) break;
            if (k == 0) tl_fwd(t, j, 6);
            if (j + 1 < n) {
              ok = issue_s(t, kb + j + 1, t == 1 || it.n1 <= j + 1);
              if (!ok) break;
              if (k == 0) tl_fwd(t, j + 1, 0);
              if (j + 2 == n) ptx::mma_commit(q_empty(t));  // the tile's last S of the item
            } else {
              ptx::mma_commit(o_full(t));  // the tile's last PV of the item
              if (t) done1 = true; else done0 = true;
            }
          }
          // a tile whose item ended in this round starts the next item
          if (ok && done0 && has_next) ok = start_tile(nx, inext, k + 1, 0, kb_next);
          if (ok && done1 && has_next && nx.n1 > 0) ok = start_tile(nx, inext, k + 1, 1, kb_next);
        }
        // a tile with no blocks in this item starts the next one here
        if (ok && has_next && it.n1 == 0 && nx.n1 > 0) ok = start_tile(nx, inext, k + 1, 1, kb_next);
        kb = kb_next;
        it = nx;
        i = inext;
        ++k;
      }
      ptx::mma_commit(bar_drain);  // completes once every MMA issued above has
      if (!ptx::mbar_wait(bar_drain, 0)) {
        ok = false;
        wait_failed(18);
      }
    }
  } else {
    const int t = (warp - 2) >> 2, qq = warp & 3;
    const int row = qq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    const uint32_t t_s = tmem + 128u * t + lane_off, t_o = tmem + 256u + 128u * t + lane_off;
    uint32_t sc = 0u, oc = 0u;  // S_t blocks and finished items of this tile so far
    for (int k = 0; ok; ++k) {
      const int i = fwd_item_at(a, k, cta, G);
      if (i >= a.items) break;
      const FwdItem it = fwd_item(a, i);
      const int nt = t ? it.n1 : it.n0;
      if (nt == 0) continue;
      const int h = it.h, row0 = it.b * a.S;
      const int qt0 = it.q0 + t * BQ;  // first query of the tile
      const int qi = qt0 + row;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < nt && ok; ++j, ++sc) {
        if (!__all_sync(0xffffffffu, ptx::mbar_wait(s_full(t), sc & 1))) {
          ok = false;
          if (lane == 0) wait_failed(19);
          break;
        }
        ptx::tc_fence_after();
        if (k == 0 && qq == 2 && lane == 0) tl_fwd(t, j, 1);
        if (j == 0 && t == 0 && qq == 0 && lane == 0) tl_fitem(i, 3);
        float sv[BKV];
        ptx::tmem_ld128(t_s, sv);
        const int kbase = j * BKV;
        // a block every row of the tile sees whole needs no mask (warp-uniform)
        const bool full = (j + 1) * BKV <= a.S && (!a.causal || (j + 1) * BKV <= qt0 + 1);
        if (!full) {
          // keys kbase + i with i >= nvis are past the diagonal or the sequence end
          const int nvis = (a.causal ? min(qi + 1, a.S) : a.S) - kbase;
#pragma unroll
          for (int i = 0; i < BKV; ++i)
            if (i >= nvis) sv[i] = -INFINITY;
        }
        // row maximum of the raw scores in eight independent chains (the scale
        // is positive, so it is applied to the maximum alone)
        float pm[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) pm[c] = sv[c];
#pragma unroll
        for (int i = 8; i < BKV; ++i) pm[i % 8] = fmaxf(pm[i % 8], sv[i]);
        const float mx = fmaxf(fmaxf(fmaxf(pm[0], pm[1]), fmaxf(pm[2], pm[3])),
                               fmaxf(fmaxf(pm[4], pm[5]), fmaxf(pm[6], pm[7]))) * a.scale_log2;
        const float m_new = fmaxf(m_ref, mx);
        // O_t is rescaled by f (below, once P no longer needs S's registers)
        // where the reference maximum is raised
        float f = 1.f;
        bool rescale = false;
        if (j == 0) {
          m_ref = m_new;
        } else {
          const bool need = m_new > m_ref + RESCALE_LOG2;
          rescale = __any_sync(0xffffffffu, need);  // warp-uniform: tcgen05.ld/st are collective
          if (need) {
            f = exp2f(m_ref - m_new);
            l *= f;
            m_ref = m_new;
          }
        }
        // P = exp2(s * scale - m_ref) as packed bf16 over S's first 64 columns.
        // Scale and shift in one fp32x2 FMA per pair, the row sum in four fp32x2
        // accumulators.
        const bool live = m_ref != -INFINITY;
        const uint64_t sc2 = f2_splat(a.scale_log2), nm2 = f2_splat(-m_ref);
        uint64_t acc[4] = {0ull, 0ull, 0ull, 0ull};
        // the packed word of keys (2i, 2i+1) goes to sv[i] (already consumed), so
        // P needs no registers beyond S's
#pragma unroll
        for (int i = 0; i < BKV / 2; ++i) {
          const uint64_t x = f2_fma(f2_pack(sv[2 * i], sv[2 * i + 1]), sc2, nm2);
          float p0 = fast_exp2(f2_lo(x)), p1 = fast_exp2(f2_hi(x));
          if (!live) p0 = p1 = 0.f;  // (a row with no visible key; x is NaN there)
          acc[i % 4] = f2_add(acc[i % 4], f2_pack(p0, p1));
          sv[i] = __uint_as_float(pack2(p0, p1));
        }
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t w[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(sv[32 * half + i]);
          ptx::tmem_st32_nowait(t_s + 32u * half, w);
        }
        const uint64_t acc2 = f2_add(f2_add(acc[0], acc[1]), f2_add(acc[2], acc[3]));
        const float rs = f2_lo(acc2) + f2_hi(acc2);
        if (rescale) {
          // S_t(j) complete => PV_t(j-1) complete: O_t may be rescaled in
          // place; PV_t(j) waits for this warp's arrival below
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            float v[32];
            ptx::tmem_ld32(t_o + c0, v);
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i] * f);
            ptx::tmem_st32_nowait(t_o + c0, w);
          }
        }
        ptx::tmem_wait_st();
        l += rs;
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(p_full(t));
        if (k == 0 && lane == 0) tl_fwd(t, j, 2 + qq);
      }
      if (!ok) break;
      {
        // the tile's last PV of the item is complete (or the MMA thread gave up)
        const bool fin = __all_sync(0xffffffffu, ptx::mbar_wait(o_full(t), oc & 1));
        ++oc;
        if (!fin && lane == 0) wait_failed(20);
        if (qq == 0 && lane == 0) tl_fitem(i, 4 + t);
        ptx::tc_fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const bool store = ok && fin && qi < a.S;
        // O rows through this warp's 4 KB slice of shared memory, 64 columns
        // at a time: lane r writes its row's 128 bytes as eight 16-byte
        // chunks (chunk c at c ^ (r & 7), so eight lanes cover all banks),
        // then each store instruction writes 4 rows x 128 contiguous bytes
        uint8_t* stg = gbase + F_OFF_EPI + (warp - 2) * 4096;
        const int rw0 = qt0 + qq * 32;  // first query row of this warp
        __nv_bfloat16* ow = a.o + (int64_t)(row0 + rw0) * a.H + h * D;
        float v[D];
        ptx::tmem_ld128(t_o, v);  // the whole row in one load (every lane: warp-collective)
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 64) {
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float* x = v + c0 + 8 * c;
            *reinterpret_cast<uint4*>(stg + lane * 128 + ((c ^ (lane & 7)) << 4)) =
                make_uint4(pack2(x[0] * inv, x[1] * inv), pack2(x[2] * inv, x[3] * inv),
                           pack2(x[4] * inv, x[5] * inv), pack2(x[6] * inv, x[7] * inv));
          }
          __syncwarp();
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int r = 4 * u + (lane >> 3), c = lane & 7;
            const uint4 w = *reinterpret_cast<const uint4*>(stg + r * 128 + ((c ^ (r & 7)) << 4));
            if (ok && fin && rw0 + r < a.S)
              *reinterpret_cast<uint4*>(ow + (int64_t)r * a.H + c0 + 8 * c) = w;
          }
          __syncwarp();
        }
        if (store) a.lse[(int64_t)h * a.M + row0 + qi] = (m_ref + log2f(l)) * 0.69314718055994531f;
        if (!(ok && fin)) ok = false;
        if (t == 1 && qq == 0 && lane == 0) tl_fitem(i, 6);
      }
    }
  }
  if (!ok) atomicExch(&g_attn_error, 1);
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  progress(0, 999);
  if (tid == 0) tl_fitems(a, cta, G, 7);
}

// ---------------------------------------------------------------------------
// Backward.  With s = Q K^T / sqrt(d), P = exp(s - LSE), delta = rowsum(dO * O):
//   dP = dO V^T,  dS = P * (dP - delta),
//   dQ = dS K / sqrt(d),  dK = dS^T Q / sqrt(d),  dV = P^T dO.
// Two kernels own disjoint outputs, so there are no atomics:
//   dq kernel   persistent: one CTA per SM over work items of 128 queries,
//               each looped over 128-key blocks (row = query)
//   dkv kernel  one CTA per 128 keys, loops over 64-query blocks (row = key)
// ---------------------------------------------------------------------------
struct BwdArgs {
  const float* lse;
  const float* delta;
  __nv_bfloat16* dqkv;
  int S, H, heads, M, causal;
  float scale_log2;  // log2(e) / sqrt(d)
  float scale;       // 1 / sqrt(d)
  int batch, tiles;  // sequences; 128-row tiles per sequence
  int items;         // batch * heads * tiles
  // optional: column sums of dqkv as stored, one partial row of 3H floats per
  // (sequence, 128-row tile, lane quarter): row (b tiles + t) 4 + q; null = off
  float* bias_part;
};

// Column sums over the warp's 32 rows: lane l holds x[c] = its row's value in
// column c (c < 32); on return lane l's x[0] is the sum over the 32 lanes of
// column l (a fixed butterfly: 31 shuffles).
__device__ __forceinline__ void warp_column_sums(float (&x)[32], int lane) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float send = upper ? x[i] : x[i + off];
      const float keep = upper ? x[i + off] : x[i];
      x[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
  }
}
// A value as a bf16 store keeps it.
__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16(v)); }

// Both backward kernels are warp-specialised pipelines: one warp issues the
// TMA loads, one thread the MMAs, sixteen warps do the element-wise work
// between them (their layouts are described at each kernel).
constexpr int BK = 64;                  // keys or queries per block
constexpr int BOX64 = 64 * 64 * 2;      // one TMA box: 64 rows x 64 bf16 (8 KB)
constexpr int T64 = 2 * BOX64;          // 64 rows x 128 dims (16 KB)
constexpr int PB = 128 * 64 * 2;        // 128 rows x 64 bf16, one box width (16 KB)
constexpr uint64_t BWD_WAIT = 1ull << 29;  // cycles before a wait gives up (~0.25 s)
// S^T = K Q_i^T and dP^T = V dO_i^T (dkv): M = 128 keys, N = 64 queries,
// both operands K-major over d.
constexpr uint32_t IDESC_N64 = ptx::idesc_bf16_f32(128, BK, false, false);
// dV += P^T dO_i, dK += dS^T Q_i (dkv): M = 128 keys, N = 128 dims, A K-major
// over the 64 queries of the block, B MN-major.
constexpr uint32_t IDESC_ACC = ptx::idesc_bf16_f32(128, D, false, true);

// [64 rows][128 cols] K-major tile stored as two 64-column boxes, k-step kk of 8.
__device__ __forceinline__ uint64_t kmajor64_desc(uint32_t tile, int kk) {
  return desc_step(ptx::smem_desc_sw128(tile, 16, 1024), (kk >> 2) * BOX64 + (kk & 3) * 32);
}
// [64 k-rows][128 n-cols] MN-major tile stored as two 64-column boxes, k-step kk of 4.
__device__ __forceinline__ uint64_t mnmajor64_desc(uint32_t tile, int kk) {
  return desc_step(ptx::smem_desc_sw128(tile, BOX64, 1024), kk * 2048);
}
// [128 rows][64 cols] K-major buffer (one box width), k-step kk of 4.
__device__ __forceinline__ uint64_t kmajor_blk_desc(uint32_t buf, int kk) {
  return desc_step(ptx::smem_desc_sw128(buf, 16, 1024), kk * 32);
}
// Warp-uniform bounded wait (every lane waits; the warp agrees on the outcome).
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity) {
  return __all_sync(0xffffffffu, ptx::mbar_wait(bar, parity, BWD_WAIT));
}

// dq kernel: persistent, one CTA per SM.  A work item is 128 queries of one
// (sequence, head), looped over 128-key blocks; items are numbered heaviest
// first (the causal tiles nearest the end of a sequence see the most keys)
// and CTA c of G takes items c, 2G - 1 - c, 2G + c, ...  608 threads:
//   warp 0       TMA loads in the order they are consumed: per item K_0 and
//                V_0, then Q and dO (once the previous item's last S and dP
//                MMAs have read them), then K_j into a three-stage and V_j
//                into a two-stage ring; the rings run on across items;
//   warp 1       TMEM allocation; one thread issues the S and dP MMAs;
//   warps 2..17  element-wise: warp w owns TMEM lanes 32 (w % 4) .. + 31 (one
//                query row each) and columns 32 ((w - 2) / 4) .. + 31 of a block;
//   warp 18      one thread issues the dQ accumulation MMAs.
// Per block j:
//   S_j = Q K_j^T, dP_j = dO V_j^T    N = 128, into TMEM (one buffer each); the
//                                    element-wise warps load their 32 columns of
//                                    both and release the buffers at once, so
//                                    S_{j+1}, dP_{j+1} are computed while they
//                                    form dS_j = P_j * (dP_j - delta)
//   dS_j                             packed bf16 into TMEM (64 columns)
//   dQ += dS_j K_j                   A = dS_j from TMEM, B = K_j (MN-major)
// The two kinds of MMA come from two threads, so neither waits behind the
// other's barrier (an issuing thread cannot run ahead of its own waits, and
// the tensor core drains while it waits); their outputs are disjoint and each
// thread's commits track its own MMAs.
// V_j is released when SdP_j completes, K_j when ACC_j completes: with three
// K stages and two V stages the loads of the next blocks are never behind the
// MMAs that wait for them.  Every MMA is 128 x 128 x 16 (one MMA's tensor
// work, 64 clocks, exceeds its issue cost).
// TMEM: S 0..127, dP 128..255, dQ 256..383, dS 384..447.
// Across items: the next item's first dQ MMA (which overwrites dQ) waits for
// its first dS, which the element-wise warps hand over only after they have
// read the finished item's dQ out of TMEM.
constexpr int DQ_NT = 608;
constexpr int DQ_ACC_WARP = 18;  // issues the dQ accumulation MMAs
constexpr int DQ_EW = 16;               // element-wise warps, four per lane quarter
constexpr int DQ_KST = 3, DQ_VST = 2;   // K and V stages of 128 keys
constexpr int DQ_OFF_Q = 0, DQ_OFF_DO = TILE, DQ_OFF_K = 2 * TILE;
constexpr int DQ_OFF_V = DQ_OFF_K + DQ_KST * TILE, DQ_OFF_BAR = DQ_OFF_V + DQ_VST * TILE;
// qdo_full, qdo_empty, k_full[3], k_empty[3], v_full[2], v_empty[2], sdp_full,
// sdp_empty, ds_full, ds_empty, fin, sdp_drain
constexpr int DQ_NBAR = 2 + 2 * DQ_KST + 2 * DQ_VST + 6;
constexpr int DQ_SMEM = DQ_OFF_BAR + 8 * DQ_NBAR + 16 + 1024;
static_assert(DQ_SMEM <= 232448, "dq kernel: more than 227 KB of shared memory");

// Brings a 2-D box of the tensor map into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2(const void* tmap, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(x), "r"(y)
               : "memory");
}

struct DqItem {
  int h, bb, q0, n;  // head, sequence, first query, key blocks
};
__device__ __forceinline__ DqItem dq_item(const BwdArgs& a, int i) {
  const int bh = a.heads * a.batch;
  const int tile = a.tiles - 1 - i / bh, r = i % bh;
  const int nkv_all = (a.S + BKV - 1) / BKV;
  DqItem it;
  it.h = r % a.heads;
  it.bb = r / a.heads;
  it.q0 = tile * BQ;
  it.n = a.causal ? min(tile + 1, nkv_all) : nkv_all;
  return it;
}

__global__ void __launch_bounds__(DQ_NT, 1)
attn_bwd_dq_tc_kernel(const __grid_constant__ CUtensorMap tq128,
                      const __grid_constant__ CUtensorMap tdo128, const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + DQ_OFF_BAR;
  const uint32_t qdo_full = bars, qdo_empty = bars + 8u;
  auto k_full = [&](uint32_t s) { return bars + 8u * (2 + s); };
  auto k_empty = [&](uint32_t s) { return bars + 8u * (2 + DQ_KST + s); };
  auto v_full = [&](uint32_t s) { return bars + 8u * (2 + 2 * DQ_KST + s); };
  auto v_empty = [&](uint32_t s) { return bars + 8u * (2 + 2 * DQ_KST + DQ_VST + s); };
  const uint32_t sdp_full = bars + 8u * (2 + 2 * DQ_KST + 2 * DQ_VST), sdp_empty = sdp_full + 8u;
  const uint32_t ds_full = sdp_full + 16u, ds_empty = sdp_full + 24u, bar_fin = sdp_full + 32u;
  const uint32_t sdp_drain = sdp_full + 40u;
  const uint32_t tslot = bars + 8u * DQ_NBAR;

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int cta = blockIdx.x, G = gridDim.x;

  if (tid == 0) {
    ptx::mbar_init(qdo_full, 1);
    ptx::mbar_init(qdo_empty, 1);
    for (int s = 0; s < DQ_KST; ++s) {
      ptx::mbar_init(k_full(s), 1);
      ptx::mbar_init(k_empty(s), 1);
    }
    for (int s = 0; s < DQ_VST; ++s) {
      ptx::mbar_init(v_full(s), 1);
      ptx::mbar_init(v_empty(s), 1);
    }
    ptx::mbar_init(sdp_full, 1);
    ptx::mbar_init(sdp_empty, DQ_EW);
    ptx::mbar_init(ds_full, DQ_EW);
    ptx::mbar_init(ds_empty, 1);
    ptx::mbar_init(bar_fin, 1);
    ptx::mbar_init(sdp_drain, 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tq128);
    ptx::prefetch_tmap(&tdo128);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tslot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + (tslot - base));
  const uint32_t t_s = tmem, t_dp = tmem + 128, t_dq = tmem + 256, t_ds = tmem + 384;
  progress(1, 2);
  pdl_wait();
  pdl_trigger();
  progress(1, 3);
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      // K and V ring entries loaded (entry e in stage e % depth), Q/dO loads
      uint32_t ke = 0, ve = 0, nq = 0;
      auto load_kv = [&](int r, int col_k, int col_v) {
        const uint32_t sk = ke % DQ_KST, uk = ke / DQ_KST;
        if (uk > 0 && !ptx::mbar_wait(k_empty(sk), (uk - 1) & 1, BWD_WAIT)) return false;
        const uint32_t kt = base + DQ_OFF_K + sk * TILE;
        ptx::mbar_arrive_expect_tx(k_full(sk), TILE);
        ptx::tma_load_2d(kt, &tq128, k_full(sk), col_k, r);
        ptx::tma_load_2d(kt + BOX, &tq128, k_full(sk), col_k + 64, r);
        ++ke;
        const uint32_t sv = ve % DQ_VST, uv = ve / DQ_VST;
        if (uv > 0 && !ptx::mbar_wait(v_empty(sv), (uv - 1) & 1, BWD_WAIT)) return false;
        const uint32_t vt = base + DQ_OFF_V + sv * TILE;
        ptx::mbar_arrive_expect_tx(v_full(sv), TILE);
        ptx::tma_load_2d(vt, &tq128, v_full(sv), col_v, r);
        ptx::tma_load_2d(vt + BOX, &tq128, v_full(sv), col_v + 64, r);
        ++ve;
        return true;
      };
      for (int k = 0; ok; ++k) {
        const int i = persistent_item(k, cta, G);
        if (i >= a.items) break;
        const DqItem it = dq_item(a, i);
        const int row0 = it.bb * a.S, col_k = a.H + it.h * D, col_v = 2 * a.H + it.h * D;
        ok = load_kv(row0, col_k, col_v);
        // Q and dO are free once the previous item's last S and dP are done
        if (ok && nq > 0 && !ptx::mbar_wait(qdo_empty, (nq - 1) & 1, BWD_WAIT)) ok = false;
        if (!ok) {
          wait_failed(101);
          break;
        }
        ptx::mbar_arrive_expect_tx(qdo_full, 2 * TILE);
        ptx::tma_load_2d(base + DQ_OFF_Q, &tq128, qdo_full, it.h * D, row0 + it.q0);
        ptx::tma_load_2d(base + DQ_OFF_Q + BOX, &tq128, qdo_full, it.h * D + 64, row0 + it.q0);
        ptx::tma_load_2d(base + DQ_OFF_DO, &tdo128, qdo_full, it.h * D, row0 + it.q0);
        ptx::tma_load_2d(base + DQ_OFF_DO + BOX, &tdo128, qdo_full, it.h * D + 64, row0 + it.q0);
        ++nq;
        // the next item's Q and dO into L2, so that their load at the item
        // change (Q and dO are single-buffered) comes from L2
        const int inext = persistent_item(k + 1, cta, G);
        if (inext < a.items) {
          const DqItem nx = dq_item(a, inext);
          const int rn = nx.bb * a.S + nx.q0;
          tma_prefetch_l2(&tq128, nx.h * D, rn);
          tma_prefetch_l2(&tq128, nx.h * D + 64, rn);
          tma_prefetch_l2(&tdo128, nx.h * D, rn);
          tma_prefetch_l2(&tdo128, nx.h * D + 64, rn);
        }
        for (int j = 1; j < it.n && ok; ++j) ok = load_kv(row0 + j * BKV, col_k, col_v);
        if (!ok) wait_failed(101);
      }
      // every load issued has landed before the CTA may exit: the last entry
      // of each stage, the last Q/dO
      bool dr = true;
      for (uint32_t s = 0; s < DQ_KST; ++s)
        if (ke > s) {
          const uint32_t e = ke - 1 - (ke - 1 - s) % DQ_KST;
          dr = ptx::mbar_wait(k_full(s), (e / DQ_KST) & 1, BWD_WAIT) && dr;
        }
      for (uint32_t s = 0; s < DQ_VST; ++s)
        if (ve > s) {
          const uint32_t e = ve - 1 - (ve - 1 - s) % DQ_VST;
          dr = ptx::mbar_wait(v_full(s), (e / DQ_VST) & 1, BWD_WAIT) && dr;
        }
      if (nq > 0) dr = ptx::mbar_wait(qdo_full, (nq - 1) & 1, BWD_WAIT) && dr;
      if (!dr) wait_failed(102);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t g = 0;  // blocks so far over all items (= K/V ring entries)
      for (int k = 0; ok; ++k) {
        const int i = persistent_item(k, cta, G);
        if (i >= a.items) break;
        const DqItem it = dq_item(a, i);
        if (!ptx::mbar_wait(qdo_full, k & 1, BWD_WAIT)) {
          ok = false;
          wait_failed(103);
          break;
        }
        for (int j = 0; j < it.n && ok; ++j, ++g) {  // S_j = Q K_j^T, dP_j = dO V_j^T
          const uint32_t sk = g % DQ_KST, sv = g % DQ_VST;
          if (!ptx::mbar_wait(k_full(sk), (g / DQ_KST) & 1, BWD_WAIT) ||
              !ptx::mbar_wait(v_full(sv), (g / DQ_VST) & 1, BWD_WAIT)) {
            ok = false;
            wait_failed(104);
            break;
          }
          // the element-wise warps have loaded the previous block's S and dP
          if (g >= 1 && !ptx::mbar_wait(sdp_empty, (g - 1) & 1, BWD_WAIT)) {
            ok = false;
            wait_failed(105);
            break;
          }
          ptx::tc_fence_after();
          if (j == 0) tl_unit(1, i, 0);
          const uint32_t kt = base + DQ_OFF_K + sk * TILE, vt = base + DQ_OFF_V + sv * TILE;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_bf16(t_s, kmajor_desc(base + DQ_OFF_Q, kk), kmajor_desc(kt, kk), IDESC_S, kk > 0);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            ptx::mma_bf16(t_dp, kmajor_desc(base + DQ_OFF_DO, kk), kmajor_desc(vt, kk), IDESC_S, kk > 0);
          ptx::mma_commit(sdp_full);
          ptx::mma_commit(v_empty(sv));
          if (j + 1 == it.n) ptx::mma_commit(qdo_empty);  // the item's last read of Q and dO
          if (k == 0) tl_block(1, j, 0);
        }
      }
      ptx::mma_commit(sdp_drain);  // completes once every MMA this thread issued has
      if (!ptx::mbar_wait(sdp_drain, 0, BWD_WAIT)) {
        ok = false;
        wait_failed(107);
      }
    }
  } else if (warp == DQ_ACC_WARP) {
    if (lane == 0) {
      uint32_t g = 0;
      int nk = 0;  // items finished
      for (int k = 0; ok; ++k) {
        const int i = persistent_item(k, cta, G);
        if (i >= a.items) break;
        const DqItem it = dq_item(a, i);
        for (int j = 0; j < it.n && ok; ++j, ++g) {  // dQ += dS_j K_j (over the block's 128 keys)
          const uint32_t sk = g % DQ_KST;
          if (!ptx::mbar_wait(ds_full, g & 1, BWD_WAIT)) {
            ok = false;
            wait_failed(106);
            break;
          }
          ptx::tc_fence_after();
          const uint32_t kt = base + DQ_OFF_K + sk * TILE;
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            ptx::mma_bf16_ts(t_dq, t_ds + 8u * kk, mnmajor_desc(kt, kk), IDESC_PV,
                             (j > 0 || kk > 0) ? 1u : 0u);
          // S_j, dP_j (which also read K_j) completed before the element-wise
          // warps could hand over dS_j, so K_j is free once these MMAs are
          ptx::mma_commit(ds_empty);
          ptx::mma_commit(k_empty(sk));
          if (k == 0) tl_block(1, j, 1);
        }
        if (!ok) break;
        ptx::mma_commit(bar_fin);  // the item's dQ is complete once this does
        nk = k + 1;
      }
      // every MMA this thread issued is complete before the CTA may exit
      if (nk > 0 && !ptx::mbar_wait(bar_fin, (nk - 1) & 1, BWD_WAIT)) {
        ok = false;
        wait_failed(111);
      }
      if (!ok) {  // one more commit drains whatever was issued after the last finished item
        ptx::mma_commit(bar_fin);
        (void)ptx::mbar_wait(bar_fin, nk & 1, BWD_WAIT);
      }
    }
  } else {
    const int qq = warp & 3, sub = (warp - 2) >> 2;  // lane quarter; columns 32 sub .. + 31
    const int row = qq * 32 + lane;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    uint32_t g = 0;
    // this row's LSE (base 2) and delta of an item, read one item ahead
    auto stats = [&](int i, float& lse2, float& dlt) {
      lse2 = 0.f;
      dlt = 0.f;
      if (i >= a.items) return;
      const DqItem it = dq_item(a, i);
      const int qi = it.q0 + row;
      if (qi < a.S) {
        const int64_t o = (int64_t)it.h * a.M + it.bb * a.S + qi;
        lse2 = a.lse[o] * 1.4426950408889634f;
        dlt = a.delta[o];
      }
    };
    float lse2_next, dlt_next;
    stats(persistent_item(0, cta, G), lse2_next, dlt_next);
    for (int k = 0; ok; ++k) {
      const int i = persistent_item(k, cta, G);
      if (i >= a.items) break;
      const DqItem it = dq_item(a, i);
      const int q0 = it.q0, row0 = it.bb * a.S, h = it.h, n = it.n;
      const int qi = q0 + row;
      const bool valid_q = qi < a.S;
      const float lse2 = lse2_next, dlt = dlt_next;
      stats(persistent_item(k + 1, cta, G), lse2_next, dlt_next);
      for (int j = 0; j < n && ok; ++j, ++g) {
        if (!warp_wait(sdp_full, g & 1)) {
          ok = false;
          if (lane == 0) wait_failed(108);
          break;
        }
        if (k == 0 && warp == 2 && lane == 0) tl_block(1, j, 2);
        ptx::tc_fence_after();
        float v[32], w[32];
        ptx::tmem_ld32x2(t_s + lane_off + sub * 32, t_dp + lane_off + sub * 32, v, w);
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(sdp_empty);  // the TMEM buffers may be overwritten
        // a block wholly visible to every row of the tile needs no mask (CTA-uniform)
        const bool full = q0 + BQ <= a.S && (j + 1) * BKV <= a.S && (!a.causal || (j + 1) * BKV <= q0 + 1);
        uint32_t pk[16];  // dS as packed bf16 pairs (keys 2i, 2i+1 of these 32)
        if (full) {
          const uint64_t sc = f2_splat(a.scale_log2), nl = f2_splat(-lse2), nd = f2_splat(-dlt);
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            const uint64_t x = f2_fma(f2_pack(v[2 * i2], v[2 * i2 + 1]), sc, nl);
            const uint64_t p = f2_pack(fast_exp2(f2_lo(x)), fast_exp2(f2_hi(x)));
            const uint64_t ds = f2_mul(p, f2_add(f2_pack(w[2 * i2], w[2 * i2 + 1]), nd));
            pk[i2] = pack2(f2_lo(ds), f2_hi(ds));
          }
        } else {
          // keys j BKV + 32 sub + c with c >= nvis are past the diagonal or the
          // sequence end (all of them for a row past the end)
          const int nvis = valid_q ? (a.causal ? min(qi + 1, a.S) : a.S) - (j * BKV + sub * 32) : 0;
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float p = c < nvis ? fast_exp2(v[c] * a.scale_log2 - lse2) : 0.f;
            v[c] = p * (w[c] - dlt);
          }
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) pk[i2] = pack2(v[2 * i2], v[2 * i2 + 1]);
        }
        // the dS columns are free once the previous block's dQ MMAs are done
        if (g >= 1 && !warp_wait(ds_empty, (g - 1) & 1)) {
          ok = false;
          if (lane == 0) wait_failed(109);
          break;
        }
        ptx::tc_fence_after();
        ptx::tmem_st16_nowait(t_ds + lane_off + sub * 16, pk);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ds_full);
        if (k == 0 && warp == 2 && lane == 0) tl_block(1, j, 3);
      }
      if (!ok) break;
      // the item's last accumulation is complete (or the MMA thread gave up)
      const bool fin = warp_wait(bar_fin, k & 1);
      ptx::tc_fence_after();
      float v0[32];  // tcgen05.ld is warp-collective: every lane loads
      ptx::tmem_ld32(t_dq + lane_off + sub * 32, v0);
      if (fin && valid_q) {
        uint4* out = reinterpret_cast<uint4*>(a.dqkv + (int64_t)(row0 + qi) * 3 * a.H + h * D + sub * 32);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          out[u] = make_uint4(pack2(v0[8 * u] * a.scale, v0[8 * u + 1] * a.scale),
                              pack2(v0[8 * u + 2] * a.scale, v0[8 * u + 3] * a.scale),
                              pack2(v0[8 * u + 4] * a.scale, v0[8 * u + 5] * a.scale),
                              pack2(v0[8 * u + 6] * a.scale, v0[8 * u + 7] * a.scale));
      }
      if (a.bias_part != nullptr) {  // this warp's 32 rows of the dQ columns, as stored
#pragma unroll
        for (int c = 0; c < 32; ++c) v0[c] = (fin && valid_q) ? bf16_round(v0[c] * a.scale) : 0.f;
        warp_column_sums(v0, lane);
        a.bias_part[((int64_t)(it.bb * a.tiles + q0 / BQ) * 4 + qq) * 3 * a.H + h * D + sub * 32 + lane] = v0[0];
      }
      if (!fin) ok = false;
      if (warp == 2 && lane == 0) tl_unit(1, i, 1);
    }
    if (!ok && lane == 0) atomicExch(&g_attn_error, 3);
  }
  progress(1, 990);
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  progress(1, 999);
}

// dkv kernel: one CTA per 128 keys, 64-query blocks, 608 threads:
//   warp 0       TMA loads (K and V once, then Q_i and dO_i into a four-stage
//                ring, each stage with its queries' LSE and delta, which the
//                warp reads from global memory a block ahead);
//   warp 1       TMEM allocation; one thread issues the S^T and dP^T MMAs;
//   warps 2..17  element-wise: warp w owns TMEM lanes 32 (w % 4) .. + 31 (one
//                key row each) and columns 16 ((w - 2) / 4) .. + 15 of a block;
//   warp 18      one thread issues the dV and dK accumulation MMAs.
// Per query block i:
//   S^T = K Q_i^T, dP^T = V dO_i^T     N = 64, into one of two TMEM buffers
//   P^T = exp2(S^T scale - LSE), dS^T = P^T (dP^T - delta)
//                                     (LSE and delta of the block's queries
//                                     from the stage, broadcast loads),
//                                     bf16 into one shared-memory buffer each
//   dV += P^T dO_i, dK += dS^T Q_i     N = 128 (d), contraction over the 64 queries
// The two kinds of MMA come from two threads, as in the dq kernel.
// The element-wise warps write block i's P^T and dS^T once the MMAs of
// block i-1's accumulation are done; they are still computing when those
// MMAs end, so one buffer each suffices.
constexpr int KV_NT = 608;
constexpr int KV_ACC_WARP = 18;  // issues the dV and dK accumulation MMAs
constexpr int KV_EW = 16;               // element-wise warps, four per lane quarter
constexpr int KV_QST = 4;               // Q/dO stages of 64 queries
constexpr int KV_OFF_K = 0, KV_OFF_V = TILE, KV_OFF_Q = 2 * TILE;
constexpr int KV_OFF_DO = KV_OFF_Q + KV_QST * T64;
constexpr int KV_OFF_PT = KV_OFF_DO + KV_QST * T64, KV_OFF_DST = KV_OFF_PT + PB;
constexpr int KV_OFF_STAT = KV_OFF_DST + PB;  // [stage][lse2[64] | delta[64]] fp32
constexpr int KV_OFF_BAR = KV_OFF_STAT + KV_QST * 2 * BK * 4;
// kv, q_full[3], q_empty[3], sdp_full[2], sdp_empty[2], pd_full, pd_empty, fin, sdp_drain
constexpr int KV_NBAR = 1 + 2 * KV_QST + 4 + 4;
// The dynamic shared memory is rounded up to a 1024-byte boundary (the
// swizzled tiles need it); this kernel's layout leaves room for at most
// KV_SLACK bytes of rounding, and the kernel checks the actual amount (the
// window starts 1024-byte aligned on this GPU, so none is used).
constexpr int KV_SLACK = 232448 - (KV_OFF_BAR + 8 * KV_NBAR + 16);
constexpr int KV_SMEM = 232448;
static_assert(KV_SLACK >= 0, "dkv kernel: more than 227 KB of shared memory");

// Writes 8 words of packed bf16 pairs (16 values: columns 16 c .. + 15 of this
// thread's row) into a [128 rows][64 cols] 128-byte-swizzled buffer.
__device__ __forceinline__ void store_row_quarter(uint8_t* buf, int row, int c, const uint32_t (&w)[8]) {
  uint8_t* r = buf + row * 128;
  *reinterpret_cast<uint4*>(r + (((2 * c) ^ (row & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
  *reinterpret_cast<uint4*>(r + (((2 * c + 1) ^ (row & 7)) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
}

__global__ void __launch_bounds__(KV_NT, 1)
attn_bwd_dkv_tc_kernel(const __grid_constant__ CUtensorMap tkv, const __grid_constant__ CUtensorMap tq64,
                       const __grid_constant__ CUtensorMap tdo64, const BwdArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  if (base - raw > (uint32_t)KV_SLACK) {  // the layout would not fit (uniform: every thread leaves)
    if (threadIdx.x == 0) atomicExch(&g_attn_error, 6);
    return;
  }
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + KV_OFF_BAR;
  const uint32_t bar_kv = bars;
  auto q_full = [&](int s) { return bars + 8u * (1 + s); };
  auto q_empty = [&](int s) { return bars + 8u * (1 + KV_QST + s); };
  auto sdp_full = [&](int b) { return bars + 8u * (1 + 2 * KV_QST + b); };
  auto sdp_empty = [&](int b) { return bars + 8u * (3 + 2 * KV_QST + b); };
  const uint32_t pd_full = bars + 8u * (5 + 2 * KV_QST), pd_empty = pd_full + 8u, bar_fin = pd_full + 16u;
  const uint32_t sdp_drain = pd_full + 24u;
  const uint32_t tslot = bars + 8u * KV_NBAR;
  float* stat = reinterpret_cast<float*>(gbase + KV_OFF_STAT);

  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  // grid (heads, batch, tiles): key tile 0 (the most query blocks) first
  const int ktile = blockIdx.z, h = blockIdx.x, bb = blockIdx.y;
  const int k0 = ktile * 128, row0 = bb * a.S;
  const int nq_all = (a.S + BK - 1) / BK;
  const int i0 = a.causal ? k0 / BK : 0;  // query blocks before the diagonal see none of these keys
  const int n = nq_all - i0;
  const int col_q = h * D, col_k = a.H + h * D, col_v = 2 * a.H + h * D;
  if (tid == 0) tl_cta(2, 0);

  if (tid == 0) {
    ptx::mbar_init(bar_kv, 1);
    for (int s = 0; s < KV_QST; ++s) {
      ptx::mbar_init(q_full(s), 1);
      ptx::mbar_init(q_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(sdp_full(b), 1);
      ptx::mbar_init(sdp_empty(b), KV_EW);
    }
    ptx::mbar_init(pd_full, KV_EW);
    ptx::mbar_init(pd_empty, 1);
    ptx::mbar_init(bar_fin, 1);
    ptx::mbar_init(sdp_drain, 1);
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&tkv);
    ptx::prefetch_tmap(&tq64);
    ptx::prefetch_tmap(&tdo64);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tslot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + (tslot - base));
  auto t_st = [&](int b) { return tmem + (uint32_t)(b * 128); };
  auto t_dpt = [&](int b) { return tmem + (uint32_t)(b * 128 + 64); };
  const uint32_t t_dv = tmem + 256, t_dk = tmem + 384;
  progress(2, 2);
  pdl_wait();
  pdl_trigger();
  progress(2, 3);
  bool ok = true;

  if (warp == 0) {
    if (lane == 0) {
      ptx::mbar_arrive_expect_tx(bar_kv, 2 * TILE);
      ptx::tma_load_2d(base + KV_OFF_K, &tkv, bar_kv, col_k, row0 + k0);
      ptx::tma_load_2d(base + KV_OFF_K + BOX, &tkv, bar_kv, col_k + 64, row0 + k0);
      ptx::tma_load_2d(base + KV_OFF_V, &tkv, bar_kv, col_v, row0 + k0);
      ptx::tma_load_2d(base + KV_OFF_V + BOX, &tkv, bar_kv, col_v + 64, row0 + k0);
    }
    // LSE (log2 units) and delta of block ii's 64 queries, two of each per lane;
    // the next block's are loaded before the wait for its stage
    auto ld_stat = [&](int ii, float (&v)[4]) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int q = (i0 + ii) * BK + lane + 32 * u;
        const bool vq = ii < n && q < a.S;
        const int64_t at = (int64_t)h * a.M + row0 + q;
        v[u] = vq ? a.lse[at] * 1.4426950408889634f : 0.f;
        v[2 + u] = vq ? a.delta[at] : 0.f;
      }
    };
    float cur[4];
    ld_stat(0, cur);
    int nl = 0;  // query blocks whose loads were issued
    for (int ii = 0; ii < n; ++ii) {
      const int s = ii % KV_QST;
      float nxt[4];
      ld_stat(ii + 1, nxt);
      bool w = true;
      if (lane == 0 && ii >= KV_QST) w = ptx::mbar_wait(q_empty(s), ((ii / KV_QST) & 1) ^ 1, BWD_WAIT);
      if (!__shfl_sync(0xffffffffu, w, 0)) {
        ok = false;
        if (lane == 0) wait_failed(201);
        break;
      }
      float* st = stat + s * 2 * BK;
      st[lane] = cur[0];
      st[lane + 32] = cur[1];
      st[BK + lane] = cur[2];
      st[BK + lane + 32] = cur[3];
      __syncwarp();  // the warp's stores precede lane 0's arrive on the stage barrier
      if (lane == 0) {
        ptx::mbar_arrive_expect_tx(q_full(s), 2 * T64);
        const uint32_t qt = base + KV_OFF_Q + s * T64, dt = base + KV_OFF_DO + s * T64;
        const int r = row0 + (i0 + ii) * BK;
        ptx::tma_load_2d(qt, &tq64, q_full(s), col_q, r);
        ptx::tma_load_2d(qt + BOX64, &tq64, q_full(s), col_q + 64, r);
        ptx::tma_load_2d(dt, &tdo64, q_full(s), h * D, r);
        ptx::tma_load_2d(dt + BOX64, &tdo64, q_full(s), h * D + 64, r);
      }
      nl = ii + 1;
#pragma unroll
      for (int u = 0; u < 4; ++u) cur[u] = nxt[u];
    }
    if (lane == 0) {
      // every load issued has landed before the CTA may exit (stage s last
      // held block s + R ((m - 1 - s) / R) of the m issued)
      bool dr = ptx::mbar_wait(bar_kv, 0, BWD_WAIT);
      for (int s = 0; s < KV_QST && s < nl; ++s)
        dr = ptx::mbar_wait(q_full(s), ((nl - 1 - s) / KV_QST) & 1, BWD_WAIT) && dr;
      if (!dr) wait_failed(202);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      ok = ptx::mbar_wait(bar_kv, 0, BWD_WAIT);
      if (!ok) wait_failed(203);
      auto sdp = [&](int ii) {  // S^T = K Q_i^T, dP^T = V dO_i^T into TMEM buffer ii % 2
        const int s = ii % KV_QST, b = ii & 1;
        if (!ptx::mbar_wait(q_full(s), (ii / KV_QST) & 1, BWD_WAIT)) { wait_failed(204); return false; }
        // the element-wise warps have loaded block ii-2 from this buffer
        if (ii >= 2 && !ptx::mbar_wait(sdp_empty(b), ((ii / 2) & 1) ^ 1, BWD_WAIT)) {
          wait_failed(205);
          return false;
        }
        ptx::tc_fence_after();
        const uint32_t qt = base + KV_OFF_Q + s * T64, dt = base + KV_OFF_DO + s * T64;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_bf16(t_st(b), kmajor_desc(base + KV_OFF_K, kk), kmajor64_desc(qt, kk), IDESC_N64, kk > 0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          ptx::mma_bf16(t_dpt(b), kmajor_desc(base + KV_OFF_V, kk), kmajor64_desc(dt, kk), IDESC_N64, kk > 0);
        ptx::mma_commit(sdp_full(b));
        tl_block(2, ii, 0);
        return true;
      };
      for (int ii = 0; ii < n && ok; ++ii) ok = sdp(ii);
      ptx::mma_commit(sdp_drain);  // completes once every MMA this thread issued has
      if (!ptx::mbar_wait(sdp_drain, 0, BWD_WAIT)) { ok = false; wait_failed(207); }
    }
  } else if (warp == KV_ACC_WARP) {
    if (lane == 0) {
      ok = ptx::mbar_wait(bar_kv, 0, BWD_WAIT);
      if (!ok) wait_failed(210);
      auto acc = [&](int ii) {  // dV += P^T dO_i, dK += dS^T Q_i
        const int s = ii % KV_QST;
        if (!ptx::mbar_wait(pd_full, ii & 1, BWD_WAIT)) { wait_failed(206); return false; }
        ptx::tc_fence_after();
        const uint32_t qt = base + KV_OFF_Q + s * T64, dt = base + KV_OFF_DO + s * T64;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint32_t accum = (ii > 0 || kk > 0) ? 1u : 0u;
          ptx::mma_bf16(t_dv, kmajor_blk_desc(base + KV_OFF_PT, kk), mnmajor64_desc(dt, kk), IDESC_ACC, accum);
          ptx::mma_bf16(t_dk, kmajor_blk_desc(base + KV_OFF_DST, kk), mnmajor64_desc(qt, kk), IDESC_ACC, accum);
        }
        // S^T, dP^T of block ii (which also read Q_i, dO_i) completed before
        // the element-wise warps could hand over P^T, dS^T: the stage is free
        // once these MMAs are
        ptx::mma_commit(pd_empty);
        ptx::mma_commit(q_empty(s));
        tl_block(2, ii, 1);
        return true;
      };
      for (int ii = 0; ii < n && ok; ++ii) ok = acc(ii);
      ptx::mma_commit(bar_fin);  // completes once every MMA this thread issued has
      if (!ptx::mbar_wait(bar_fin, 0, BWD_WAIT)) { ok = false; wait_failed(211); }
    }
  } else {
    const int qq = warp & 3, c = (warp - 2) >> 2;  // lane quarter; columns 16 c .. + 15
    const int row = qq * 32 + lane, kj = k0 + row;
    const bool valid_k = kj < a.S;
    const uint32_t lane_off = (uint32_t)(qq * 32) << 16;
    for (int ii = 0; ii < n && ok; ++ii) {
      const int s = ii % KV_QST, b = ii & 1, i = i0 + ii;
      // this block's S^T, dP^T are in TMEM (which also means its stage, and
      // the LSE / delta stored with it, have landed)
      if (!warp_wait(sdp_full(b), (ii / 2) & 1) || !warp_wait(q_full(s), (ii / KV_QST) & 1)) {
        ok = false;
        if (lane == 0) wait_failed(208);
        break;
      }
      if (warp == 2 && lane == 0) tl_block(2, ii, 2);
      ptx::tc_fence_after();
      float v[16], w[16];
      ptx::tmem_ld16x2(t_st(b) + lane_off + c * 16, t_dpt(b) + lane_off + c * 16, v, w);
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(sdp_empty(b));
      const float* st = stat + s * 2 * BK + c * 16;  // LSE of these 16 queries; delta at + BK
      uint32_t pp[8], pd[8];
      // a query block that sees every key of the tile needs no mask (CTA-uniform)
      const bool full = k0 + 128 <= a.S && (i + 1) * BK <= a.S && (!a.causal || i * BK >= k0 + 127);
      if (full) {
        const uint64_t sc = f2_splat(a.scale_log2);
#pragma unroll
        for (int k = 0; k < 16; k += 4) {
          const float4 l4 = *reinterpret_cast<const float4*>(st + k);
          const float4 d4 = *reinterpret_cast<const float4*>(st + BK + k);
#pragma unroll
          for (int e = 0; e < 4; e += 2) {
            const float l0 = e == 0 ? l4.x : l4.z, l1 = e == 0 ? l4.y : l4.w;
            const float d0 = e == 0 ? d4.x : d4.z, d1 = e == 0 ? d4.y : d4.w;
            const int kk = k + e;
            const uint64_t x = f2_fma(f2_pack(v[kk], v[kk + 1]), sc, f2_pack(-l0, -l1));
            const uint64_t p = f2_pack(fast_exp2(f2_lo(x)), fast_exp2(f2_hi(x)));
            const uint64_t ds = f2_mul(p, f2_add(f2_pack(w[kk], w[kk + 1]), f2_pack(-d0, -d1)));
            pp[kk / 2] = pack2(f2_lo(p), f2_hi(p));
            pd[kk / 2] = pack2(f2_lo(ds), f2_hi(ds));
          }
        }
      } else {
        // queries i BK + 16 c + k with k < k_lo are before this key (causal),
        // those with k >= k_hi past the sequence end; a key past the end sees none
        const int qbase = i * BK + c * 16;
        const int k_lo = a.causal ? kj - qbase : -(1 << 30), k_hi = valid_k ? a.S - qbase : 0;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float l2 = st[k], dl = st[BK + k];
          const float p = (k >= k_lo && k < k_hi) ? fast_exp2(v[k] * a.scale_log2 - l2) : 0.f;
          v[k] = p;
          w[k] = p * (w[k] - dl);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          pp[k] = pack2(v[2 * k], v[2 * k + 1]);
          pd[k] = pack2(w[2 * k], w[2 * k + 1]);
        }
      }
      // the P^T / dS^T buffers are free once block ii-1's accumulation is done
      if (ii >= 1 && !warp_wait(pd_empty, (ii - 1) & 1)) {
        ok = false;
        if (lane == 0) wait_failed(209);
        break;
      }
      store_row_quarter(gbase + KV_OFF_PT, row, c, pp);
      store_row_quarter(gbase + KV_OFF_DST, row, c, pd);
      ptx::fence_async_smem();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(pd_full);
      if (warp == 2 && lane == 0) tl_block(2, ii, 3);
    }
    const bool fin = warp_wait(bar_fin, 0);
    ptx::tc_fence_after();
    __nv_bfloat16* rowp = a.dqkv + (int64_t)(row0 + kj) * 3 * a.H;
#pragma unroll
    for (int part = 0; part < 2; ++part) {  // dK (scaled), then dV
      float v0[32];  // tcgen05.ld is warp-collective: every lane loads
      ptx::tmem_ld32((part == 0 ? t_dk : t_dv) + lane_off + c * 32, v0);
      const float sc = part == 0 ? a.scale : 1.f;
      if (ok && fin && valid_k) {
        uint4* out = reinterpret_cast<uint4*>(rowp + (part == 0 ? a.H : 2 * a.H) + h * D + c * 32);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          out[u] = make_uint4(pack2(v0[8 * u] * sc, v0[8 * u + 1] * sc), pack2(v0[8 * u + 2] * sc, v0[8 * u + 3] * sc),
                              pack2(v0[8 * u + 4] * sc, v0[8 * u + 5] * sc), pack2(v0[8 * u + 6] * sc, v0[8 * u + 7] * sc));
      }
      if (a.bias_part != nullptr) {  // this warp's 32 keys of the dK or dV columns, as stored
#pragma unroll
        for (int x = 0; x < 32; ++x) v0[x] = (ok && fin && valid_k) ? bf16_round(v0[x] * sc) : 0.f;
        warp_column_sums(v0, lane);
        a.bias_part[((int64_t)(bb * a.tiles + ktile) * 4 + qq) * 3 * a.H + (part == 0 ? a.H : 2 * a.H) +
                    h * D + c * 32 + lane] = v0[0];
      }
    }
    if (!(ok && fin) && lane == 0) atomicExch(&g_attn_error, 5);
  }
  progress(2, 990);
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  progress(2, 999);
  if (tid == 0) tl_cta(2, 1);
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
  static DeviceOnce attr;
  const cudaError_t ea = attr.run([] {
    return cudaFuncSetAttribute(attn_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                FWD_SMEM);
  });
  if (ea != cudaSuccess) return ea;
  FwdArgs fa;
  fa.o = static_cast<__nv_bfloat16*>(a.o);
  fa.lse = a.lse;
  fa.S = a.seq;
  fa.H = a.hidden;
  fa.heads = a.heads;
  fa.M = M;
  fa.causal = a.causal ? 1 : 0;
  fa.scale_log2 = 1.4426950408889634f / sqrtf((float)a.head_dim);
  const int64_t pairs = (a.seq + 2 * BQ - 1) / (2 * BQ);
  const int64_t items = pairs * a.batch * a.heads;
  if (items > (int64_t)INT32_MAX / 2) return cudaErrorInvalidConfiguration;
  fa.batch = a.batch;
  fa.pairs = (int)pairs;
  fa.items = (int)items;
  // persistent: one CTA per SM (shared memory and tensor memory allow one)
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int grid = (int)std::min<int64_t>(items, std::max(sms, 1));
  fa.use_sched = 0;
  if (items <= FWD_SCHED_ITEMS && grid <= FWD_SCHED_CTAS) {
    // longest processing time first: items in index order (heaviest first),
    // each to the CTA with the least work so far (ties: the lower CTA); the
    // work of an item is its key blocks plus a share for the item change
    const int nkv_all = (a.seq + BKV - 1) / BKV, bh = a.batch * a.heads;
    std::vector<int> load(grid, 0), cnt(grid, 0), owner((size_t)items);
    std::priority_queue<std::pair<int, int>, std::vector<std::pair<int, int>>, std::greater<>> q;
    for (int c = 0; c < grid; ++c) q.push({0, c});
    for (int i = 0; i < (int)items; ++i) {
      const int pair = (int)pairs - 1 - i / bh, q1 = pair * 2 * BQ + BQ;
      const int n1 = q1 >= a.seq ? 0 : (a.causal ? std::min(q1 / BKV + 1, nkv_all) : nkv_all);
      const int n0 = a.causal ? std::min(pair * 2 * BQ / BKV + 1, nkv_all) : nkv_all;
      const int w = 4 * std::max(n0, n1) + 3;
      const auto top = q.top();
      q.pop();
      owner[i] = top.second;
      ++cnt[top.second];
      q.push({top.first + w, top.second});
    }
    fa.sched.start[0] = 0;
    for (int c = 0; c < grid; ++c) fa.sched.start[c + 1] = (uint16_t)(fa.sched.start[c] + cnt[c]);
    std::vector<int> fill(fa.sched.start, fa.sched.start + grid);
    for (int i = 0; i < (int)items; ++i) fa.sched.order[fill[owner[i]]++] = (uint16_t)i;
    fa.use_sched = 1;
  }
  return launch_pdl(attn_fwd_tc_kernel, dim3(grid), dim3(F_NT), FWD_SMEM, st, m, fa);
}

cudaError_t attention_delta(const AttnArgs& a, cudaStream_t st);

cudaError_t attention_bwd_tc_bias(const AttnArgs& a, float* bias_part, cudaStream_t st);

cudaError_t attention_bwd_tc(const AttnArgs& a, cudaStream_t st) {
  return attention_bwd_tc_bias(a, nullptr, st);
}

// The same, and the column sums of dqkv as stored (the QKV bias gradient) as
// batch * ceil(seq / 128) * 4 partial rows of 3 hidden floats in bias_part,
// every element written, for a fixed-order reduction by the caller.
cudaError_t attention_bwd_tc_bias(const AttnArgs& a, float* bias_part, cudaStream_t st) {
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
  static DeviceOnce attr;
  const cudaError_t ea = attr.run([] {
    cudaError_t e = cudaFuncSetAttribute(attn_bwd_dq_tc_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, DQ_SMEM);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(attn_bwd_dkv_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                KV_SMEM);
  });
  if (ea != cudaSuccess) return ea;
  cudaError_t e = a.delta_ready ? cudaSuccess : attention_delta(a, st);
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
  ba.bias_part = bias_part;
  const int tiles = (a.seq + 127) / 128;
  if (tiles > 65535) return cudaErrorInvalidConfiguration;
  const int64_t items = (int64_t)tiles * a.batch * a.heads;
  if (items > (int64_t)INT32_MAX / 2) return cudaErrorInvalidConfiguration;
  ba.batch = a.batch;
  ba.tiles = tiles;
  ba.items = (int)items;
  // the dq kernel is persistent: one CTA per SM
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_bwd_dq_tc_kernel, dim3((int)std::min<int64_t>(items, std::max(sms, 1))),
                 dim3(DQ_NT), DQ_SMEM, st, tq128, tdo128, ba);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_bwd_dkv_tc_kernel, dim3(a.heads, a.batch, tiles), dim3(KV_NT), KV_SMEM,
                    st, tq128, tq64, tdo64, ba);
}

cudaError_t attention_set_progress(int* p) {
  return cudaMemcpyToSymbol(g_attn_progress, &p, sizeof(p));
}

namespace {
// One thread waits, with the bounded wait every tensor-core kernel here uses,
// on an mbarrier that nothing arrives on: the wait gives up after
// limit_cycles and records site 999, as a real stalled wait would.
__global__ void attn_wait_probe_kernel(uint64_t limit_cycles) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = ptx::smem_u32(&bar);
  ptx::mbar_init(b, 1);
  ptx::fence_mbar_init();
  if (!ptx::mbar_wait(b, 0, limit_cycles)) wait_failed(999);
}
}  // namespace

cudaError_t attention_wait_probe(uint64_t limit_cycles, cudaStream_t st) {
  attn_wait_probe_kernel<<<1, 1, 0, st>>>(limit_cycles);
  ++g_launch_count;
  return cudaGetLastError();
}

cudaError_t attention_set_timeline(unsigned long long* p) {
  return cudaMemcpyToSymbol(g_attn_timeline, &p, sizeof(p));
}

int attention_read_and_clear_error() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_attn_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_attn_error, &z, sizeof(int));
  return v;
}

}  // namespace oases
