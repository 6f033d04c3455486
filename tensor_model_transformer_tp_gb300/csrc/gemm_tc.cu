// bf16 GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
//   D[m, n] = sum_k A(m, k) B(n, k), fp32 accumulation in tensor memory,
//   followed by the block's fused epilogue (bias, GeLU, residual, GeLU',
//   fp32 accumulate).
//
// One CTA per SM, persistent over 128 x BN output tiles (BN = 128 or 256);
// for M > 128, CTA pairs share 256 x BN tiles through cta_group::2 MMAs.
// Warp roles (320 threads):
//   warp 0      one thread issues TMA loads of A and B K-slices (64 bf16 =
//               128 bytes deep, 128-byte swizzle) into a STAGES-deep ring;
//   warp 1      allocates 2*BN TMEM columns (two accumulators) and one thread
//               issues tcgen05.mma (M = 128, N = BN, K = 16 per instruction);
//               tcgen05.commit frees a ring slot once its MMAs are done and
//               hands a finished accumulator to the epilogue;
//   warps 2..9  read the accumulator (TMEM lane = output row; a warp may only
//               touch lanes 32*(warp % 4) .. +31; two warps share a lane
//               quarter and split its columns), apply the epilogue and store.
// The accumulator is double-buffered so the epilogue of tile t overlaps the
// main loop of tile t+1.  Operands may be K-major or MN-major; MN-major tiles
// are loaded as 64-element-wide chunks and described with LBO = chunk stride.
//
// The row-parallel GEMM (F_j) of a segment contracts over all w shards'
// K-slices into one accumulator: that is the on-chip form of the AllReduce
// y = sum_k P_k of Oases §IV, Eq. (1).
//
// Every mbarrier wait is bounded (2 s); on expiry the thread records an error
// in g_gemm_error, drains what it has in flight and leaves, so the kernel
// always terminates.
#include <cuda.h>

#include <mutex>
#include <unordered_map>

#include "epilogue.cuh"
#include "sm100_ptx.cuh"

namespace oases {

__device__ int g_gemm_error;
// Optional timeline (debugging aid, off when null): per CTA 16 globaltimer
// stamps: [0] entry, [1] after the prologue, [2] first stage landed (MMA
// thread), [3 + 2t] MMAs of local tile t done, [4 + 2t] its epilogue done
// (t < 5), [15] exit.
__device__ unsigned long long* g_gemm_timeline;

namespace {

constexpr int BM = 128;
constexpr int BKE = 64;  // K elements per stage (128 bytes of bf16)
constexpr int GROUP_M = 8;  // row blocks per group of the tile order when A is large
constexpr int64_t A_L2_BYTES = 48ll << 20;  // A up to this size stays in L2 across tile rounds
constexpr int NTHREADS = 320;  // 2 control warps + 8 epilogue warps

// CL = 2: a CTA pair shares each MMA; a CTA holds BN / 2 rows of the B tile.
// MX: E4M3 operands (128 elements = 128 bytes of K per stage, the same bytes
// as 64 bf16) and, per stage, the A and B scale tiles (128 rows x 4 K blocks,
// 512 bytes each), which the MMA thread copies into TMEM columns
// SF_COL0 + 8 * stage (A) and + 4 (B).
template <int BN, int CL, bool MX = false>
struct TcCfg {
  static constexpr int KE = MX ? 128 : BKE;  // K elements per stage
  static constexpr int A_BYTES = BM * 128;
  static constexpr int B_BYTES = BN / CL * 128;
  static constexpr int SF_BYTES = MX ? 512 + BN * 4 : 0;
  static constexpr int STAGE = A_BYTES + B_BYTES + SF_BYTES;
  static constexpr int STAGES = (192 * 1024) / STAGE;
  static constexpr int EPI_OFF = STAGES * STAGE;        // per epilogue warp: 32 rows x 128 B
  static constexpr int EPI_BYTES = 8 * 32 * 128;
  static constexpr int BAR_BYTES = 8 * (2 * STAGES + 5) + 8;
  static constexpr int SMEM = STAGES * STAGE + EPI_BYTES + BAR_BYTES + 1024;
  static constexpr int SF_COL0 = 2 * BN;
  static constexpr int TMEM_COLS = MX ? 512 : 2 * BN;
  static_assert(!MX || (BN == 128 && CL == 1), "the MX path takes 128 x 128 single-CTA tiles");
  static_assert(!MX || SF_COL0 + 8 * STAGES <= TMEM_COLS, "MX scale ring exceeds TMEM");
  static_assert(STAGE % 1024 == 0, "stages keep the 1024-byte alignment of swizzled tiles");
};

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ void unpack8(uint4 u, float* f) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 t = __bfloat1622float2(h[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
__device__ __forceinline__ void load32_bf16(const void* p, float* f) {
  const uint4* q = static_cast<const uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i) unpack8(__ldg(q + i), f + 8 * i);
}
__device__ __forceinline__ void store32_bf16(void* p, const float* f) {
  uint4* q = static_cast<uint4*>(p);
#pragma unroll
  for (int i = 0; i < 4; ++i)
    q[i] = make_uint4(pack_bf16(f[8 * i], f[8 * i + 1]), pack_bf16(f[8 * i + 2], f[8 * i + 3]),
                      pack_bf16(f[8 * i + 4], f[8 * i + 5]), pack_bf16(f[8 * i + 6], f[8 * i + 7]));
}

// Epilogue of 32 consecutive outputs (m, n .. n+31) held in v.
__device__ __forceinline__ void epi_chunk(const GemmArgs& g, int m, int n, float (&v)[32]) {
  const bool vec = (n + 32 <= g.N) && g.in_t == DType::BF16 &&
                   (g.c_t == DType::BF16 ? (g.ldc % 8 == 0) : (g.ldc % 4 == 0)) &&
                   (g.aux == nullptr || (g.ld_aux % 8 == 0 && g.aux_t == DType::BF16)) &&
                   (((uintptr_t)g.C | (uintptr_t)g.C2 | (uintptr_t)g.aux | (uintptr_t)g.bias) & 15) == 0;
  if (!vec) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (n + i < g.N) epi_apply(g, m, n + i, v[i]);
    return;
  }
  const int64_t ci = (int64_t)m * g.ldc + n;
  if (g.epi == Epi::Accum) {
    float4* c = reinterpret_cast<float4*>(static_cast<float*>(g.C) + ci);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      float4 o = c[i];
      o.x += v[4 * i];
      o.y += v[4 * i + 1];
      o.z += v[4 * i + 2];
      o.w += v[4 * i + 3];
      c[i] = o;
    }
    return;
  }
  float t[32];
  if (g.epi == Epi::Bias || g.epi == Epi::BiasGelu || g.epi == Epi::BiasResid) {
    load32_bf16(static_cast<const __nv_bfloat16*>(g.bias) + n, t);
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] += t[i];
  }
  if (g.epi == Epi::BiasResid || g.epi == Epi::Mul) {
    load32_bf16(static_cast<const __nv_bfloat16*>(g.aux) + (int64_t)m * g.ld_aux + n, t);
    if (g.epi == Epi::BiasResid) {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] += t[i];
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= t[i];
    }
  }
  if (g.epi == Epi::BiasGelu) {
    if (g.C2) {
      float d[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) d[i] = gelu_grad_f(v[i]);
      if (g.c_t == DType::BF16) store32_bf16(static_cast<__nv_bfloat16*>(g.C2) + ci, d);
      else {
        float4* c = reinterpret_cast<float4*>(static_cast<float*>(g.C2) + ci);
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = make_float4(d[4 * i], d[4 * i + 1], d[4 * i + 2], d[4 * i + 3]);
      }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = gelu_f(v[i]);
  }
  if (g.c_t == DType::BF16) {
    store32_bf16(static_cast<__nv_bfloat16*>(g.C) + ci, v);
  } else {
    float4* c = reinterpret_cast<float4*>(static_cast<float*>(g.C) + ci);
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
  }
}

// Epilogue through shared memory and TMA: the warp's 32 rows x CW columns
// (CW * element size = 128 bytes) are written into its 128-byte-swizzled
// staging buffer, one row per lane, then lane 0 stores the box with one TMA
// store (or fp32 reduce-add for Accum).  The TMA unit clips rows >= M and
// columns >= N.  v holds this lane's CW accumulator values for row m.
template <int CW>
__device__ __forceinline__ void epi_tma_chunk(const GemmArgs& g, const CUtensorMap* tmC,
                                              const CUtensorMap* tmC2, uint8_t* stg,
                                              uint32_t stg_s, int m, int mw, int n, int z,
                                              int lane, float (&v)[CW], float* rowdot = nullptr) {
  const bool bf = g.c_t == DType::BF16;
  if (g.epi == Epi::Bias || g.epi == Epi::BiasGelu || g.epi == Epi::BiasResid) {
    const __nv_bfloat16* b = static_cast<const __nv_bfloat16*>(g.bias) + n;
    if (n + CW <= g.N) {
#pragma unroll
      for (int i = 0; i < CW / 8; ++i) {
        float t[8];
        unpack8(__ldg(reinterpret_cast<const uint4*>(b) + i), t);
#pragma unroll
        for (int k = 0; k < 8; k += 2) add2_inplace(v[8 * i + k], v[8 * i + k + 1], t[k], t[k + 1]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < CW; ++i)
        if (n + i < g.N) v[i] += __bfloat162float(b[i]);
    }
  }
  if ((g.epi == Epi::BiasResid || g.epi == Epi::Mul) && m < g.M) {
    const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(g.aux) + (int64_t)m * g.ld_aux + n;
    float t[CW];
    if (n + CW <= g.N) {
#pragma unroll
      for (int i = 0; i < CW / 8; ++i) unpack8(__ldg(reinterpret_cast<const uint4*>(x) + i), t + 8 * i);
    } else {
#pragma unroll
      for (int i = 0; i < CW; ++i) t[i] = n + i < g.N ? __bfloat162float(x[i]) : 0.f;
    }
    if (g.epi == Epi::BiasResid) {
#pragma unroll
      for (int i = 0; i < CW; i += 2) add2_inplace(v[i], v[i + 1], t[i], t[i + 1]);
    } else {
#pragma unroll
      for (int i = 0; i < CW; i += 2) {
        const uint64_t r = f2_mul(f2_pack(v[i], v[i + 1]), f2_pack(t[i], t[i + 1]));
        v[i] = f2_lo(r);
        v[i + 1] = f2_hi(r);
      }
    }
  }
  // one staged store of v (as stored in C's type) to the box at (n, mw)
  auto stage_and_store = [&](const CUtensorMap* tm, bool reduce) {
    if (lane == 0) ptx::bulk_wait_read0();  // the previous store has read the buffer
    __syncwarp();
    uint8_t* row = stg + lane * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      uint4 w;
      if (bf) {
        w = make_uint4(pack_bf16(v[8 * u], v[8 * u + 1]), pack_bf16(v[8 * u + 2], v[8 * u + 3]),
                       pack_bf16(v[8 * u + 4], v[8 * u + 5]), pack_bf16(v[8 * u + 6], v[8 * u + 7]));
      } else {
        w = make_uint4(__float_as_uint(v[4 * u]), __float_as_uint(v[4 * u + 1]),
                       __float_as_uint(v[4 * u + 2]), __float_as_uint(v[4 * u + 3]));
      }
      *reinterpret_cast<uint4*>(row + ((u ^ (lane & 7)) << 4)) = w;
    }
    ptx::fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (reduce)
        ptx::tma_reduce_add_2d(tm, stg_s, n, mw);
      else if (g.splits > 1)
        ptx::tma_store_3d(tm, stg_s, n, mw, z);
      else
        ptx::tma_store_2d(tm, stg_s, n, mw);
      ptx::bulk_commit();
    }
  };
  if (g.epi == Epi::BiasGelu && g.C2) {
    // v becomes gelu(v); gelu'(v) is packed straight into the staging buffer
    // 16 bytes at a time and stored through C2 before v is staged for C
    if (lane == 0) ptx::bulk_wait_read0();  // the previous store has read the buffer
    __syncwarp();
    uint8_t* row = stg + lane * 128;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      constexpr int E = CW / 8;  // elements per 16-byte unit
      float d[E];
#pragma unroll
      for (int i = 0; i < E; i += 2) gelu_and_grad2(v[E * u + i], v[E * u + i + 1], d[i], d[i + 1]);
      uint4 w;
      if constexpr (E == 8) {  // bf16 output
        w = make_uint4(pack_bf16(d[0], d[1]), pack_bf16(d[2], d[3]), pack_bf16(d[4], d[5]),
                       pack_bf16(d[6], d[7]));
      } else {  // fp32 output
        w = make_uint4(__float_as_uint(d[0]), __float_as_uint(d[1]), __float_as_uint(d[2]),
                       __float_as_uint(d[3]));
      }
      *reinterpret_cast<uint4*>(row + ((u ^ (lane & 7)) << 4)) = w;
    }
    ptx::fence_async_smem();
    __syncwarp();
    if (lane == 0) {
      ptx::tma_store_2d(tmC2, stg_s, n, mw);
      ptx::bulk_commit();
    }
  } else if (g.epi == Epi::BiasGelu) {
#pragma unroll
    for (int i = 0; i < CW; i += 2) gelu2_inplace(v[i], v[i + 1]);
  }
  stage_and_store(tmC, g.epi == Epi::Accum);
  if constexpr (CW == 64) {
    if (g.colsum_part != nullptr) {
      // this warp's 32 rows of the 64 columns as stored: each lane reads its
      // own row back from the staging buffer (bf16, 16-byte chunk u at
      // u ^ (lane & 7)), and a butterfly of 31 shuffles per 32 columns leaves
      // lane l with column n + 32 h + l of the slab's partial row
      const uint8_t* row = stg + lane * 128;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float x[32];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const uint4 w = *reinterpret_cast<const uint4*>(row + (((4 * h + u) ^ (lane & 7)) << 4));
          unpack8(w, x + 8 * u);
        }
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (!(m < g.M && n + 32 * h + i < g.N)) x[i] = 0.f;
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) {
          const bool upper = (lane & off) != 0;
#pragma unroll
          for (int i = 0; i < off; ++i) {
            const float send = upper ? x[i] : x[i + off];
            x[i] = (upper ? x[i + off] : x[i]) + __shfl_xor_sync(0xffffffffu, send, off);
          }
        }
        if (n + 32 * h + lane < g.N) g.colsum_part[(int64_t)(mw / 32) * g.N + n + 32 * h + lane] = x[0];
      }
    }
    if (rowdot != nullptr && m < g.M) {
      // this lane's row of the 64 columns as stored (read back from the
      // staging buffer) times the same row and columns of rowdot_aux
      const uint8_t* row = stg + lane * 128;
      const __nv_bfloat16* ax = static_cast<const __nv_bfloat16*>(g.rowdot_aux) + (int64_t)m * g.rowdot_lda + n;
      float acc = 0.f;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (n + 8 * u >= g.N) break;
        float c[8], o[8];
        unpack8(*reinterpret_cast<const uint4*>(row + ((u ^ (lane & 7)) << 4)), c);
        unpack8(__ldg(reinterpret_cast<const uint4*>(ax) + u), o);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc = fmaf(c[i], o[i], acc);
      }
      *rowdot += acc;
    }
  }
}

// CL = 1: one CTA per 128 x BN tile.  CL = 2: a CTA pair (cluster of two)
// takes a 256 x BN tile with M = 256 pair MMAs (cta_group::2) issued by the
// even CTA: CTA r loads A rows [128 r, 128 r + 128) and B rows [r BN/2, (r+1) BN/2)
// of the tile into its own shared memory and holds output rows 128 r .. in its
// TMEM, so per stage each SM stores and reads A + B/2 instead of A + B.  Both
// CTAs' loads complete on the even CTA's full barrier (it expects both byte
// counts); its commits arrive on both CTAs' empty and accumulator-full
// barriers; both CTAs' epilogue warps release an accumulator on the even CTA's
// barrier.
template <int BN, bool A_K, bool B_K, int CL, bool GRP, bool MX>
__global__ void __launch_bounds__(NTHREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmC2,
               const GemmArgs g) {
  using C = TcCfg<BN, CL, MX>;
  constexpr int BNH = BN / CL;  // B rows of the tile held by this CTA
  constexpr uint32_t IDESC = MX ? ptx::idesc_mx_e4m3(BM, BN)
                                : ptx::idesc_bf16_f32(BM * CL, BN, !A_K, !B_K);
  static_assert(!MX || (A_K && B_K), "MX operands are K-major");
  unsigned long long* tl = g_gemm_timeline ? g_gemm_timeline + 16 * blockIdx.x : nullptr;
  if (tl && threadIdx.x == 0) tl[0] = ptx::globaltimer();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = ptx::smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + C::EPI_OFF + C::EPI_BYTES;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (C::STAGES + s); };
  auto tfull = [&](int b) { return bars + 8u * (2 * C::STAGES + b); };
  auto tempty = [&](int b) { return bars + 8u * (2 * C::STAGES + 2 + b); };
  const uint32_t drain = bars + 8u * (2 * C::STAGES + 4);
  const uint32_t tslot = bars + 8u * (2 * C::STAGES + 5);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int rank = CL > 1 ? (int)ptx::cluster_rank() : 0;
  const int num_m = (g.M + BM - 1) / BM, num_n = (g.N + BN - 1) / BN;
  const int num_mp = (num_m + CL - 1) / CL;  // row blocks of CL * 128 rows
  // tiles of split s are [s * tiles1, (s + 1) * tiles1); K blocks walk the
  // pieces of that split's contraction range in order
  const int tiles1 = num_mp * num_n, tiles = tiles1 * g.splits;
  const int kpl = g.K / g.kpieces, nkb_p = (kpl + C::KE - 1) / C::KE, nkb = nkb_p * g.kpieces;
  const int first = blockIdx.x / CL, stride = gridDim.x / CL;
  // Tile order within a split: the row block varies fastest.  Without GRP it
  // does so over every row block: each round of tiles re-reads A from L2 and
  // B comes from DRAM once, which holds while all of A fits in L2.  A larger
  // A (dW1 += dA^T u: 64 row blocks, 128 MB) would then be streamed from DRAM
  // again for every column block, so with GRP the tiles go in groups of
  // GROUP_M row blocks: the tiles in flight share GROUP_M row blocks of A and
  // a few column blocks of B, and B is read once per group.
  auto tile_split = [&](int t) { return t / tiles1; };
  auto tile_mb = [&](int t) {
    const int r = t % tiles1;
    if constexpr (!GRP) {
      return r % num_mp;
    } else {
      const int q = r / (GROUP_M * num_n), gm = min(GROUP_M, num_mp - q * GROUP_M);
      return q * GROUP_M + (r - q * GROUP_M * num_n) % gm;
    }
  };
  auto tile_nb = [&](int t) {
    const int r = t % tiles1;
    if constexpr (!GRP) {
      return r / num_mp;
    } else {
      const int q = r / (GROUP_M * num_n), gm = min(GROUP_M, num_mp - q * GROUP_M);
      return (r - q * GROUP_M * num_n) / gm;
    }
  };
  auto tile_m0 = [&](int t) { return (tile_mb(t) * CL + rank) * BM; };
  auto tile_n0 = [&](int t) { return tile_nb(t) * BN; };
  constexpr uint16_t MASK = (1u << CL) - 1u;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      ptx::mbar_init(full(s), 1);
      ptx::mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(tfull(b), 1);
      ptx::mbar_init(tempty(b), 8 * CL);  // one arrival per epilogue warp of the pair
    }
    ptx::mbar_init(drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    if (CL > 1) {
      ptx::tmem_alloc_pair(tslot, C::TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(tslot, C::TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  if (warp == 0 && lane == 0) {
    ptx::prefetch_tmap(&tmA);
    ptx::prefetch_tmap(&tmB);
    if (g.tma_store) {
      ptx::prefetch_tmap(&tmC);
      if (g.C2) ptx::prefetch_tmap(&tmC2);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gbase + (tslot - base));
  if (CL > 1) ptx::cluster_sync();  // partner's barriers initialised before any cross-CTA arrival
  // Everything above touched only shared memory, TMEM and kernel parameters, so
  // it overlapped the previous kernel on the stream; global memory from here on.
  pdl_wait();
  pdl_trigger();
  if (tl && threadIdx.x == 0) tl[1] = ptx::globaltimer();

  if (warp == 0) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      uint32_t issued = 0;  // bit s: stage s has a load outstanding at some phase
      uint32_t iphase = 0;  // bit s: parity of the last load issued into stage s
      for (int tile = first; tile < tiles && ok; tile += stride) {
        const int m0 = tile_m0(tile), n0 = tile_n0(tile), ks = tile_split(tile) * kpl;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ptx::mbar_wait(empty(stage), phase ^ 1u)) { ok = false; break; }
          // the pair's loads complete on the even CTA's barrier, which expects both
          const uint32_t fb = CL > 1 ? ptx::mapa(full(stage), 0) : full(stage);
          if (rank == 0) ptx::mbar_arrive_expect_tx(full(stage), CL * C::STAGE);
          auto load = [&](uint32_t dst, const CUtensorMap* tm, int x, int y) {
            if (CL > 1)
              ptx::tma_load_2d_pair(dst, tm, fb, x, y);
            else
              ptx::tma_load_2d(dst, tm, fb, x, y);
          };
          const uint32_t sa = base + stage * C::STAGE, sb = sa + C::A_BYTES;
          const int pc = kb / nkb_p;
          const int k0 = (int)(pc * g.kpiece_stride) + ks + (kb - pc * nkb_p) * C::KE;
          if constexpr (MX) {  // the stage's scale tiles (K group kb)
            const uint32_t ssf = sb + C::B_BYTES;
            ptx::bulk_load(ssf, g.a_sf + ((int64_t)(m0 / BM) * nkb + kb) * 512, 512, fb);
            ptx::bulk_load(ssf + 512, g.b_sf + ((int64_t)(n0 / 128) * nkb + kb) * 512, 512, fb);
          }
          if (A_K) {
            load(sa, &tmA, k0, m0);
          } else {
            load(sa, &tmA, m0, k0);
            load(sa + 8192, &tmA, m0 + 64, k0);
          }
          const int nb = n0 + rank * BNH;  // this CTA's B rows
          if (B_K) {
            load(sb, &tmB, k0, nb);
          } else {
#pragma unroll
            for (int c = 0; c < BNH / 64; ++c) load(sb + c * 8192, &tmB, nb + 64 * c, k0);
          }
          issued |= 1u << stage;
          iphase = (iphase & ~(1u << stage)) | (phase << stage);
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
      }
      // Drain: every TMA load this thread issued has landed before the CTA exits
      // (the odd CTA of a pair sees that through the release of each stage).
      for (int s = 0; s < C::STAGES; ++s)
        if ((issued >> s) & 1u)
          if (!ptx::mbar_wait(rank == 0 ? full(s) : empty(s), (iphase >> s) & 1u)) ok = false;
      if (!ok) atomicExch(&g_gemm_error, 1);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {  // the even CTA issues the pair's MMAs
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      int t = 0;
      for (int tile = first; tile < tiles && ok; tile += stride, ++t) {
        const int buf = t & 1;
        if (!ptx::mbar_wait(tempty(buf), (((uint32_t)t >> 1) & 1u) ^ 1u)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t dt = tmem + (uint32_t)(buf * BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ptx::mbar_wait(full(stage), phase)) { ok = false; break; }
          ptx::tc_fence_after();
          if (tl && t == 0 && kb == 0) tl[2] = ptx::globaltimer();
          const uint32_t sa = base + stage * C::STAGE, sb = sa + C::A_BYTES;
          if constexpr (MX) {
            // scale tiles -> TMEM (ordered before the MMAs below, which read them),
            // then four K = 32 MMAs, each with its K block's scale byte
            const uint32_t ssf = sb + C::B_BYTES;
            const uint32_t tsa = tmem + (uint32_t)(C::SF_COL0 + 8 * stage), tsb = tsa + 4;
            ptx::tmem_cp_32x128b_x4(tsa, ptx::smem_desc_noswz(ssf, 128, 128));
            ptx::tmem_cp_32x128b_x4(tsb, ptx::smem_desc_noswz(ssf + 512, 128, 128));
            const uint64_t ad0 = ptx::smem_desc_sw128(sa, 16, 1024), bd0 = ptx::smem_desc_sw128(sb, 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // start address += 32 bytes per K = 32 step
              ptx::mma_mx(dt, ad0 + 2 * kk, bd0 + 2 * kk, IDESC | ptx::idesc_sf_ids(kk, kk), tsa, tsb,
                          (kb | kk) != 0 ? 1u : 0u);
          } else {
            // descriptors formed once per stage; the start-address field (16-byte
            // units, shared addresses < 2^18) is stepped per K = 16 MMA
            const uint64_t ad0 = A_K ? ptx::smem_desc_sw128(sa, 16, 1024) : ptx::smem_desc_sw128(sa, 8192, 1024);
            const uint64_t bd0 = B_K ? ptx::smem_desc_sw128(sb, 16, 1024) : ptx::smem_desc_sw128(sb, 8192, 1024);
#pragma unroll
            for (int kk = 0; kk < BKE / 16; ++kk) {
              const uint64_t ad = ad0 + (uint64_t)(A_K ? 2 * kk : 128 * kk);
              const uint64_t bd = bd0 + (uint64_t)(B_K ? 2 * kk : 128 * kk);
              if (CL > 1)
                ptx::mma_bf16_pair(dt, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
              else
                ptx::mma_bf16(dt, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          if (CL > 1)
            ptx::mma_commit_pair_mc(empty(stage), MASK);
          else
            ptx::mma_commit(empty(stage));
          if (++stage == C::STAGES) { stage = 0; phase ^= 1u; }
        }
        if (!ok) break;
        if (CL > 1)
          ptx::mma_commit_pair_mc(tfull(buf), MASK);
        else
          ptx::mma_commit(tfull(buf));
        if (tl && t < 5) tl[3 + 2 * t] = ptx::globaltimer();
      }
      // Drain: all MMAs issued by this thread are complete before TMEM is freed.
      if (CL > 1)
        ptx::mma_commit_pair(drain);
      else
        ptx::mma_commit(drain);
      if (!ptx::mbar_wait(drain, 0)) ok = false;
      if (!ok) atomicExch(&g_gemm_error, 2);
    }
  } else {
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;  // which half of the BN columns
    int t = 0;
    for (int tile = first; tile < tiles; tile += stride, ++t) {
      const int buf = t & 1;
      // the decision is warp-uniform: tcgen05.ld below is warp-collective
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(tfull(buf), ((uint32_t)t >> 1) & 1u))) {
        if (lane == 0) atomicExch(&g_gemm_error, 3);
        break;
      }
      ptx::tc_fence_after();
      const int mw = tile_m0(tile) + q * 32, m = mw + lane;
      const int nb0 = tile_n0(tile), z = tile_split(tile);
      const uint32_t trow = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(buf * BN);
      if (g.tma_store && g.c_t == DType::BF16) {
        uint8_t* stg = gbase + C::EPI_OFF + (warp - 2) * 4096;
        const uint32_t stg_s = base + C::EPI_OFF + (warp - 2) * 4096;
        float rd = 0.f;  // rowdot: this half of a 256-wide tile is one 128-column group
#pragma unroll 1
        for (int c0 = half * (BN / 2); c0 < (half + 1) * (BN / 2); c0 += 64) {
          float v[64];
          ptx::tmem_ld32(trow + c0, *reinterpret_cast<float(*)[32]>(v));
          ptx::tmem_ld32(trow + c0 + 32, *reinterpret_cast<float(*)[32]>(v + 32));
          if (mw < g.M && nb0 + c0 < g.N)
            epi_tma_chunk<64>(g, &tmC, &tmC2, stg, stg_s, m, mw, nb0 + c0, z, lane, v,
                              g.rowdot_out != nullptr ? &rd : nullptr);
        }
        if (g.rowdot_out != nullptr && m < g.M && nb0 + half * (BN / 2) < g.N)
          g.rowdot_out[(int64_t)((nb0 + half * (BN / 2)) / 128) * g.rowdot_ld + m] = rd;
      } else if (g.tma_store) {
        uint8_t* stg = gbase + C::EPI_OFF + (warp - 2) * 4096;
        const uint32_t stg_s = base + C::EPI_OFF + (warp - 2) * 4096;
#pragma unroll 1
        for (int c0 = half * (BN / 2); c0 < (half + 1) * (BN / 2); c0 += 32) {
          float v[32];
          ptx::tmem_ld32(trow + c0, v);
          if (mw < g.M && nb0 + c0 < g.N)
            epi_tma_chunk<32>(g, &tmC, &tmC2, stg, stg_s, m, mw, nb0 + c0, z, lane, v);
        }
      } else {
#pragma unroll 1
        for (int c0 = half * (BN / 2); c0 < (half + 1) * (BN / 2); c0 += 32) {
          float v[32];
          ptx::tmem_ld32(trow + c0, v);
          if (m < g.M && nb0 + c0 < g.N) epi_chunk(g, m, nb0 + c0, v);
        }
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (CL > 1)
          ptx::mbar_arrive_cluster(ptx::mapa(tempty(buf), 0));
        else
          ptx::mbar_arrive(tempty(buf));
      }
      if (tl && t < 5 && warp == 2 && lane == 0) tl[4 + 2 * t] = ptx::globaltimer();
    }
    if (g.tma_store && lane == 0) ptx::bulk_wait0();  // stores performed before the CTA retires
  }
  ptx::tc_fence_before();
  __syncthreads();
  // the pair's MMAs (which write both CTAs' TMEM) and every cross-CTA arrival
  // are complete before either CTA frees TMEM or leaves
  if (CL > 1) ptx::cluster_sync();
  if (warp == 1) {
    ptx::tc_fence_after();
    if (CL > 1)
      ptx::tmem_dealloc_pair(tmem, C::TMEM_COLS);
    else
      ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
  if (CL > 1) ptx::cluster_sync();
  if (tl && threadIdx.x == 0) tl[15] = ptx::globaltimer();
}

// ---- host side -------------------------------------------------------------
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

struct MapKey {
  uintptr_t ptr;
  uint64_t inner, outer, ld, depth, ld2;
  uint32_t box_inner, box_outer;
  bool operator==(const MapKey& o) const {
    return ptr == o.ptr && inner == o.inner && outer == o.outer && ld == o.ld &&
           depth == o.depth && ld2 == o.ld2 && box_inner == o.box_inner &&
           box_outer == o.box_outer;
  }
};
struct MapKeyHash {
  size_t operator()(const MapKey& k) const {
    size_t h = k.ptr * 0x9E3779B97F4A7C15ull;
    h ^= k.inner + 0x9E37 + (h << 6) + (h >> 2);
    h ^= k.outer + 0x79B9 + (h << 6) + (h >> 2);
    h ^= k.ld + (h << 6) + (h >> 2);
    h ^= (k.depth * 0x100000001B3ull ^ k.ld2) + (h << 6) + (h >> 2);
    h ^= ((uint64_t)k.box_inner << 32 | k.box_outer) + (h << 6) + (h >> 2);
    return h;
  }
};

// 2-D bf16 (or fp32) tensor map over a row-major [outer, inner] matrix with
// leading dimension ld (elements), box [box_outer, box_inner], 128-byte
// swizzle, out-of-bounds elements read as zero.  depth > 1 adds a third
// dimension of `depth` such matrices, ld2 elements apart (box depth 1).
// Cached by its arguments.
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_map_cache;

enum class MapT : uint32_t { BF16 = 0, F32 = 1, U8 = 2 };

bool make_map(CUtensorMap* out, const void* ptr, uint64_t inner, uint64_t outer, uint64_t ld,
              uint32_t box_inner, uint32_t box_outer, MapT mt = MapT::BF16, uint64_t depth = 1,
              uint64_t ld2 = 0) {
  std::mutex& mu = g_map_mu;
  auto& cache = g_map_cache;
  if (depth < 1) depth = 1;
  // device pointers are 16-byte aligned: the low bits carry the element kind
  const MapKey key{(uintptr_t)ptr | (uintptr_t)mt, inner, outer, ld, depth,
                   depth > 1 ? ld2 : 0, box_inner, box_outer};
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return true;
  }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const uint64_t esz = mt == MapT::F32 ? 4 : mt == MapT::BF16 ? 2 : 1;
  const cuuint64_t dims[3] = {inner, outer, depth};
  const cuuint64_t strides[2] = {ld * esz, ld2 * esz};
  const cuuint32_t box[3] = {box_inner, box_outer, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMap m;
  const CUtensorMapDataType dt = mt == MapT::F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : mt == MapT::BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  if (fn(&m, dt, depth > 1 ? 3u : 2u,
         const_cast<void*>(ptr), dims, strides, box, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return false;
  if (cache.size() > 4096) cache.clear();
  cache.emplace(key, m);
  *out = m;
  return true;
}

int num_sms() {  // of the current device, cached per device
  static std::atomic<int> cache[64];
  const int dev = current_device();
  if (dev < 64) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (n <= 0) n = 1;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

template <int BN, bool A_K, bool B_K, int CL, bool GRP = false, bool MX = false>
cudaError_t launch_tc(const GemmArgs& g, cudaStream_t st) {
  using C = TcCfg<BN, CL, MX>;
  CUtensorMap ma, mb;
  const uint64_t kext = g.k_extent > 0 ? (uint64_t)g.k_extent : (uint64_t)g.K;
  bool ok;
  if constexpr (MX) {  // E4M3 codes: 128 elements (bytes) of K per box row
    ok = make_map(&ma, g.A, kext, g.M, g.lda, C::KE, BM, MapT::U8) &&
         make_map(&mb, g.B, kext, g.N, g.ldb, C::KE, BN, MapT::U8);
  } else {
    ok = A_K ? make_map(&ma, g.A, kext, g.M, g.lda, BKE, BM)
             : make_map(&ma, g.A, g.M, kext, g.lda, 64, BKE);
    ok = ok && (B_K ? make_map(&mb, g.B, kext, g.N, g.ldb, BKE, BN / CL)
                    : make_map(&mb, g.B, g.N, kext, g.ldb, 64, BKE));
  }
  if (!ok) return cudaErrorInvalidValue;
  // outputs through TMA stores when C (and C2) rows are 16-byte multiples
  GemmArgs ga = g;
  CUtensorMap mc = ma, mc2 = ma;
  const bool f32c = g.c_t == DType::F32;
  const int esz = f32c ? 4 : 2, cw = f32c ? 32 : 64;
  const bool aligned = ((g.ldc * esz) % 16 == 0) && (((uintptr_t)g.C | (uintptr_t)g.C2) & 15) == 0 &&
                       (((uintptr_t)g.bias | (uintptr_t)g.aux) & 15) == 0 &&
                       (g.aux == nullptr || (g.ld_aux % 8 == 0 && g.aux_t == DType::BF16));
  ga.tma_store = 0;
  const MapT ct = f32c ? MapT::F32 : MapT::BF16;
  if (aligned && make_map(&mc, g.C, g.N, g.M, g.ldc, cw, 32, ct, (uint64_t)g.splits,
                          (uint64_t)(g.c_split_rows * g.ldc)) &&
      (g.C2 == nullptr || make_map(&mc2, g.C2, g.N, g.M, g.ldc, cw, 32, ct)))
    ga.tma_store = 1;
  if (g.splits > 1 && !ga.tma_store) return cudaErrorNotSupported;  // slabs need the 3-D map
  // row dots only in the bf16 TMA-store epilogue of 256-wide tiles (a warp's
  // half of a tile is one 128-column group)
  if (ga.rowdot_out != nullptr) {
    if (BN == 256 && ga.tma_store && g.c_t == DType::BF16 && g.splits == 1 && g.epi != Epi::Accum &&
        g.N % 128 == 0 && g.rowdot_aux != nullptr && g.rowdot_lda % 8 == 0 && g.rowdot_ld >= g.M &&
        (((uintptr_t)g.rowdot_aux & 15) == 0) && (((uintptr_t)g.rowdot_out & 3) == 0)) {
      if (g.rowdot_done) *g.rowdot_done = 1;
    } else {
      ga.rowdot_out = nullptr;
    }
  }
  // column sums of C only in the bf16 TMA-store epilogue (64-column chunks)
  if (ga.colsum_part != nullptr) {
    if (ga.tma_store && g.c_t == DType::BF16 && g.splits == 1 && g.epi != Epi::Accum &&
        ((uintptr_t)g.colsum_part & 3) == 0) {
      if (g.colsum_rows) *g.colsum_rows = (g.M + 31) / 32;
    } else {
      ga.colsum_part = nullptr;
    }
  }
  auto kern = gemm_tc_kernel<BN, A_K, B_K, CL, GRP, MX>;
  static DeviceOnce attr;
  cudaError_t ea = attr.run([&] {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (ea != cudaSuccess) return ea;
  const int num_mp = ((g.M + BM - 1) / BM + CL - 1) / CL;
  const int tiles = num_mp * ((g.N + BN - 1) / BN) * g.splits;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = C::SMEM;
  cfg.stream = st;
  // persistent grid: as many clusters as can be resident at once (per device)
  static std::atomic<int> slots_by_dev[64];
  const int dev = current_device();
  int slots = dev < 64 ? slots_by_dev[dev].load(std::memory_order_relaxed) : 0;
  if (slots == 0) {
    slots = num_sms() / CL;
    if (CL > 1) {
      cudaLaunchAttribute ca[1];
      ca[0].id = cudaLaunchAttributeClusterDimension;
      ca[0].val.clusterDim.x = CL;
      ca[0].val.clusterDim.y = 1;
      ca[0].val.clusterDim.z = 1;
      cudaLaunchConfig_t q = cfg;
      q.gridDim = dim3(num_sms() / CL * CL);
      q.attrs = ca;
      q.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, kern, &q) == cudaSuccess && n > 0 && n < slots)
        slots = n;
      cudaGetLastError();
    }
    if (dev < 64) slots_by_dev[dev].store(slots, std::memory_order_relaxed);
  }
  // as few clusters as finish in the same number of tile rounds: the rest of
  // the SMs stay free for other streams' kernels at no cost to this one
  const int rounds = (tiles + slots - 1) / slots;
  const int grid = ((tiles + rounds - 1) / rounds) * CL;
  cfg.gridDim = dim3(grid);
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = CL;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.attrs = attrs;
  cfg.numAttrs = CL > 1 ? 2 : 1;
  ++g_launch_count;
  return cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, mc2, ga);
}

// The grouped tile order (the kernel's GRP): CTA-pair 256-wide tiles over more
// than GROUP_M row blocks, with an A operand too large to stay in L2.
bool grouped_order(const GemmArgs& g) {
  const int num_mp = ((g.M + BM - 1) / BM + 1) / 2;
  return num_mp > GROUP_M && (int64_t)g.M * g.K * 2 > A_L2_BYTES;
}

template <int BN, int CL>
cudaError_t dispatch_major(const GemmArgs& g, cudaStream_t st) {
  if constexpr (BN == 256 && CL == 2) {
    if (grouped_order(g)) {
      if (g.a_kmajor)
        return g.b_kmajor ? launch_tc<BN, true, true, CL, true>(g, st)
                          : launch_tc<BN, true, false, CL, true>(g, st);
      return g.b_kmajor ? launch_tc<BN, false, true, CL, true>(g, st)
                        : launch_tc<BN, false, false, CL, true>(g, st);
    }
  }
  if (g.a_kmajor)
    return g.b_kmajor ? launch_tc<BN, true, true, CL>(g, st) : launch_tc<BN, true, false, CL>(g, st);
  return g.b_kmajor ? launch_tc<BN, false, true, CL>(g, st) : launch_tc<BN, false, false, CL>(g, st);
}

}  // namespace

bool gemm_mx_supported(const GemmArgs& g) {
  if (g.in_t != DType::E4M3 || !g.a_kmajor || !g.b_kmajor) return false;
  if (g.M <= 0 || g.N <= 0 || g.K <= 0 || !g.a_sf || !g.b_sf) return false;
  if (g.splits != 1 || g.kpieces != 1 || g.k_extent != 0) return false;
  if (g.lda < g.K || g.ldb < g.K || g.lda % 16 != 0 || g.ldb % 16 != 0) return false;
  if ((((uintptr_t)g.A) | ((uintptr_t)g.B) | ((uintptr_t)g.a_sf) | ((uintptr_t)g.b_sf)) & 15)
    return false;
  if (g.epi == Epi::Accum && g.c_t != DType::F32) return false;
  if (g.c_t == DType::E4M3 || (g.aux && g.aux_t != DType::BF16)) return false;
  return encode_fn() != nullptr;
}

cudaError_t gemm_mx(const GemmArgs& g, cudaStream_t st) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  if (!gemm_mx_supported(g)) return cudaErrorNotSupported;
  return launch_tc<128, true, true, 1, false, true>(g, st);
}

bool gemm_tc_supported(const GemmArgs& g) {
  if (g.in_t != DType::BF16) return false;
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return false;
  if (g.lda % 8 != 0 || g.ldb % 8 != 0) return false;
  if ((((uintptr_t)g.A) | ((uintptr_t)g.B)) & 15) return false;
  if (g.epi == Epi::Accum && g.c_t != DType::F32) return false;
  if (g.splits < 1 || g.kpieces < 1 || g.K % g.kpieces != 0) return false;
  if (g.splits > 1 || g.kpieces > 1) {
    // every K block of a piece lies inside it; slabs are disjoint, 16-byte aligned
    const int64_t kpl = g.K / g.kpieces, esz = g.c_t == DType::F32 ? 4 : 2;
    if (g.epi != Epi::Store || kpl % BKE != 0 || g.k_extent <= 0) return false;
    if ((g.kpieces - 1) * g.kpiece_stride + (int64_t)g.splits * kpl > g.k_extent) return false;
    if (g.splits > 1 && (g.c_split_rows < g.M || (g.c_split_rows * g.ldc * esz) % 16 != 0 ||
                         (g.ldc * esz) % 16 != 0 || ((uintptr_t)g.C & 15) != 0))
      return false;
  }
  return encode_fn() != nullptr;
}

cudaError_t gemm_tc(const GemmArgs& g, cudaStream_t st) {
  if (!gemm_tc_supported(g)) return cudaErrorNotSupported;
  const int tiles256 = ((g.M + BM - 1) / BM) * ((g.N + 255) / 256) * g.splits;
  const bool pair = g.M > BM;  // a second row block exists for the cluster partner
  // Pair MMAs with N = 128 move 1.5x the operand bytes per FLOP of N = 256
  // and run at about half its rate: the pair path takes 256-wide tiles unless
  // that would leave more than half of the SMs idle with nothing else to run.
  const bool narrow = pair ? (g.N <= 128 || (!g.concurrent && 2 * tiles256 < num_sms()))
                           : (g.N <= 128 || tiles256 < num_sms());
  if (narrow)
    return pair ? dispatch_major<128, 2>(g, st) : dispatch_major<128, 1>(g, st);
  return pair ? dispatch_major<256, 2>(g, st) : dispatch_major<256, 1>(g, st);
}

cudaError_t gemm(const GemmArgs& g, cudaStream_t st) {
  if (g.M == 0 || g.N == 0) return cudaSuccess;
  if (g.in_t == DType::E4M3) return gemm_mx(g, st);  // the MX path or nothing
  if (gemm_tc_supported(g)) return gemm_tc(g, st);
  if (g.splits != 1 || g.kpieces != 1) return cudaErrorNotSupported;  // tensor-core path only
  return gemm_simt(g, st);
}

void gemm_release_host_caches() {
  std::lock_guard<std::mutex> lock(g_map_mu);
  g_map_cache.clear();
}

cudaError_t gemm_set_timeline(unsigned long long* p) {
  return cudaMemcpyToSymbol(g_gemm_timeline, &p, sizeof(p));
}

int gemm_read_and_clear_error() {
  int v = 0, z = 0;
  if (cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(int)) != cudaSuccess) return -1;
  if (v) cudaMemcpyToSymbol(g_gemm_error, &z, sizeof(int));
  return v;
}

}  // namespace oases
