// C ABI and two-stream sub-batch scheduler of the Oases block library.
//
// The scheduler turns a call into the operator schedule of Oases §IV,
// Algorithm 1 — a list of steps (event, operator, segment, sub-batch) — and
// then executes every step by enqueueing its kernels on stream (sub-batch % 2):
//
//   forward    for every segment s, for every sub-batch b:
//                F(ln) F(col) F(row) C(F)       C(F) is fused into the row GEMM:
//                                              it contracts over all w shards'
//                                              K-slices into one accumulator
//   backward   for every segment s in reverse, for every sub-batch b:
//                Sync  B(ln) of the later segment  (its input-gradient sum is done)
//                R(ln) R(col) [R(row) C(R) in FULL mode]
//                B(g)  B(row)  B(col)  C(B)
//              and finally Sync B(ln) of segment 0.
//
// Because sub-batch b always runs on the same stream, a Sync needs no event:
// stream order already places it after the sub-batch's own reduction.  The
// other sub-batch's stream runs meanwhile, which is the pages' overlap of one
// sub-batch's reduction with the other's compute (Fig. 4b, Fig. 4d).  The only
// cross-stream dependencies are the weight-gradient accumulations, which are
// chained sub-batch 0 -> 1 -> ... per (segment, parameter) with events so the
// sums are taken in a fixed order.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <string>
#include <functional>
#include <vector>

#include "common.cuh"
#include "oases.h"

namespace oases {
int norm_read_and_clear_error();  // norm.cu: a LayerNorm kernel's wait gave up
cudaError_t layer_norm_bwd_dx_colsum(const float* du, const void* x, const float* mean,
                                     const float* rstd, const void* gamma, const void* dres, void* dx,
                                     float* part_g, float* part_b, float2* stat, float* dgamma,
                                     float* dbeta, int M, int H, DType t, cudaStream_t st,
                                     float* part_x, int part_x_cap, int* n_part_x, float* out_x,
                                     const std::function<void(bool)>* before_reduce);
cudaError_t reduce_partial_rows(float* part, float* out, int nparts, int N, cudaStream_t st);
// attn_tc.cu: the tensor-core attention backward that also leaves the QKV
// bias gradient's partial rows (batch * ceil(seq / 128) * 4 rows of 3H)
cudaError_t attention_bwd_tc_bias(const AttnArgs& a, float* bias_part, cudaStream_t st);
thread_local int g_launch_count = 0;

uint64_t current_ctx_id() {
  typedef CUresult (*GetCurrentFn)(CUcontext*);
  typedef CUresult (*GetIdFn)(CUcontext, unsigned long long*);
  static GetCurrentFn get_current = nullptr;
  static GetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<GetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<GetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext c = nullptr;
  if (get_current(&c) != CUDA_SUCCESS) return 0;
  if (!c) {
    // no context bound to this thread yet: cudaSetDevice binds (and, if need
    // be, creates) the current device's primary context
    int d = 0;
    if (cudaGetDevice(&d) != cudaSuccess || cudaSetDevice(d) != cudaSuccess) return 0;
    if (get_current(&c) != CUDA_SUCCESS || !c) return 0;
  }
  unsigned long long id = 0;
  return get_id(c, &id) == CUDA_SUCCESS ? (uint64_t)id : 0;
}
}  // namespace oases

namespace oases {
// Entry-point bookkeeping shared with the other translation units that define
// extern "C" functions: reset per call, record a CUDA or argument error.
void api_begin();
void api_set_error(const char* what);
oases_status api_end(cudaError_t e);
// Host caches of the other translation units, emptied by oases_shutdown().
void gemm_release_host_caches();
void noalloc_release_host_caches();
}

namespace {
using namespace oases;

thread_local std::string t_last_error;
thread_local int t_last_launches = 0;

// Optional per-operator event timeline of this thread's last call (debugging
// aid); its events are kept per device and reused across calls.
struct TraceRec {
  int ev, op, seg, sb;
  cudaEvent_t e0, e1;
};
struct TraceEvents {
  uint64_t ctx = 0;  // context the events belong to
  std::vector<cudaEvent_t> ev;
  void release() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    ev.clear();
  }
  ~TraceEvents() { release(); }
};
std::atomic<bool> g_trace_on{false};
thread_local std::vector<TraceRec> g_trace;
thread_local std::unordered_map<int, TraceEvents> g_trace_events;

enum Ev { EV_F = 0, EV_R = 1, EV_B = 2, EV_CF = 3, EV_CR = 4, EV_CB = 5, EV_SYNC = 6 };
enum OpN { OP_LN = 0, OP_F = 1, OP_COL = 2, OP_ROW = 3, OP_G = 4, OP_ATTN = 5 };
enum SegKind { SEG_FFN = 0, SEG_ATTN = 1 };
// Weight-gradient groups of one segment, each accumulated in sub-batch order.
enum Grp { GRP_BR = 0, GRP_WR = 1, GRP_BC = 2, GRP_WC = 3, GRP_LN = 4, GRP_N = 5 };

struct Step {
  int ev, op, seg, sb;
};

struct Shape {
  int kind, B, S, H, F, nh, d, w, nsb, pre_ln, residual, causal, mode, reduce;
  DType t;
  bool mx;  // MX-FP8 GEMM operands (bf16 storage)
  float eps;
  int64_t M, Ms;
  size_t esz;
  int segs_per_layer, nseg;
  int seg_kind(int s) const {
    if (kind == OASES_BLOCK_LAYER) return (s % 2 == 0) ? SEG_ATTN : SEG_FFN;
    return kind == OASES_BLOCK_ATTN ? SEG_ATTN : SEG_FFN;
  }
};

oases_status validate(const oases_block_desc* d, int n_layers, Shape* s) {
  if (!d || n_layers < 1) return OASES_ERR_INVALID_ARG;
  if (d->kind < 0 || d->kind > 2 || d->dtype < 0 || d->dtype > 2) return OASES_ERR_INVALID_ARG;
  if (d->batch < 0 || d->seq < 0 || d->hidden <= 0 || d->w < 1 || d->sub_batches < 1)
    return OASES_ERR_INVALID_ARG;
  if (d->batch % d->sub_batches != 0) return OASES_ERR_INVALID_ARG;
  if (d->recompute < 0 || d->recompute > 3) return OASES_ERR_INVALID_ARG;
  if (d->reduce < 0 || d->reduce > 1) return OASES_ERR_INVALID_ARG;
  if (!(d->ln_eps >= 0.f)) return OASES_ERR_INVALID_ARG;
  const bool has_ffn = d->kind != OASES_BLOCK_ATTN, has_attn = d->kind != OASES_BLOCK_FFN;
  if (has_ffn && (d->ffn <= 0 || d->ffn % d->w != 0)) return OASES_ERR_INVALID_ARG;
  if (has_attn) {
    if (d->heads <= 0 || d->hidden % d->heads != 0 || d->heads % d->w != 0)
      return OASES_ERR_INVALID_ARG;
    const int hd = d->hidden / d->heads;
    if (hd > 128 || hd % 8 != 0) return OASES_ERR_UNSUPPORTED;
  }
  if (d->dtype == OASES_BF16 && (d->hidden % 8 != 0 || (has_ffn && d->ffn % 8 != 0)))
    return OASES_ERR_UNSUPPORTED;
  // MX-FP8: scale blocks of 32 along every contraction must not straddle a
  // shard's slice (so the shard sum of Eq. (1) is the full-width product), and
  // the shard partials exist only inside the fused GEMMs
  if (d->dtype == OASES_MXFP8 &&
      (d->hidden % 32 != 0 || (has_ffn && (d->ffn / d->w) % 32 != 0) ||
       (has_attn && (d->hidden / d->w) % 32 != 0) || d->reduce != OASES_REDUCE_FUSED))
    return OASES_ERR_UNSUPPORTED;
  const int64_t M = (int64_t)d->batch * d->seq;
  const int64_t widest = has_ffn ? (d->ffn > 3 * d->hidden ? d->ffn : 3 * (int64_t)d->hidden)
                                 : 3 * (int64_t)d->hidden;
  if (M > (1ll << 30) || widest > (1ll << 30)) return OASES_ERR_UNSUPPORTED;
  s->kind = d->kind;
  s->B = d->batch;
  s->S = d->seq;
  s->H = d->hidden;
  s->F = has_ffn ? d->ffn : 0;
  s->nh = has_attn ? d->heads : 0;
  s->d = has_attn ? d->hidden / d->heads : 0;
  s->w = d->w;
  s->nsb = d->sub_batches;
  s->pre_ln = d->pre_ln != 0;
  s->residual = d->residual != 0;
  s->causal = d->causal != 0;
  s->mode = d->recompute;
  s->reduce = d->reduce;
  s->t = d->dtype == OASES_F32 ? DType::F32 : DType::BF16;
  s->mx = d->dtype == OASES_MXFP8;
  s->eps = d->ln_eps;
  s->M = M;
  s->Ms = M / d->sub_batches;
  s->esz = dtype_size(s->t);
  s->segs_per_layer = d->kind == OASES_BLOCK_LAYER ? 2 : 1;
  s->nseg = s->segs_per_layer * n_layers;
  return OASES_OK;
}

// ---------------------------------------------------------------------------
// Workspace layout.  Every region spans all M rows; sub-batch b uses rows
// [b*Ms, (b+1)*Ms) (per-head statistics: block b of [nsb][heads][Ms]).
// ---------------------------------------------------------------------------
constexpr size_t ALIGN = 256;
inline size_t up(size_t v) { return (v + ALIGN - 1) / ALIGN * ALIGN; }

struct ActSet {  // offsets relative to the workspace base
  size_t u = 0, mu = 0, rstd = 0, a = 0, h = 0, qkv = 0, o = 0, lse = 0, delta = 0, d_o = 0,
         dqkv = 0, du = 0, cpart = 0, lpart_g = 0, lpart_b = 0, lstat = 0,
         red = 0;  // separate-reduction partials, fp32 [w][M][H]
};

struct MxScratch {  // one sub-batch stream's quantised GEMM operands
  size_t qa = 0, sfa = 0, qb = 0, sfb = 0;
};

struct Layout {
  size_t stage[4] = {0, 0, 0, 0};  // x, g, y, dx staging for host buffers
  MxScratch mx[2];                 // MX-FP8 blocks: per stream
  std::vector<size_t> ckpt;        // input of segment s (s >= 1)
  size_t grad[2] = {0, 0};
  size_t yr = 0;
  std::vector<ActSet> act;  // per segment
  size_t cpart_n = 0;       // floats per sub-batch in a colsum partial buffer
  size_t lpart_n = 0;       // floats per sub-batch in an LN partial buffer
  size_t total = 0;
};

Layout make_layout(const Shape& s) {
  Layout L;
  size_t off = ALIGN;  // first 256 bytes reserved
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += up(bytes);
    return o;
  };
  const size_t MH = (size_t)s.M * s.H * s.esz;
  for (int i = 0; i < 4; ++i) L.stage[i] = take(MH);
  L.ckpt.assign(s.nseg, 0);
  for (int i = 1; i < s.nseg; ++i) L.ckpt[i] = take(MH);
  L.grad[0] = take(MH);
  L.grad[1] = take(MH);
  L.yr = take(MH);
  const size_t maxN = (size_t)std::max<int64_t>(std::max(s.H, s.F), 3 * (int64_t)s.H);
  L.cpart_n = (size_t)colsum_blocks((int)s.Ms) * maxN;
  L.lpart_n = (size_t)ln_bwd_blocks((int)s.Ms) * s.H;
  // A segment's buffers.  `share` (the first set of the same kind, or null)
  // supplies the backward scratch, which sub-batch streams use one segment
  // at a time, and, in SELECTIVE mode, the attention output O and its LSE,
  // which that mode recomputes before each attention segment's backward.
  auto make_set = [&](int kind, const ActSet* share) {
    ActSet a;
    const size_t M = (size_t)s.M;
    if (s.pre_ln) a.u = take(M * s.H * s.esz);
    a.mu = take(M * 4);
    a.rstd = take(M * 4);
    if (kind == SEG_FFN) {
      a.a = take(M * s.F * s.esz);
      a.h = take(M * s.F * s.esz);
    } else {
      a.qkv = take(M * 3 * s.H * s.esz);
      if (share && s.mode == OASES_RECOMPUTE_SELECTIVE) {
        a.o = share->o;
        a.lse = share->lse;
      } else {
        a.o = take(M * s.H * s.esz);
        a.lse = take(M * s.nh * 4);
      }
    }
    if (share) {
      a.delta = share->delta;
      a.d_o = share->d_o;
      a.dqkv = share->dqkv;
      a.du = share->du;
      a.cpart = share->cpart;
      a.lpart_g = share->lpart_g;
      a.lpart_b = share->lpart_b;
      a.lstat = share->lstat;
      a.red = share->red;
      return a;
    }
    if (kind == SEG_ATTN) {
      a.delta = take(M * s.nh * 4);
      a.d_o = take(M * s.H * s.esz);
      a.dqkv = take(M * 3 * s.H * s.esz);
    }
    a.du = take(M * s.H * 4);
    a.cpart = take(s.nsb * L.cpart_n * 4);
    a.lpart_g = take(s.nsb * L.lpart_n * 4);
    a.lpart_b = take(s.nsb * L.lpart_n * 4);
    a.lstat = take(M * 8);
    if (s.reduce == OASES_REDUCE_SEPARATE) a.red = take((size_t)s.w * M * s.H * 4);
    return a;
  };
  L.act.resize(s.nseg);
  if (s.mode == OASES_RECOMPUTE_NONE || s.mode == OASES_RECOMPUTE_SELECTIVE) {
    // activations kept per segment, scratch per kind
    int first[2] = {-1, -1};
    for (int i = 0; i < s.nseg; ++i) {
      const int k = s.seg_kind(i);
      L.act[i] = make_set(k, first[k] >= 0 ? &L.act[first[k]] : nullptr);
      if (first[k] < 0) first[k] = i;
    }
  } else {
    ActSet per_kind[2];
    bool made[2] = {false, false};
    for (int i = 0; i < s.nseg; ++i) {
      const int k = s.seg_kind(i);
      if (!made[k]) {
        per_kind[k] = make_set(k, nullptr);
        made[k] = true;
      }
      L.act[i] = per_kind[k];
    }
  }
  if (s.mx) {
    // the largest A and B operands (rows x contraction) of any GEMM of the
    // block, as MX codes (rows padded to 16 bytes) and scale tiles
    const int64_t Ms = s.Ms, H = s.H, W = std::max<int64_t>(std::max<int64_t>(s.F, 3 * (int64_t)s.H), s.H);
    auto rup = [](int64_t v) { return (v + 15) / 16 * 16; };
    const std::pair<int64_t, int64_t> As[] = {{Ms, W}, {W, Ms}, {Ms, H}, {H, Ms}};
    const std::pair<int64_t, int64_t> Bs[] = {{W, H}, {H, W}, {W, Ms}, {H, Ms}};
    size_t qa = 0, sfa = 0, qb = 0, sfb = 0;
    for (auto p : As) {
      qa = std::max(qa, (size_t)(p.first * rup(p.second)));
      sfa = std::max(sfa, (size_t)mx_sf_bytes((int)p.first, (int)p.second));
    }
    for (auto p : Bs) {
      qb = std::max(qb, (size_t)(p.first * rup(p.second)));
      sfb = std::max(sfb, (size_t)mx_sf_bytes((int)p.first, (int)p.second));
    }
    for (int k = 0; k < 2; ++k) {
      L.mx[k].qa = take(qa);
      L.mx[k].sfa = take(sfa);
      L.mx[k].qb = take(qb);
      L.mx[k].sfb = take(sfb);
    }
  }
  L.total = off;
  return L;
}

// ---------------------------------------------------------------------------
// Schedule (Algorithm 1).
// ---------------------------------------------------------------------------
std::vector<Step> schedule(const Shape& s, int phase) {
  std::vector<Step> out;
  if (phase == 0) {
    for (int seg = 0; seg < s.nseg; ++seg)
      for (int b = 0; b < s.nsb; ++b) {
        if (seg > 0) out.push_back({EV_SYNC, OP_G, seg - 1, b});
        out.push_back({EV_F, OP_LN, seg, b});
        out.push_back({EV_F, OP_COL, seg, b});
        out.push_back({EV_F, OP_ROW, seg, b});
        out.push_back({EV_CF, OP_G, seg, b});
      }
    for (int b = 0; b < s.nsb; ++b) out.push_back({EV_SYNC, OP_G, s.nseg - 1, b});
    return out;
  }
  for (int seg = s.nseg - 1; seg >= 0; --seg)
    for (int b = 0; b < s.nsb; ++b) {
      if (seg < s.nseg - 1) {
        out.push_back({EV_SYNC, OP_F, seg + 1, b});
        out.push_back({EV_B, OP_LN, seg + 1, b});
      }
      if (s.mode == OASES_RECOMPUTE_SELECTIVE) {
        if (s.seg_kind(seg) == SEG_ATTN) out.push_back({EV_R, OP_ATTN, seg, b});
      } else if (s.mode != OASES_RECOMPUTE_NONE) {
        out.push_back({EV_R, OP_LN, seg, b});
        out.push_back({EV_R, OP_COL, seg, b});
        if (s.mode == OASES_RECOMPUTE_FULL) {
          out.push_back({EV_R, OP_ROW, seg, b});
          out.push_back({EV_CR, OP_G, seg, b});
        }
      }
      out.push_back({EV_B, OP_G, seg, b});
      out.push_back({EV_B, OP_ROW, seg, b});
      out.push_back({EV_B, OP_COL, seg, b});
      out.push_back({EV_CB, OP_F, seg, b});
    }
  for (int b = 0; b < s.nsb; ++b) {
    out.push_back({EV_SYNC, OP_F, 0, b});
    out.push_back({EV_B, OP_LN, 0, b});
  }
  return out;
}

bool injected(const std::vector<Step>& steps) {
  const char* v = std::getenv("OASES_TEST_FAIL_AT");
  if (!v || !*v) return false;
  int e, o, sg, b;
  if (std::sscanf(v, "%d:%d:%d:%d", &e, &o, &sg, &b) != 4) return false;
  for (const Step& st : steps)
    if (st.ev == e && st.op == o && st.seg == sg && st.sb == b) return true;
  return false;
}

// ---------------------------------------------------------------------------
// Execution.
// ---------------------------------------------------------------------------
struct EventPool {
  uint64_t ctx = 0;  // context the events belong to
  std::vector<cudaEvent_t> ev;
  // an event with pending work is released when that work completes
  void release() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
    ev.clear();
  }
  ~EventPool() { release(); }  // at thread exit
  cudaError_t ensure(size_t n) {
    while (ev.size() < n) {
      cudaEvent_t e;
      cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
      if (r != cudaSuccess) return r;
      ev.push_back(e);
    }
    return cudaSuccess;
  }
};
// The events of this host thread's calls on the current device.  Per thread,
// so concurrent calls from several threads never share an event (calls from
// one thread are enqueued in order, and a wait captures an event's state when
// it is enqueued, so reuse across that thread's calls is safe); per device,
// because an event can be recorded only on streams of its own device.  Events
// made under a context that has since been destroyed are dropped, not used.
thread_local std::unordered_map<int, EventPool> t_pools;
EventPool& pool() {
  EventPool& p = t_pools[current_device()];
  const uint64_t id = current_ctx_id();
  if (p.ctx != id) {
    p.ev.clear();  // the old context took its events with it
    p.ctx = id;
  }
  return p;
}

// A non-blocking stream per device for host<->device staging copies, so they
// overlap the compute streams (created on first use, kept until
// oases_shutdown() or until the device's context is destroyed).
struct CopyStream {
  uint64_t ctx = 0;
  cudaStream_t st = nullptr;
};
std::mutex g_copy_mu;
std::unordered_map<int, CopyStream> g_copy;

cudaStream_t copy_stream() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  const uint64_t id = current_ctx_id();
  std::lock_guard<std::mutex> lock(g_copy_mu);
  auto it = g_copy.find(dev);
  if (it != g_copy.end() && it->second.ctx == id && id != 0) return it->second.st;
  cudaStream_t st = nullptr;
  if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  g_copy[dev] = CopyStream{id, st};
  return st;
}

struct SegParams {  // one segment's weights / grads, typed by role
  const void *g, *b, *wc, *bc, *wr, *br;
  float *dg, *db, *dwc, *dbc, *dwr, *dbr;
};

struct Exec {
  Shape s;
  Layout L;
  uint8_t* ws;
  cudaStream_t st[2];
  std::vector<SegParams> sp;  // per segment
  const void* x;              // input of segment 0
  void* y;                    // output of the last segment
  const void* dy;             // gradient w.r.t. y
  void* dx;                   // gradient w.r.t. x
  cudaError_t err = cudaSuccess;
  // partial rows of colsum(grad_out(seg)) for sub-batch b that the LayerNorm
  // backward of segment seg + 1 left in cpart(seg, b) (0: none; -1: that
  // backward already added them into db_row; [seg * nsb + b])
  std::vector<int> xparts;
  // partial rows of colsum(dA) that the dA GEMM's epilogue left in
  // cpart(seg, b) for db1 (0: none; [seg * nsb + b])
  std::vector<int> aparts;
  // 1: the dO GEMM's epilogue wrote delta = rowsum(dO * O) for (seg, b)
  std::vector<int> dready;
  EventPool* P = nullptr;  // this thread's events on the call's device
  size_t ev_base = 2;      // P->ev[0], [1]: call entry / exit joins

  template <typename T = void>
  T* at(size_t off) const { return reinterpret_cast<T*>(ws + off); }
  size_t rows_off(int b, int64_t width, size_t esz) const {
    return (size_t)b * s.Ms * width * esz;
  }
  const void* seg_in(int seg) const { return seg == 0 ? x : at(L.ckpt[seg]); }
  void* seg_out(int seg) const { return seg == s.nseg - 1 ? y : at(L.ckpt[seg + 1]); }
  const void* grad_out(int seg) const {  // dL/d(output of seg)
    return seg == s.nseg - 1 ? dy : at(L.grad[seg & 1]);
  }
  void* grad_in(int seg) const {  // dL/d(input of seg)
    return seg == 0 ? dx : at(L.grad[(seg - 1) & 1]);
  }
  template <typename P>
  P rowp(P base, int b, int64_t width, size_t esz) const {
    return reinterpret_cast<P>(reinterpret_cast<uintptr_t>(base) + rows_off(b, width, esz));
  }
  cudaStream_t stream(int b) const { return st[b & 1]; }

  void ok(cudaError_t e) {
    if (err == cudaSuccess && e != cudaSuccess) err = e;
  }

  // Weight-gradient ordering across sub-batches on different streams.
  cudaEvent_t gev(int seg, int grp) const { return P->ev[ev_base + seg * GRP_N + grp]; }
  void grad_wait(int seg, int grp, int b) {
    if (b > 0 && st[0] != st[1]) ok(cudaStreamWaitEvent(stream(b), gev(seg, grp), 0));
  }
  void grad_done(int seg, int grp, int b) {
    if (b + 1 < s.nsb && st[0] != st[1]) ok(cudaEventRecord(gev(seg, grp), stream(b)));
  }

  // One of the block's GEMMs: bf16 (or fp32) as described, or, for an MX-FP8
  // block, both operands quantised along the contraction into this stream's
  // scratch (row-wise for a K-major operand, transposed for an MN-major one)
  // and multiplied by the block-scaled MMA with the same epilogue.
  cudaError_t run_gemm(const GemmArgs& g, int b) {
    if (!s.mx) return gemm(g, stream(b));
    if (g.M == 0 || g.N == 0) return cudaSuccess;
    const MxScratch& sc = L.mx[b & 1];
    const int64_t lqa = (g.K + 15) / 16 * 16, lqb = lqa;
    uint8_t* qa = at<uint8_t>(sc.qa);
    uint8_t* qb = at<uint8_t>(sc.qb);
    uint8_t* sfa = at<uint8_t>(sc.sfa);
    uint8_t* sfb = at<uint8_t>(sc.sfb);
    cudaError_t e = g.a_kmajor ? mx_quantize_rows(g.A, g.lda, g.M, g.K, g.in_t, qa, lqa, sfa, stream(b))
                               : mx_quantize_cols(g.A, g.lda, g.K, g.M, g.in_t, qa, lqa, sfa, stream(b));
    if (e != cudaSuccess) return e;
    e = g.b_kmajor ? mx_quantize_rows(g.B, g.ldb, g.N, g.K, g.in_t, qb, lqb, sfb, stream(b))
                   : mx_quantize_cols(g.B, g.ldb, g.K, g.N, g.in_t, qb, lqb, sfb, stream(b));
    if (e != cudaSuccess) return e;
    GemmArgs m = g;
    m.in_t = DType::E4M3;
    m.A = qa;
    m.lda = lqa;
    m.a_kmajor = true;
    m.a_sf = sfa;
    m.B = qb;
    m.ldb = lqb;
    m.b_kmajor = true;
    m.b_sf = sfb;
    m.aux_t = DType::BF16;
    return gemm_mx(m, stream(b));
  }

  GemmArgs base_gemm() const {
    GemmArgs g;
    g.in_t = s.t;
    g.c_t = s.t;
    g.aux_t = s.t;
    g.concurrent = st[0] != st[1] && s.nsb > 1;  // the other sub-batch stream runs beside it
    return g;
  }

  // u = LN(x_seg) (or u = x_seg without LayerNorm).
  const void* ln_fwd(int seg, int b) {
    const ActSet& a = L.act[seg];
    const void* xin = rowp(seg_in(seg), b, s.H, s.esz);
    if (!s.pre_ln) return xin;
    void* u = rowp(at(a.u), b, s.H, s.esz);
    ok(layer_norm_fwd(xin, sp[seg].g, sp[seg].b, u, rowp(at<float>(a.mu), b, 1, 4),
                      rowp(at<float>(a.rstd), b, 1, 4), (int)s.Ms, s.H, s.eps, s.t, stream(b)));
    return u;
  }
  const void* u_of(int seg, int b) const {
    return s.pre_ln ? rowp(at(L.act[seg].u), b, s.H, s.esz) : rowp(seg_in(seg), b, s.H, s.esz);
  }

  // Column GEMM F_i.  FFN: H = GeLU(u W1^T + b1), and with keep_grad also
  // G = GeLU'(u W1^T + b1) (into the A buffer), all the GeLU backward needs.
  void col_fwd(int seg, int b, bool keep_grad) {
    const ActSet& a = L.act[seg];
    const SegParams& p = sp[seg];
    const void* u = u_of(seg, b);
    GemmArgs g = base_gemm();
    g.M = (int)s.Ms;
    g.K = s.H;
    g.A = u;
    g.lda = s.H;
    if (s.seg_kind(seg) == SEG_FFN) {
      g.N = s.F;
      g.B = p.wc;
      g.ldb = s.H;
      g.epi = Epi::BiasGelu;
      g.bias = p.bc;
      g.C = rowp(at(a.h), b, s.F, s.esz);
      g.ldc = s.F;
      g.C2 = keep_grad ? rowp(at(a.a), b, s.F, s.esz) : nullptr;
      ok(run_gemm(g, b));
    } else {
      g.N = 3 * s.H;
      g.B = p.wc;
      g.ldb = s.H;
      g.epi = Epi::Bias;
      g.bias = p.bc;
      g.C = rowp(at(a.qkv), b, 3 * s.H, s.esz);
      g.ldc = 3 * s.H;
      ok(run_gemm(g, b));
      ok(attention_fwd(attn_args(seg, b), stream(b)));
    }
  }

  // Causal attention of sub-batch b over the segment's kept Q, K, V.
  AttnArgs attn_args(int seg, int b) const {
    const ActSet& a = L.act[seg];
    AttnArgs at_;
    at_.batch = s.B / s.nsb;
    at_.seq = s.S;
    at_.heads = s.nh;
    at_.head_dim = s.d;
    at_.hidden = s.H;
    at_.causal = s.causal;
    at_.t = s.t;
    at_.qkv = rowp(at(a.qkv), b, 3 * s.H, s.esz);
    at_.o = rowp(at(a.o), b, s.H, s.esz);
    at_.lse = at<float>(a.lse) + (size_t)b * s.nh * s.Ms;
    at_.d_o = rowp(at(a.d_o), b, s.H, s.esz);
    at_.delta = at<float>(a.delta) + (size_t)b * s.nh * s.Ms;
    at_.dqkv = rowp(at(a.dqkv), b, 3 * s.H, s.esz);
    return at_;
  }

  // Row GEMM with the shard sum fused (C_i(F)); out = seg output or recompute scratch.
  void row_fwd(int seg, int b, void* out) {
    const ActSet& a = L.act[seg];
    const SegParams& p = sp[seg];
    const bool ffn = s.seg_kind(seg) == SEG_FFN;
    GemmArgs g = base_gemm();
    g.M = (int)s.Ms;
    g.N = s.H;
    g.K = ffn ? s.F : s.H;
    g.A = ffn ? rowp(at(a.h), b, s.F, s.esz) : rowp(at(a.o), b, s.H, s.esz);
    g.lda = g.K;
    g.B = p.wr;
    g.ldb = g.K;
    g.bias = p.br;
    g.C = rowp(out, b, s.H, s.esz);
    g.ldc = s.H;
    if (s.residual) {
      g.epi = Epi::BiasResid;
      g.aux = rowp(seg_in(seg), b, s.H, s.esz);
      g.ld_aux = s.H;
    } else {
      g.epi = Epi::Bias;
    }
    ok(run_gemm(g, b));
  }

  // SEPARATE mode: shard k's partial of sub-batch b, fp32 [Ms, H] rows of [w][M][H].
  float* red_part(int seg, int k, int b) const {
    return at<float>(L.act[seg].red) + ((size_t)k * s.M + (size_t)b * s.Ms) * s.H;
  }
  // P_k = hin[:, slice k] W_row[:, slice k]^T for every shard k (its K-slice
  // only): one split-contraction launch over all shards where the tensor-core
  // path takes it, else one GEMM per shard.
  void row_partials(int seg, int b) {
    const ActSet& a = L.act[seg];
    const bool ffn = s.seg_kind(seg) == SEG_FFN;
    const int Kin = ffn ? s.F : s.H, Kw = Kin / s.w;
    const uint8_t* hin = reinterpret_cast<const uint8_t*>(
        ffn ? rowp(at(a.h), b, s.F, s.esz) : rowp(at(a.o), b, s.H, s.esz));
    const uint8_t* wr = reinterpret_cast<const uint8_t*>(sp[seg].wr);
    GemmArgs all = base_gemm();
    all.M = (int)s.Ms;
    all.N = s.H;
    all.K = Kw;
    all.A = hin;
    all.lda = Kin;
    all.B = wr;
    all.ldb = Kin;
    all.epi = Epi::Store;
    all.C = red_part(seg, 0, b);
    all.c_t = DType::F32;
    all.ldc = s.H;
    all.splits = s.w;
    all.k_extent = Kin;
    all.c_split_rows = s.M;
    if (gemm_tc_supported(all)) {
      ok(gemm(all, stream(b)));
      return;
    }
    for (int k = 0; k < s.w; ++k) {
      GemmArgs g = base_gemm();
      g.M = (int)s.Ms;
      g.N = s.H;
      g.K = Kw;
      g.A = hin + (size_t)k * Kw * s.esz;
      g.lda = Kin;
      g.B = wr + (size_t)k * Kw * s.esz;
      g.ldb = Kin;
      g.epi = Epi::Store;
      g.C = red_part(seg, k, b);
      g.c_t = DType::F32;
      g.ldc = s.H;
      ok(gemm(g, stream(b)));
    }
  }
  // y = sum_k P_k + bias (+ x): the C(F) / C(R) step in SEPARATE mode.
  void reduce_rows(int seg, int b, void* out) {
    ok(shard_sum(red_part(seg, 0, b), (int64_t)s.M * s.H, s.w, sp[seg].br,
                 s.residual ? rowp(seg_in(seg), b, s.H, s.esz) : nullptr,
                 rowp(out, b, s.H, s.esz), s.t, s.t, (int)s.Ms, s.H, stream(b)));
  }

  float* cpart(int seg, int b) const {
    return at<float>(L.act[seg].cpart) + (size_t)b * L.cpart_n;
  }

  void bwd_g(int seg, int b) {  // db_row += colsum(dy); Eq. (1): dP_k = dy, nothing else to do
    int& xp = xparts[(size_t)seg * s.nsb + b];
    if (xp < 0) {  // summed and accumulated by the next segment's LayerNorm backward
      xp = 0;
      return;
    }
    grad_wait(seg, GRP_BR, b);
    if (xp > 0)  // the column sums of dy were taken as it was written (LayerNorm backward)
      ok(reduce_partial_rows(cpart(seg, b), sp[seg].dbr, xp, s.H, stream(b)));
    else
      ok(colsum_accum(rowp(grad_out(seg), b, s.H, s.esz), s.H, (int)s.Ms, s.H, s.t, cpart(seg, b),
                      sp[seg].dbr, stream(b)));
    xp = 0;
    grad_done(seg, GRP_BR, b);
  }

  void bwd_row(int seg, int b) {
    const ActSet& a = L.act[seg];
    const SegParams& p = sp[seg];
    const bool ffn = s.seg_kind(seg) == SEG_FFN;
    const int Kin = ffn ? s.F : s.H;  // width of the row GEMM's input
    const void* dyb = rowp(grad_out(seg), b, s.H, s.esz);
    const void* hin = ffn ? rowp(at(a.h), b, s.F, s.esz) : rowp(at(a.o), b, s.H, s.esz);
    // dW_row[H, Kin] += dy^T hin   (contraction over the sub-batch rows)
    GemmArgs w = base_gemm();
    w.M = s.H;
    w.N = Kin;
    w.K = (int)s.Ms;
    w.A = dyb;
    w.lda = s.H;
    w.a_kmajor = false;
    w.B = hin;
    w.ldb = Kin;
    w.b_kmajor = false;
    w.epi = Epi::Accum;
    w.C = p.dwr;
    w.c_t = DType::F32;
    w.ldc = Kin;
    grad_wait(seg, GRP_WR, b);
    ok(run_gemm(w, b));
    grad_done(seg, GRP_WR, b);
    // d(hin) = dy W_row; FFN: dA = dH * G with G = gelu'(A) kept by the forward or the
    // recompute, written over G.
    GemmArgs d = base_gemm();
    d.M = (int)s.Ms;
    d.N = Kin;
    d.K = s.H;
    d.A = dyb;
    d.lda = s.H;
    d.B = p.wr;
    d.ldb = Kin;
    d.b_kmajor = false;
    d.ldc = Kin;
    if (ffn) {
      void* G = rowp(at(a.a), b, s.F, s.esz);  // GeLU'(A), overwritten by dA
      d.epi = Epi::Mul;
      d.aux = G;
      d.ld_aux = s.F;
      d.C = G;
      // db1 = colsum(dA): the epilogue sums dA's columns as it stores them,
      // into this segment's colsum scratch (nothing else of this sub-batch
      // uses it before bwd_col reduces it)
      int& ap = aparts[(size_t)seg * s.nsb + b];
      ap = 0;
      if ((size_t)((s.Ms + 31) / 32) * (size_t)s.F <= L.cpart_n) {
        d.colsum_part = cpart(seg, b);
        d.colsum_rows = &ap;
      }
    } else {
      d.epi = Epi::Store;
      d.C = rowp(at(a.d_o), b, s.H, s.esz);
      // the attention backward's delta = rowsum(dO * O) per head, summed by
      // the epilogue as it stores dO (one head is 128 columns)
      int& dr = dready[(size_t)seg * s.nsb + b];
      dr = 0;
      if (s.d == 128) {
        d.rowdot_aux = rowp(at(a.o), b, s.H, s.esz);
        d.rowdot_lda = s.H;
        d.rowdot_out = at<float>(a.delta) + (size_t)b * s.nh * s.Ms;
        d.rowdot_ld = (int64_t)s.Ms;
        d.rowdot_done = &dr;
      }
    }
    ok(run_gemm(d, b));
  }

  void bwd_col(int seg, int b) {
    const ActSet& a = L.act[seg];
    const SegParams& p = sp[seg];
    const bool ffn = s.seg_kind(seg) == SEG_FFN;
    const int Nc = ffn ? s.F : 3 * s.H;  // column GEMM output width
    const void* dcol;
    int bias_rows = 0;  // > 0: the bias gradient's partial rows are in cpart(seg, b)
    if (ffn) {
      dcol = rowp(at(a.a), b, s.F, s.esz);  // dA
    } else {
      AttnArgs at_ = attn_args(seg, b);
      at_.delta_ready = dready[(size_t)seg * s.nsb + b] != 0;
      dready[(size_t)seg * s.nsb + b] = 0;
      // the tensor-core backward sums dqkv's columns as it stores them
      const int rows = at_.batch * ((at_.seq + 127) / 128) * 4;
      if (attention_tc_supported(at_) && !(((uintptr_t)at_.d_o | (uintptr_t)at_.dqkv) & 15) &&
          (size_t)rows * (size_t)Nc <= L.cpart_n && rows <= 512) {
        ok(attention_bwd_tc_bias(at_, cpart(seg, b), stream(b)));
        bias_rows = rows;
      } else {
        ok(attention_bwd(at_, stream(b)));
      }
      dcol = at_.dqkv;
    }
    if (ffn) {
      bias_rows = aparts[(size_t)seg * s.nsb + b];
      aparts[(size_t)seg * s.nsb + b] = 0;
    }
    grad_wait(seg, GRP_BC, b);
    if (bias_rows > 0)
      ok(reduce_partial_rows(cpart(seg, b), p.dbc, bias_rows, Nc, stream(b)));
    else
      ok(colsum_accum(dcol, Nc, (int)s.Ms, Nc, s.t, cpart(seg, b), p.dbc, stream(b)));
    grad_done(seg, GRP_BC, b);
    // dW_col[Nc, H] += dcol^T u
    GemmArgs w = base_gemm();
    w.M = Nc;
    w.N = s.H;
    w.K = (int)s.Ms;
    w.A = dcol;
    w.lda = Nc;
    w.a_kmajor = false;
    w.B = u_of(seg, b);
    w.ldb = s.H;
    w.b_kmajor = false;
    w.epi = Epi::Accum;
    w.C = p.dwc;
    w.c_t = DType::F32;
    w.ldc = s.H;
    grad_wait(seg, GRP_WC, b);
    ok(run_gemm(w, b));
    grad_done(seg, GRP_WC, b);
  }

  // C_i(B): du = sum over shards of dcol_k W_col_k = dcol W_col (full-K contraction), fp32.
  void comm_bwd(int seg, int b) {
    if (s.reduce == OASES_REDUCE_SEPARATE) {
      comm_bwd_separate(seg, b);
      return;
    }
    const ActSet& a = L.act[seg];
    const bool ffn = s.seg_kind(seg) == SEG_FFN;
    const int Nc = ffn ? s.F : 3 * s.H;
    GemmArgs g = base_gemm();
    g.M = (int)s.Ms;
    g.N = s.H;
    g.K = Nc;
    g.A = ffn ? rowp(at(a.a), b, s.F, s.esz) : rowp(at(a.dqkv), b, 3 * s.H, s.esz);
    g.lda = Nc;
    g.B = sp[seg].wc;
    g.ldb = s.H;
    g.b_kmajor = false;
    g.epi = Epi::Store;
    g.C = rowp(at<float>(a.du), b, s.H, 4);
    g.c_t = DType::F32;
    g.ldc = s.H;
    ok(run_gemm(g, b));
  }

  // SEPARATE mode: du_k = dcol[:, cols of shard k] W_col[rows of shard k, :] in
  // fp32 partials, then du = sum_k du_k.  An attention shard's columns are three
  // ranges (its Q, K and V heads), accumulated into the same partial.
  void comm_bwd_separate(int seg, int b) {
    const ActSet& a = L.act[seg];
    const bool ffn = s.seg_kind(seg) == SEG_FFN;
    const int Nc = ffn ? s.F : 3 * s.H;
    const uint8_t* dcol = reinterpret_cast<const uint8_t*>(
        ffn ? rowp(at(a.a), b, s.F, s.esz) : rowp(at(a.dqkv), b, 3 * s.H, s.esz));
    const uint8_t* wc = reinterpret_cast<const uint8_t*>(sp[seg].wc);
    const int parts = ffn ? 1 : 3, Kw = ffn ? s.F / s.w : s.H / s.w;
    GemmArgs all = base_gemm();
    all.M = (int)s.Ms;
    all.N = s.H;
    all.K = parts * Kw;
    all.kpieces = parts;
    all.kpiece_stride = s.H;  // attention: the Q, K and V column blocks
    all.k_extent = Nc;
    all.A = dcol;
    all.lda = Nc;
    all.B = wc;
    all.ldb = s.H;
    all.b_kmajor = false;
    all.epi = Epi::Store;
    all.C = red_part(seg, 0, b);
    all.c_t = DType::F32;
    all.ldc = s.H;
    all.splits = s.w;
    all.c_split_rows = s.M;
    const bool one_launch = gemm_tc_supported(all);
    if (one_launch) ok(gemm(all, stream(b)));
    for (int k = 0; k < s.w && !one_launch; ++k)
      for (int p = 0; p < parts; ++p) {
        const size_t c0 = (ffn ? 0 : (size_t)p * s.H) + (size_t)k * Kw;  // first column / W row
        GemmArgs g = base_gemm();
        g.M = (int)s.Ms;
        g.N = s.H;
        g.K = Kw;
        g.A = dcol + c0 * s.esz;
        g.lda = Nc;
        g.B = wc + c0 * s.H * s.esz;
        g.ldb = s.H;
        g.b_kmajor = false;
        g.epi = p == 0 ? Epi::Store : Epi::Accum;
        g.C = red_part(seg, k, b);
        g.c_t = DType::F32;
        g.ldc = s.H;
        ok(gemm(g, stream(b)));
      }
    ok(shard_sum(red_part(seg, 0, b), (int64_t)s.M * s.H, s.w, nullptr, nullptr,
                 rowp(at<float>(a.du), b, s.H, 4), DType::F32, s.t, (int)s.Ms, s.H, stream(b)));
  }

  void bwd_ln(int seg, int b) {
    const ActSet& a = L.act[seg];
    const float* du = rowp(at<float>(a.du), b, s.H, 4);
    const void* dres = s.residual ? rowp(grad_out(seg), b, s.H, s.esz) : nullptr;
    void* dxo = rowp(grad_in(seg), b, s.H, s.esz);
    if (s.pre_ln) {
      // dx is the previous segment's output gradient: its column sums (that
      // segment's row-bias gradient) are taken here, as dx is written, into
      // the previous segment's colsum scratch, and added into db_row by the
      // same reduction launch as dgamma and dbeta (else by that segment's
      // bwd_g).  The sub-batch order of both accumulations is kept by waits
      // placed right before that launch: this sub-batch's LayerNorm kernel
      // itself waits for nothing of the other's.
      float* px = seg >= 1 ? cpart(seg - 1, b) : nullptr;
      const int cap = (int)std::min<size_t>(L.cpart_n / (size_t)s.H, 1u << 20);
      int np = 0;
      const std::function<void(bool)> before_reduce = [&](bool with_x) {
        grad_wait(seg, GRP_LN, b);
        if (with_x) grad_wait(seg - 1, GRP_BR, b);
      };
      ok(layer_norm_bwd_dx_colsum(du, rowp(seg_in(seg), b, s.H, s.esz), rowp(at<float>(a.mu), b, 1, 4),
                                  rowp(at<float>(a.rstd), b, 1, 4), sp[seg].g, dres, dxo,
                                  at<float>(a.lpart_g) + (size_t)b * L.lpart_n,
                                  at<float>(a.lpart_b) + (size_t)b * L.lpart_n,
                                  rowp(at<float2>(a.lstat), b, 1, 8), sp[seg].dg, sp[seg].db,
                                  (int)s.Ms, s.H, s.t, stream(b), px, cap, &np,
                                  seg >= 1 ? sp[seg - 1].dbr : nullptr, &before_reduce));
      if (seg >= 1) {
        xparts[(size_t)(seg - 1) * s.nsb + b] = np;
        if (np < 0) grad_done(seg - 1, GRP_BR, b);
      }
      grad_done(seg, GRP_LN, b);
    } else {
      ok(add_into(dres, du, dxo, (int64_t)s.Ms * s.H, s.t, stream(b)));
    }
  }

  void run(const Step& st_) {
    const int seg = st_.seg, b = st_.sb;
    switch (st_.ev) {
      case EV_F:
        if (st_.op == OP_LN) ln_fwd(seg, b);
        else if (st_.op == OP_COL)
          col_fwd(seg, b, s.mode == OASES_RECOMPUTE_NONE || s.mode == OASES_RECOMPUTE_SELECTIVE);
        else if (st_.op == OP_ROW) {
          if (s.reduce == OASES_REDUCE_SEPARATE) row_partials(seg, b);
          else row_fwd(seg, b, seg_out(seg));
        }
        break;
      case EV_CF:
        if (s.reduce == OASES_REDUCE_SEPARATE) reduce_rows(seg, b, seg_out(seg));
        break;
      case EV_R:
        if (st_.op == OP_LN) ln_fwd(seg, b);
        else if (st_.op == OP_ATTN) ok(attention_fwd(attn_args(seg, b), stream(b)));
        else if (st_.op == OP_COL) col_fwd(seg, b, true);
        else if (st_.op == OP_ROW) {
          if (s.reduce == OASES_REDUCE_SEPARATE) row_partials(seg, b);
          else row_fwd(seg, b, at(L.yr));
        }
        break;
      case EV_CR:
        if (s.reduce == OASES_REDUCE_SEPARATE) reduce_rows(seg, b, at(L.yr));
        break;
      case EV_B:
        if (st_.op == OP_G) bwd_g(seg, b);
        else if (st_.op == OP_ROW) bwd_row(seg, b);
        else if (st_.op == OP_COL) bwd_col(seg, b);
        else if (st_.op == OP_LN) bwd_ln(seg, b);
        break;
      case EV_CB:
        comm_bwd(seg, b);
        break;
      default:  // Sync: stream order
        break;
    }
  }
};

SegParams seg_params(const Shape& s, int seg, const oases_weights* w, const oases_grads* gr) {
  const int layer = seg / s.segs_per_layer;
  const oases_weights& W = w[layer];
  SegParams p{};
  const oases_grads* G = gr ? &gr[layer] : nullptr;
  if (s.seg_kind(seg) == SEG_FFN) {
    p = {W.ln2_g, W.ln2_b, W.w1, W.b1, W.w2, W.b2,
         G ? G->ln2_g : nullptr, G ? G->ln2_b : nullptr, G ? G->w1 : nullptr,
         G ? G->b1 : nullptr, G ? G->w2 : nullptr, G ? G->b2 : nullptr};
  } else {
    p = {W.ln1_g, W.ln1_b, W.wqkv, W.bqkv, W.wo, W.bo,
         G ? G->ln1_g : nullptr, G ? G->ln1_b : nullptr, G ? G->wqkv : nullptr,
         G ? G->bqkv : nullptr, G ? G->wo : nullptr, G ? G->bo : nullptr};
  }
  return p;
}

// Device pointers must be 16-byte aligned (TMA operands, 16-byte vector loads
// and stores); NULL passes.
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

bool params_ok(const Shape& s, const std::vector<SegParams>& sp, bool need_grads) {
  for (const SegParams& p : sp) {
    if (!p.wc || !p.bc || !p.wr || !p.br) return false;
    for (const void* q : {(const void*)p.g, (const void*)p.b, (const void*)p.wc,
                          (const void*)p.bc, (const void*)p.wr, (const void*)p.br,
                          (const void*)p.dg, (const void*)p.db, (const void*)p.dwc,
                          (const void*)p.dbc, (const void*)p.dwr, (const void*)p.dbr})
      if (!aligned16(q)) return false;
    if (s.pre_ln && (!p.g || !p.b)) return false;
    if (need_grads) {
      if (!p.dwc || !p.dbc || !p.dwr || !p.dbr) return false;
      if (s.pre_ln && (!p.dg || !p.db)) return false;
    }
  }
  return true;
}

oases_status cuda_fail(cudaError_t e) {
  t_last_error = cudaGetErrorString(e);
  return OASES_ERR_CUDA;
}

// Runs the given phases (0 forward, 1 recompute + backward) of an n-layer call.
oases_status execute(const Shape& s, int n_layers, const oases_weights* w, const oases_grads* gr,
                     const void* x, void* y, const void* dy, void* dx, void* ws, size_t ws_bytes,
                     void* s0, void* s1, bool fwd, bool bwd, bool stage_host,
                     const void* g_host_or_dev) {
  t_last_error.clear();
  g_launch_count = 0;
  std::vector<Step> steps;
  if (fwd) {
    auto f = schedule(s, 0);
    steps.insert(steps.end(), f.begin(), f.end());
  }
  if (bwd) {
    auto b = schedule(s, 1);
    steps.insert(steps.end(), b.begin(), b.end());
  }
  if (injected(steps)) return OASES_ERR_INJECTED;
  Exec ex;
  ex.s = s;
  ex.L = make_layout(s);
  if (!ws || ws_bytes < ex.L.total) return OASES_ERR_WORKSPACE;
  if (((uintptr_t)ws) % ALIGN != 0) return OASES_ERR_INVALID_ARG;
  ex.ws = static_cast<uint8_t*>(ws);
  ex.st[0] = static_cast<cudaStream_t>(s0);
  ex.st[1] = static_cast<cudaStream_t>(s1);
  ex.sp.resize(s.nseg);
  for (int i = 0; i < s.nseg; ++i) ex.sp[i] = seg_params(s, i, w, gr);
  ex.xparts.assign((size_t)s.nseg * s.nsb, 0);
  ex.aparts.assign((size_t)s.nseg * s.nsb, 0);
  ex.dready.assign((size_t)s.nseg * s.nsb, 0);
  if (!params_ok(s, ex.sp, bwd)) return OASES_ERR_INVALID_ARG;
  const void* io[4] = {x, dy, y, dx};  // device unless staged from host memory
  if (!stage_host)
    for (const void* p : io)
      if (!aligned16(p)) return OASES_ERR_INVALID_ARG;
  const size_t ev_stage = ex.ev_base + (size_t)s.nseg * GRP_N;  // staging-copy events
  ex.P = &pool();
  cudaError_t e = ex.P->ensure(ev_stage + 6 + 2 * (size_t)s.nsb);
  if (e != cudaSuccess) return cuda_fail(e);

  // Host buffers (oases_stack_step only) are staged through the workspace.
  const size_t MH = (size_t)s.M * s.H * s.esz;
  bool host[4] = {false, false, false, false};
  const void* ptrs[4] = {x, g_host_or_dev, y, dx};
  if (stage_host) {
    for (int i = 0; i < 4; ++i) {
      cudaPointerAttributes at{};
      e = cudaPointerGetAttributes(&at, ptrs[i]);
      if (e != cudaSuccess) return cuda_fail(e);
      host[i] = at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeUnregistered;
    }
    for (int i = 0; i < 4; ++i)
      if (!host[i] && !aligned16(io[i])) return OASES_ERR_INVALID_ARG;
  }
  ex.x = host[0] ? ex.at(ex.L.stage[0]) : x;
  ex.dy = host[1] ? ex.at(ex.L.stage[1]) : dy;
  ex.y = host[2] ? ex.at(ex.L.stage[2]) : y;
  ex.dx = host[3] ? ex.at(ex.L.stage[3]) : dx;

  const std::vector<cudaEvent_t>& pev = ex.P->ev;
  cudaEvent_t ev_in = pev[0], ev_out = pev[1];
  cudaEvent_t ev_g = pev[ev_stage + 1];
  cudaEvent_t ev_y[2] = {pev[ev_stage + 2], pev[ev_stage + 3]};
  cudaEvent_t ev_end = pev[ev_stage + 4], ev_cs = pev[ev_stage + 5];
  // per sub-batch: its rows of x landed, its rows of dx final
  auto ev_xs = [&](int b) { return pev[ev_stage + 6 + b]; };
  auto ev_dxs = [&](int b) { return pev[ev_stage + 6 + s.nsb + b]; };
  const size_t MHs = (size_t)s.Ms * s.H * s.esz;  // one sub-batch's rows
  const bool two = ex.st[0] != ex.st[1];
  // Staging copies of host buffers go on a copy stream when nothing is being
  // captured: x first, one sub-batch's rows at a time (each sub-batch's first
  // operator waits for its own rows), then g (waited for only before each
  // stream's first backward operator); y is copied back as soon as both
  // streams finish the forward, each sub-batch's rows of dx as soon as its
  // last operator is done, and s0 joins the copy stream before the call
  // returns.  Under capture they stay on s0.
  const bool any_host = host[0] || host[1] || host[2] || host[3];
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (any_host) ex.ok(cudaStreamIsCapturing(ex.st[0], &cap));
  cudaStream_t cs = (any_host && cap == cudaStreamCaptureStatusNone && MH > 0 && s.M > 0 && bwd)
                        ? copy_stream() : nullptr;
  if (cs) {
    ex.ok(cudaEventRecord(ev_in, ex.st[0]));  // everything the caller enqueued before
    ex.ok(cudaStreamWaitEvent(cs, ev_in, 0));
    if (two) ex.ok(cudaStreamWaitEvent(ex.st[1], ev_in, 0));
    if (host[0])
      for (int b = 0; b < s.nsb; ++b) {
        ex.ok(cudaMemcpyAsync(ex.at<uint8_t>(ex.L.stage[0]) + b * MHs, static_cast<const uint8_t*>(x) + b * MHs,
                              MHs, cudaMemcpyHostToDevice, cs));
        ex.ok(cudaEventRecord(ev_xs(b), cs));
      }
    if (host[1]) {
      ex.ok(cudaMemcpyAsync(ex.at(ex.L.stage[1]), g_host_or_dev, MH, cudaMemcpyHostToDevice, cs));
      ex.ok(cudaEventRecord(ev_g, cs));
    }
  } else {
    if (host[0] && MH) ex.ok(cudaMemcpyAsync(ex.at(ex.L.stage[0]), x, MH, cudaMemcpyHostToDevice, ex.st[0]));
    if (host[1] && MH) ex.ok(cudaMemcpyAsync(ex.at(ex.L.stage[1]), g_host_or_dev, MH, cudaMemcpyHostToDevice, ex.st[0]));
    if (two) {
      ex.ok(cudaEventRecord(ev_in, ex.st[0]));
      ex.ok(cudaStreamWaitEvent(ex.st[1], ev_in, 0));
    }
  }
  const int nstreams = two ? 2 : 1;
  bool in_bwd[2] = {false, false};
  int bwd_started = 0;
  const bool tracing = g_trace_on.load(std::memory_order_relaxed);
  g_trace.clear();
  std::vector<cudaEvent_t>* tevs = nullptr;
  if (tracing) {
    TraceEvents& te = g_trace_events[current_device()];
    const uint64_t id = current_ctx_id();
    if (te.ctx != id) {
      te.ev.clear();  // events of a destroyed context
      te.ctx = id;
    }
    tevs = &te.ev;
  }
  size_t tev = 0;
  std::vector<char> x_waited((size_t)s.nsb, 0);
  if (s.M > 0)
    for (const Step& st : steps) {
      if (cs && host[0] && !x_waited[(size_t)st.sb]) {  // this sub-batch's rows of x
        x_waited[(size_t)st.sb] = 1;
        ex.ok(cudaStreamWaitEvent(ex.stream(st.sb), ev_xs(st.sb), 0));
      }
      TraceRec tr{st.ev, st.op, st.seg, st.sb, nullptr, nullptr};
      if (tracing) {
        while (tevs->size() < tev + 2) {
          cudaEvent_t e;
          if (cudaEventCreate(&e) != cudaSuccess) break;
          tevs->push_back(e);
        }
        if (tevs->size() >= tev + 2) {
          tr.e0 = (*tevs)[tev++];
          tr.e1 = (*tevs)[tev++];
          ex.ok(cudaEventRecord(tr.e0, ex.stream(st.sb)));
        }
      }
      const int si = two ? (st.sb & 1) : 0;
      if (cs && !in_bwd[si] && st.ev != EV_F && st.ev != EV_CF &&
          !(st.ev == EV_SYNC && st.op == OP_G)) {
        // this stream's forward is complete; its backward needs g
        in_bwd[si] = true;
        ex.ok(cudaEventRecord(ev_y[si], ex.st[si]));
        if (host[1]) ex.ok(cudaStreamWaitEvent(ex.st[si], ev_g, 0));
        if (++bwd_started == nstreams && host[2]) {
          for (int k = 0; k < nstreams; ++k) ex.ok(cudaStreamWaitEvent(cs, ev_y[k], 0));
          ex.ok(cudaMemcpyAsync(const_cast<void*>(y), ex.y, MH, cudaMemcpyDeviceToHost, cs));
        }
      }
      ex.run(st);
      if (cs && host[3] && st.ev == EV_B && st.op == OP_LN && st.seg == 0) {
        // the sub-batch's last operator: its rows of dx are final
        ex.ok(cudaEventRecord(ev_dxs(st.sb), ex.stream(st.sb)));
        ex.ok(cudaStreamWaitEvent(cs, ev_dxs(st.sb), 0));
        ex.ok(cudaMemcpyAsync(static_cast<uint8_t*>(dx) + st.sb * MHs, ex.at<uint8_t>(ex.L.stage[3]) + st.sb * MHs,
                              MHs, cudaMemcpyDeviceToHost, cs));
      }
      if (tr.e1) {
        ex.ok(cudaEventRecord(tr.e1, ex.stream(st.sb)));
        g_trace.push_back(tr);
      }
      if (ex.err != cudaSuccess) break;
    }
  if (two) {
    ex.ok(cudaEventRecord(ev_out, ex.st[1]));
    ex.ok(cudaStreamWaitEvent(ex.st[0], ev_out, 0));
  }
  if (cs) {
    if (host[2] && bwd_started < nstreams) {  // no backward operator ran: copy y now
      ex.ok(cudaEventRecord(ev_end, ex.st[0]));
      ex.ok(cudaStreamWaitEvent(cs, ev_end, 0));
      ex.ok(cudaMemcpyAsync(const_cast<void*>(y), ex.y, MH, cudaMemcpyDeviceToHost, cs));
    }
    // (dx went back one sub-batch at a time above)
    ex.ok(cudaEventRecord(ev_cs, cs));
    ex.ok(cudaStreamWaitEvent(ex.st[0], ev_cs, 0));  // completion is signalled on s0
  } else {
    if (host[2] && MH) ex.ok(cudaMemcpyAsync(const_cast<void*>(y), ex.y, MH, cudaMemcpyDeviceToHost, ex.st[0]));
    if (host[3] && MH) ex.ok(cudaMemcpyAsync(dx, ex.dx, MH, cudaMemcpyDeviceToHost, ex.st[0]));
  }
  t_last_launches = g_launch_count;
  if (ex.err != cudaSuccess) return cuda_fail(ex.err);
  return OASES_OK;
}

}  // namespace

namespace oases {
void api_begin() {
  t_last_error.clear();
  g_launch_count = 0;
}
void api_set_error(const char* what) { t_last_error = what; }
oases_status api_end(cudaError_t e) {
  t_last_launches = g_launch_count;
  if (e != cudaSuccess) return cuda_fail(e);
  return OASES_OK;
}
}  // namespace oases

extern "C" {

size_t oases_workspace_bytes(const oases_block_desc* desc, int n_layers) {
  Shape s;
  if (validate(desc, n_layers, &s) != OASES_OK) return 0;
  return make_layout(s).total;
}

oases_status oases_block_fwd(const oases_block_desc* desc, const oases_weights* wts,
                             const void* x, void* y, void* workspace, size_t ws_bytes, void* s0,
                             void* s1) {
  Shape s;
  oases_status r = validate(desc, 1, &s);
  if (r != OASES_OK) return r;
  if (!wts || ((!x || !y) && s.M > 0)) return OASES_ERR_INVALID_ARG;
  return execute(s, 1, wts, nullptr, x, y, nullptr, nullptr, workspace, ws_bytes, s0, s1, true,
                 false, false, nullptr);
}

oases_status oases_block_recompute_bwd(const oases_block_desc* desc, const oases_weights* wts,
                                       const void* x_saved, const void* dy, void* dx,
                                       const oases_grads* grads, void* workspace,
                                       size_t ws_bytes, void* s0, void* s1) {
  Shape s;
  oases_status r = validate(desc, 1, &s);
  if (r != OASES_OK) return r;
  if (!wts || !grads || ((!x_saved || !dy || !dx) && s.M > 0)) return OASES_ERR_INVALID_ARG;
  return execute(s, 1, wts, grads, x_saved, nullptr, dy, dx, workspace, ws_bytes, s0, s1, false,
                 true, false, nullptr);
}

oases_status oases_stack_step(const oases_block_desc* desc, int n_layers,
                              const oases_weights* per_layer, const void* x, const void* g,
                              void* y, void* dx, const oases_grads* per_layer_grads,
                              void* workspace, size_t ws_bytes, void* s0, void* s1) {
  Shape s;
  oases_status r = validate(desc, n_layers, &s);
  if (r != OASES_OK) return r;
  if (!per_layer || !per_layer_grads || ((!x || !g || !y || !dx) && s.M > 0))
    return OASES_ERR_INVALID_ARG;
  return execute(s, n_layers, per_layer, per_layer_grads, x, y, g, dx, workspace, ws_bytes, s0,
                 s1, true, true, s.M > 0, g);
}

const char* oases_status_str(oases_status st) {
  switch (st) {
    case OASES_OK: return "ok";
    case OASES_ERR_INVALID_ARG: return "invalid argument";
    case OASES_ERR_UNSUPPORTED: return "unsupported shape or option";
    case OASES_ERR_WORKSPACE: return "workspace missing or too small";
    case OASES_ERR_CUDA: return "CUDA error";
    case OASES_ERR_TIMEOUT: return "bounded device wait expired";
    case OASES_ERR_INJECTED: return "injected failure (OASES_TEST_FAIL_AT)";
  }
  return "unknown status";
}

const char* oases_last_error(void) { return t_last_error.c_str(); }
const char* oases_version(void) { return "oases-gb300 0.1 (sm_103a)"; }

int oases_schedule_trace(const oases_block_desc* desc, int n_layers, int phase, int32_t* ops,
                         int cap) {
  Shape s;
  if (validate(desc, n_layers, &s) != OASES_OK || (phase != 0 && phase != 1)) return -1;
  std::vector<Step> st = schedule(s, phase);
  for (int i = 0; i < (int)st.size() && i < cap && ops; ++i)
    ops[i] = st[i].ev | (st[i].op << 4) | (st[i].sb << 8) | (st[i].seg << 16);
  return (int)st.size();
}

int oases_last_launch_count(void) { return t_last_launches; }

oases_status oases_shutdown(void) {
  t_last_error.clear();
  int cur = 0;
  if (cudaGetDevice(&cur) != cudaSuccess) cur = -1;
  cudaError_t first = cudaSuccess;
  auto note = [&](cudaError_t e) {
    if (first == cudaSuccess && e != cudaSuccess) first = e;
  };
  // Streams and events of a live context are destroyed with that context's
  // device current (pending work completes first, then CUDA frees them); those
  // of a context that no longer exists are only forgotten.
  auto on_device = [&](int dev, uint64_t ctx, auto&& destroy) {
    if (ctx == 0 || cudaSetDevice(dev) != cudaSuccess) {
      cudaGetLastError();
      return;
    }
    if (current_ctx_id() == ctx) destroy();
  };
  {
    std::lock_guard<std::mutex> lock(g_copy_mu);
    for (auto& kv : g_copy)
      on_device(kv.first, kv.second.ctx, [&] { note(cudaStreamDestroy(kv.second.st)); });
    g_copy.clear();
  }
  for (auto& kv : t_pools) {
    on_device(kv.first, kv.second.ctx, [&] { kv.second.release(); });
    kv.second.ev.clear();
  }
  t_pools.clear();
  for (auto& kv : g_trace_events) {
    on_device(kv.first, kv.second.ctx, [&] { kv.second.release(); });
    kv.second.ev.clear();
  }
  g_trace_events.clear();
  g_trace.clear();
  if (cur >= 0) cudaSetDevice(cur);
  gemm_release_host_caches();
  noalloc_release_host_caches();
  if (first != cudaSuccess) return cuda_fail(first);
  return OASES_OK;
}

oases_status oases_check_device(void* stream) {
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  const int v = gemm_read_and_clear_error(), w = attention_read_and_clear_error(),
            u = norm_read_and_clear_error();
  if (v < 0 || w < 0 || u < 0) return cuda_fail(cudaGetLastError());
  return (v || w || u) ? OASES_ERR_TIMEOUT : OASES_OK;
}

}  // extern "C"

#include "oases_debug.h"

extern "C" oases_status oases_debug_gemm(int M, int N, int K, int in_dtype, const void* A,
                                         int64_t lda, int a_kmajor, const void* B, int64_t ldb,
                                         int b_kmajor, int epilogue, void* C, int64_t ldc,
                                         int c_dtype, void* C2, const void* bias, const void* aux,
                                         int64_t ld_aux, int path, void* stream) {
  using namespace oases;
  t_last_error.clear();
  g_launch_count = 0;
  if (M < 0 || N < 0 || K < 0 || in_dtype < 0 || in_dtype > 1 || c_dtype < 0 || c_dtype > 1 ||
      epilogue < 0 || epilogue > 5 || path < 0 || path > 2)
    return OASES_ERR_INVALID_ARG;
  if ((M > 0 && N > 0) && (!C || (K > 0 && (!A || !B)))) return OASES_ERR_INVALID_ARG;
  const Epi epi = static_cast<Epi>(epilogue);
  if ((epi == Epi::Bias || epi == Epi::BiasGelu || epi == Epi::BiasResid) && !bias)
    return OASES_ERR_INVALID_ARG;
  if ((epi == Epi::BiasResid || epi == Epi::Mul) && !aux) return OASES_ERR_INVALID_ARG;
  if (epi == Epi::Accum && c_dtype != OASES_F32) return OASES_ERR_INVALID_ARG;
  GemmArgs g;
  g.M = M;
  g.N = N;
  g.K = K;
  g.in_t = static_cast<DType>(in_dtype);
  g.A = A;
  g.lda = lda;
  g.a_kmajor = a_kmajor != 0;
  g.B = B;
  g.ldb = ldb;
  g.b_kmajor = b_kmajor != 0;
  g.epi = epi;
  g.C = C;
  g.ldc = ldc;
  g.c_t = static_cast<DType>(c_dtype);
  g.C2 = C2;
  g.bias = bias;
  g.aux = aux;
  g.ld_aux = ld_aux;
  g.aux_t = g.in_t;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (path == 1) {
    e = gemm_simt(g, st);
  } else if (path == 2) {
    if (M == 0 || N == 0) return OASES_OK;
    if (!gemm_tc_supported(g)) return OASES_ERR_UNSUPPORTED;
    e = gemm_tc(g, st);
  } else {
    e = gemm(g, st);
  }
  t_last_launches = g_launch_count;
  if (e != cudaSuccess) return cuda_fail(e);
  return OASES_OK;
}

extern "C" size_t oases_debug_bias_grad_scratch_bytes(int M, int N) {
  if (M < 0 || N < 0) return 0;
  return (size_t)oases::colsum_blocks(M) * (size_t)N * sizeof(float);
}

extern "C" oases_status oases_debug_bias_grad(const void* in, int64_t ld, int M, int N, int dtype,
                                              float* out, void* scratch, size_t scratch_bytes,
                                              void* stream) {
  using namespace oases;
  t_last_error.clear();
  g_launch_count = 0;
  if (M < 0 || N < 0 || dtype < 0 || dtype > 1 || ld < N) return OASES_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return OASES_OK;
  if (!in || !out) return OASES_ERR_INVALID_ARG;
  if (!scratch || scratch_bytes < oases_debug_bias_grad_scratch_bytes(M, N))
    return OASES_ERR_WORKSPACE;
  cudaError_t e = colsum_accum(in, ld, M, N, static_cast<DType>(dtype),
                               static_cast<float*>(scratch), out,
                               static_cast<cudaStream_t>(stream));
  t_last_launches = g_launch_count;
  if (e != cudaSuccess) return cuda_fail(e);
  return OASES_OK;
}

namespace {
size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }
}  // namespace

extern "C" oases_status oases_debug_layer_norm(const void* x, const void* gamma, const void* beta,
                                               void* u, float* mean, float* rstd, int M, int H,
                                               float eps, int dtype, void* stream) {
  using namespace oases;
  t_last_error.clear();
  g_launch_count = 0;
  if (M < 0 || H <= 0 || dtype < 0 || dtype > 1 || !(eps >= 0.f)) return OASES_ERR_INVALID_ARG;
  if (M == 0) return OASES_OK;
  if (!x || !gamma || !beta || !u || !mean || !rstd) return OASES_ERR_INVALID_ARG;
  for (const void* p : {x, gamma, beta, (const void*)u, (const void*)mean, (const void*)rstd})
    if (!aligned16(p)) return OASES_ERR_INVALID_ARG;
  cudaError_t e = layer_norm_fwd(x, gamma, beta, u, mean, rstd, M, H, eps,
                                 static_cast<DType>(dtype), static_cast<cudaStream_t>(stream));
  t_last_launches = g_launch_count;
  if (e != cudaSuccess) return cuda_fail(e);
  return OASES_OK;
}

extern "C" size_t oases_debug_layer_norm_bwd_scratch_bytes(int M, int H) {
  if (M < 0 || H < 0) return 0;
  const size_t part = (size_t)oases::ln_bwd_blocks(M) * (size_t)H * sizeof(float);
  return 2 * round256(part) + round256((size_t)M * 2 * sizeof(float));
}

extern "C" oases_status oases_debug_layer_norm_bwd(const float* du, const void* x, const float* mean,
                                                   const float* rstd, const void* gamma,
                                                   const void* dres, void* dx, float* dgamma,
                                                   float* dbeta, int M, int H, int dtype,
                                                   void* scratch, size_t scratch_bytes,
                                                   void* stream) {
  using namespace oases;
  t_last_error.clear();
  g_launch_count = 0;
  if (M < 0 || H <= 0 || dtype < 0 || dtype > 1) return OASES_ERR_INVALID_ARG;
  if (M == 0) return OASES_OK;
  if (!du || !x || !mean || !rstd || !gamma || !dx || !dgamma || !dbeta)
    return OASES_ERR_INVALID_ARG;
  for (const void* p : {(const void*)du, x, (const void*)mean, (const void*)rstd, gamma, dres,
                        (const void*)dx, (const void*)dgamma, (const void*)dbeta})
    if (!aligned16(p)) return OASES_ERR_INVALID_ARG;
  if (!scratch || scratch_bytes < oases_debug_layer_norm_bwd_scratch_bytes(M, H) ||
      !aligned16(scratch))
    return OASES_ERR_WORKSPACE;
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  const size_t part = round256((size_t)ln_bwd_blocks(M) * (size_t)H * sizeof(float));
  cudaError_t e = layer_norm_bwd(du, x, mean, rstd, gamma, dres, dx, reinterpret_cast<float*>(sc),
                                 reinterpret_cast<float*>(sc + part),
                                 reinterpret_cast<float2*>(sc + 2 * part), dgamma, dbeta, M, H,
                                 static_cast<DType>(dtype), static_cast<cudaStream_t>(stream));
  t_last_launches = g_launch_count;
  if (e != cudaSuccess) return cuda_fail(e);
  return OASES_OK;
}

extern "C" oases_status oases_debug_shard_sum(const float* part, int64_t pstride, int w,
                                              const void* bias, const void* resid, void* out,
                                              int M, int N, int dtype, void* stream) {
  using namespace oases;
  t_last_error.clear();
  g_launch_count = 0;
  if (M < 0 || N < 0 || w <= 0 || dtype < 0 || dtype > 1) return OASES_ERR_INVALID_ARG;
  if ((int64_t)M * N == 0) return OASES_OK;
  if (!part || !out || pstride < (int64_t)M * N) return OASES_ERR_INVALID_ARG;
  for (const void* p : {(const void*)part, bias, resid, (const void*)out})
    if (!aligned16(p)) return OASES_ERR_INVALID_ARG;
  const DType t = static_cast<DType>(dtype);
  cudaError_t e = shard_sum(part, pstride, w, bias, resid, out, t, t, M, N,
                            static_cast<cudaStream_t>(stream));
  t_last_launches = g_launch_count;
  if (e != cudaSuccess) return cuda_fail(e);
  return OASES_OK;
}

extern "C" oases_status oases_debug_attention(const void* qkv, void* o, float* lse, const void* d_o,
                                              float* delta, void* dqkv, int batch, int seq,
                                              int heads, int head_dim, int causal, int dtype,
                                              int backward, int path, void* stream) {
  using namespace oases;
  t_last_error.clear();
  g_launch_count = 0;
  if (batch < 0 || seq < 0 || heads <= 0 || head_dim <= 0 || dtype < 0 || dtype > 1 ||
      path < 0 || path > 2)
    return OASES_ERR_INVALID_ARG;
  if (head_dim > 128 || head_dim % 8 != 0) return OASES_ERR_UNSUPPORTED;
  AttnArgs a;
  a.batch = batch;
  a.seq = seq;
  a.heads = heads;
  a.head_dim = head_dim;
  a.hidden = heads * head_dim;
  a.causal = causal != 0;
  a.t = static_cast<DType>(dtype);
  a.qkv = qkv;
  a.o = o;
  a.lse = lse;
  a.d_o = d_o;
  a.delta = delta;
  a.dqkv = dqkv;
  if ((int64_t)batch * seq > 0 && (!qkv || !o || !lse)) return OASES_ERR_INVALID_ARG;
  if (backward && (int64_t)batch * seq > 0 && (!d_o || !delta || !dqkv))
    return OASES_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (!backward) {
    if (path == 2 && !attention_tc_supported(a)) return OASES_ERR_UNSUPPORTED;
    e = path == 1 ? attention_fwd_simt(a, st) : path == 2 ? attention_fwd_tc(a, st)
                                                        : attention_fwd(a, st);
  } else {
    e = path == 1 ? attention_bwd_simt(a, st) : attention_bwd(a, st);
  }
  t_last_launches = g_launch_count;
  if (e != cudaSuccess) return cuda_fail(e);
  return OASES_OK;
}

extern "C" oases_status oases_debug_attention_progress(int* host_mapped) {
  cudaError_t e = oases::attention_set_progress(host_mapped);
  if (e != cudaSuccess) return cuda_fail(e);
  return OASES_OK;
}

extern "C" oases_status oases_debug_attention_timeline(unsigned long long* device_buffer) {
  cudaError_t e = oases::attention_set_timeline(device_buffer);
  if (e != cudaSuccess) return cuda_fail(e);
  return OASES_OK;
}

extern "C" int oases_debug_attention_error_word(void) {
  return oases::attention_read_and_clear_error();
}

namespace oases {
cudaError_t attention_wait_probe(uint64_t limit_cycles, cudaStream_t st);
}
extern "C" oases_status oases_debug_wait_probe(uint64_t limit_cycles, void* stream) {
  t_last_error.clear();
  if (limit_cycles == 0 || limit_cycles > (1ull << 32)) {
    t_last_error = "limit_cycles must be in 1 .. 2^32";
    return OASES_ERR_INVALID_ARG;
  }
  cudaError_t e = oases::attention_wait_probe(limit_cycles, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e);
  return OASES_OK;
}

namespace oases {
cudaError_t gemm_set_timeline(unsigned long long* p);
}
extern "C" oases_status oases_debug_gemm_timeline(unsigned long long* device_buffer) {
  cudaError_t e = oases::gemm_set_timeline(device_buffer);
  if (e != cudaSuccess) return cuda_fail(e);
  return OASES_OK;
}

extern "C" void oases_debug_trace_enable(int on) { g_trace_on = on != 0; }

extern "C" int oases_debug_trace_read(double* out, int cap) {
  if (g_trace.empty()) return 0;
  for (const TraceRec& r : g_trace)
    if (cudaEventSynchronize(r.e1) != cudaSuccess) return -1;
  const cudaEvent_t t0 = g_trace.front().e0;
  const int n = (int)g_trace.size();
  for (int i = 0; i < n && i < cap; ++i) {
    const TraceRec& r = g_trace[i];
    float a = 0.f, b = 0.f;
    cudaEventElapsedTime(&a, t0, r.e0);
    cudaEventElapsedTime(&b, t0, r.e1);
    double* o = out + 6 * i;
    o[0] = r.ev;
    o[1] = r.op;
    o[2] = r.seg;
    o[3] = r.sb;
    o[4] = a * 1e3;
    o[5] = b * 1e3;
  }
  return n;
}
