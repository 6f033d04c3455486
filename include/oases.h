/*
 * oases.h — C ABI of the GB300 library for the Oases tensor-parallel block.
 *
 * What it computes.  The forward, fine-grained recompute and backward of a
 * Megatron-style tensor-parallel transformer block on one GPU, after
 * "Oases: Efficient Large-Scale Model Training on Commodity Servers via
 * Overlapped and Automated Tensor Model Parallelism" (arXiv 2305.16121):
 *   - §IV-A, Fig. 4a: a segment is the operator sequence (F_i, C_i(F), F_j):
 *     a column-parallel F_i (LayerNorm, then W1 + bias + GeLU for an FFN, or
 *     the QKV projection + causal softmax attention), a row-parallel F_j (W2 or
 *     Wo), and the AllReduce C_i over the w shards.
 *   - §IV, Eq. (1): C_i is y = sum_{k<w} P_k, so dy/dP_k = 1.  All w shards live
 *     on this GPU; the sum is accumulated on chip (the row GEMM's contraction
 *     runs over every shard's K-slice into one accumulator) and the backward of
 *     C_i is the identity.  The input-gradient AllReduce C_i(B) is likewise the
 *     contraction over all shards of the column GEMM's input gradient.
 *   - §IV, Fig. 4d: fine-grained recomputation starts after the communication
 *     operator and never recomputes C_i (mode OASES_RECOMPUTE_FINE).
 *   - §IV, Fig. 4b and Algorithm 1: the batch is split into sub-batches that are
 *     pipelined on two CUDA streams; sub-batch b runs on stream b % 2.
 *
 * Conventions (all entry points).
 *   Layout    row-major.  x, y, dx, dy, g are [batch*seq, hidden] with the batch
 *             outermost, so sub-batch b is the contiguous row range
 *             [b*M/n_sb, (b+1)*M/n_sb).  Weights are in nn.Linear layout
 *             [out_features, in_features]: w1 [ffn, hidden], w2 [hidden, ffn],
 *             wqkv [3*hidden, hidden] with rows [Q heads | K heads | V heads],
 *             head h at rows h*d .. h*d+d-1 of each part, wo [hidden, hidden].
 *             Shard k owns rows [k*ffn/w, (k+1)*ffn/w) of w1 (the same columns of
 *             w2), or heads [k*heads/w, (k+1)*heads/w); one weight buffer
 *             therefore serves every w.
 *   Types     x, y, dx, dy, g and weights have the type desc->dtype (fp32 or
 *             bf16).  Gradients of weights are fp32 and are ACCUMULATED (+=):
 *             the caller zeroes them.  All arithmetic accumulates in fp32.
 *   Memory    The caller owns every buffer.  The library never allocates or
 *             frees device memory; it uses only the caller's workspace, whose
 *             size oases_workspace_bytes() returns.  Device pointers must be
 *             16-byte aligned.  It keeps a small pool of CUDA events per host
 *             thread and device and, for host-buffer steps, one copy stream
 *             per device.
 *   Threads   Calls from several host threads may run concurrently on
 *             different workspaces and streams, on one device or several; a
 *             workspace must not be used by two calls whose work overlaps.
 *   Streams   s0 and s1 are cudaStream_t (NULL = legacy default stream).  Calls
 *             are asynchronous: on return the work is enqueued.  s1 first waits
 *             for the work already enqueued on s0, and before returning s0 is
 *             made to wait for everything enqueued on s1, so completion of s0
 *             means completion of the call.
 *   Errors    Argument and shape errors are returned synchronously before any
 *             launch (nothing is enqueued).  A failed launch returns
 *             OASES_ERR_CUDA; the CUDA error string is kept and returned by
 *             oases_last_error().  The library never prints and never exits.
 *   Determinism  Identical inputs give bit-identical outputs (no atomics; weight
 *             gradients are accumulated in sub-batch order 0, 1, ...).
 */
#ifndef OASES_H
#define OASES_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OASES_OK = 0,
  OASES_ERR_INVALID_ARG = 1,  /* NULL pointer, negative size, inconsistent shape */
  OASES_ERR_UNSUPPORTED = 2,  /* valid request the library does not implement */
  OASES_ERR_WORKSPACE = 3,    /* workspace NULL or smaller than oases_workspace_bytes() */
  OASES_ERR_CUDA = 4,         /* a CUDA call failed; see oases_last_error() */
  OASES_ERR_TIMEOUT = 5,      /* a bounded device-side wait gave up */
  OASES_ERR_INJECTED = 6      /* test hook OASES_TEST_FAIL_AT matched an operator */
} oases_status;

typedef enum { OASES_BLOCK_FFN = 0, OASES_BLOCK_ATTN = 1, OASES_BLOCK_LAYER = 2 } oases_block_kind;
/* F32, BF16: storage and GEMM operand type of x, y, weights and activations
 * (fp32 accumulation, fp32 weight gradients).
 * MXFP8: storage as BF16, and every GEMM of the block (the column-parallel F_i,
 *        the row-parallel F_j, their input-gradient and weight-gradient
 *        products) multiplies MX-FP8 operands: E4M3 elements with one UE8M0
 *        scale per 32 elements along the contraction, quantised from the
 *        stored bf16 operands just before each GEMM (oases_mx.h), fp32
 *        accumulation.  The attention operation itself stays bf16.  The pages
 *        describe no 8-bit form; this variant follows the OCP Microscaling
 *        Formats v1.0 definitions.  Requires the FUSED reduction, hidden, ffn/w
 *        and hidden/w multiples of 32. */
typedef enum { OASES_F32 = 0, OASES_BF16 = 1, OASES_MXFP8 = 2 } oases_dtype;
/* NONE: keep every activation between forward and backward, no recompute.
 * FULL: keep only segment inputs; recompute the whole segment including the
 *       row GEMM and its reduction (Oases §IV-A, Fig. 4a, the default schedule).
 * FINE: keep only segment inputs; recompute LayerNorm and the column-parallel
 *       part only: C_i(R) and the row GEMM feeding it are not recomputed
 *       (Oases §IV, Eq. (1), Fig. 4d).
 * SELECTIVE: keep every activation except the output of the attention
 *       operation (O and its log-sum-exp), which is recomputed from the kept
 *       Q, K, V before the attention segment's backward: the selective
 *       recomputation the pages compare against (§VI, "Megatron SS").  FFN
 *       segments keep everything, as in NONE. */
typedef enum {
  OASES_RECOMPUTE_NONE = 0,
  OASES_RECOMPUTE_FULL = 1,
  OASES_RECOMPUTE_FINE = 2,
  OASES_RECOMPUTE_SELECTIVE = 3
} oases_recompute;
/* How the shard sums C_i(F) (and C_i(R)) and C_i(B) are formed (Oases §IV,
 * Eq. (1): y = sum_k P_k over the w shards).
 * FUSED:    the row GEMM contracts over every shard's K-slice into one TMEM
 *           accumulator (and the input-gradient GEMM likewise), so the sum
 *           never leaves the chip.
 * SEPARATE: each shard's partial P_k (its own K-slice only) is written to HBM
 *           as fp32, and a separate memory-bound reduction kernel forms the
 *           sum at the communication step — the on-device analogue of the
 *           AllReduce, which one sub-batch runs while the other computes. */
typedef enum { OASES_REDUCE_FUSED = 0, OASES_REDUCE_SEPARATE = 1 } oases_reduce;

typedef struct {
  int32_t kind;         /* oases_block_kind */
  int32_t dtype;        /* oases_dtype */
  int32_t batch;        /* sequences; >= 0, divisible by sub_batches */
  int32_t seq;          /* tokens per sequence; >= 0 */
  int32_t hidden;       /* > 0; a multiple of 8 for bf16, of 32 for MXFP8 */
  int32_t ffn;          /* FFN width (ffn/layer kinds); divisible by w; multiple of 8 for bf16 */
  int32_t heads;        /* attention heads (attn/layer kinds); divisible by w */
  int32_t w;            /* simulated tensor-parallel shards, >= 1 */
  int32_t sub_batches;  /* >= 1 */
  int32_t pre_ln;       /* 1: LayerNorm before each segment */
  int32_t residual;     /* 1: y = segment(x) + x */
  int32_t causal;       /* 1: causal attention mask (key j visible from query i iff j <= i) */
  int32_t recompute;    /* oases_recompute */
  int32_t reduce;       /* oases_reduce */
  float ln_eps;         /* LayerNorm epsilon (biased variance) */
} oases_block_desc;

/* Parameters of one layer, in desc->dtype, device memory.  A segment reads only
 * its own: attention uses ln1_*, wqkv, bqkv, wo, bo; FFN uses ln2_*, w1, b1, w2,
 * b2.  Unused pointers may be NULL; LayerNorm pointers may be NULL when
 * pre_ln == 0. */
typedef struct {
  const void *ln1_g, *ln1_b, *wqkv, *bqkv, *wo, *bo;
  const void *ln2_g, *ln2_b, *w1, *b1, *w2, *b2;
} oases_weights;

/* fp32 gradients, same shapes as oases_weights, accumulated (+=). */
typedef struct {
  float *ln1_g, *ln1_b, *wqkv, *bqkv, *wo, *bo;
  float *ln2_g, *ln2_b, *w1, *b1, *w2, *b2;
} oases_grads;

/* Bytes of workspace a call with this descriptor needs: for oases_block_fwd /
 * oases_block_recompute_bwd pass n_layers = 1 (the same workspace must be given
 * to the forward and to the backward that follows it: it carries the stored
 * activations); for oases_stack_step pass its n_layers.  Returns 0 if the
 * descriptor is invalid. */
size_t oases_workspace_bytes(const oases_block_desc *desc, int n_layers);

/* Forward of one block (Oases §IV-A: F_i, C_i(F), F_j of every segment):
 * y = block(x).  x, y: device, [batch*seq, hidden], desc->dtype; x must stay
 * unchanged until the matching oases_block_recompute_bwd, which reads it again
 * as the stored input of the first recompute sequence. */
oases_status oases_block_fwd(const oases_block_desc *desc, const oases_weights *wts,
                             const void *x, void *y, void *workspace, size_t ws_bytes,
                             void *s0, void *s1);

/* Recompute + backward of one block after oases_block_fwd (Oases §IV, Fig. 4d,
 * Algorithm 1 backward): per segment in reverse, R (LayerNorm and column part;
 * FULL also the row GEMM and its reduction), B_j (row GEMM dgrad/wgrad), B_i
 * (column GEMM dgrad/wgrad, attention backward), C_i(B) (sum over shards of the
 * input gradient), LayerNorm backward and residual.
 * x_saved: the x given to the forward.  dy: gradient of the loss w.r.t. y.
 * dx: output, gradient w.r.t. x.  grads: fp32, accumulated. */
oases_status oases_block_recompute_bwd(const oases_block_desc *desc, const oases_weights *wts,
                                       const void *x_saved, const void *dy, void *dx,
                                       const oases_grads *grads, void *workspace, size_t ws_bytes,
                                       void *s0, void *s1);

/* One training step of an n_layers stack of identical blocks with loss
 * L = sum(y * g): forward through every layer (segment inputs kept as the
 * recompute checkpoints), then the reverse cross-layer recompute + backward
 * (Oases §IV: the backward schedule runs across layers).
 * per_layer: n_layers weight structs; per_layer_grads: n_layers grad structs.
 * x, g, y, dx: [batch*seq, hidden] in desc->dtype; each may be device memory or
 * host memory (pageable or pinned): host buffers are staged through the
 * workspace with cudaMemcpyAsync.  Outside stream capture the copies run on a
 * copy stream the library creates once per device, ordered by events: x is
 * uploaded before any compute, g before each stream's first backward
 * operator, y is downloaded once the forward is done (overlapping the
 * backward) and dx at the end.  While s0 is being captured into a CUDA graph
 * they are issued on s0 instead.  Either way y and dx are complete in host
 * memory once s0 completes. */
oases_status oases_stack_step(const oases_block_desc *desc, int n_layers,
                              const oases_weights *per_layer, const void *x, const void *g,
                              void *y, void *dx, const oases_grads *per_layer_grads,
                              void *workspace, size_t ws_bytes, void *s0, void *s1);

/* Static description of a status code. */
const char *oases_status_str(oases_status st);
/* Text of the last CUDA error seen by a call on this thread ("" if none). */
const char *oases_last_error(void);
/* Library version string. */
const char *oases_version(void);

/* Host-side schedule of a call, without launching anything: writes at most
 * cap entries into ops and returns the number of entries the schedule has
 * (may exceed cap), or -1 on an invalid descriptor.  phase: 0 = forward,
 * 1 = recompute + backward, of an n_layers stack.  An entry packs:
 *   event  = e & 0xF         0 F, 1 R, 2 B (compute operations),
 *                            3 C(F), 4 C(R), 5 C(B) (communication started),
 *                            6 Sync (the sub-batch waits for its communication)
 *   op     = (e >> 4) & 0xF  0 ln, 1 f, 2 col, 3 row, 4 g, 5 attn (the attention
 *                            operation alone, recomputed in SELECTIVE mode)
 *   sub    = (e >> 8) & 0xFF sub-batch
 *   seg    = e >> 16         segment (layer * segments_per_layer + index)
 * On one GPU a "communication" is the on-chip shard sum; Sync is the event
 * wait a stream performs before it reads that sum. */
#define OASES_TRACE_EVENT(e) ((e) & 0xF)
#define OASES_TRACE_OP(e) (((e) >> 4) & 0xF)
#define OASES_TRACE_SUB(e) (((e) >> 8) & 0xFF)
#define OASES_TRACE_SEG(e) ((e) >> 16)
int oases_schedule_trace(const oases_block_desc *desc, int n_layers, int phase,
                         int32_t *ops, int cap);

/* Number of kernel launches the last call on this thread enqueued. */
int oases_last_launch_count(void);

/* Releases the host-side state the library keeps between calls: the copy
 * stream it made per device for host-buffer staging, the calling thread's
 * CUDA events (per device), the event timeline of the trace aid and the host
 * caches of tensor maps and device addresses.  Work already enqueued is not
 * waited for: CUDA frees a stream or event once its pending work completes.
 * No device memory is involved (the library never allocates any).  Events
 * that other host threads made are released when those threads exit.  Call it
 * while no other thread is inside a library call, and before cudaDeviceReset
 * (state of a context that no longer exists is dropped, not reused, either
 * way).  Any later call makes what it needs again.  Returns OASES_ERR_CUDA if
 * destroying a stream or event failed (everything is released regardless).
 * The pages fix no API; this is the release half of the executor's cached
 * state (Oases §IV, the runtime executor). */
oases_status oases_shutdown(void);

/* Synchronizes the stream, then reports whether a bounded device-side wait of
 * a tensor-core kernel expired since the last check (OASES_ERR_TIMEOUT; the
 * error word is cleared), or a CUDA error occurred (OASES_ERR_CUDA). */
oases_status oases_check_device(void *stream);

#ifdef __cplusplus
}
#endif
#endif /* OASES_H */
