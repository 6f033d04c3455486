/*
 * oases_debug.h — kernel-level entry points of liboases.so, for testing the
 * building blocks of the Oases block in isolation.
 *
 * The column-parallel F_i and row-parallel F_j of a segment (Oases, arXiv
 * 2305.16121, §IV-A, Fig. 4a) and all their backward products are GEMMs of the
 * form below with a fused epilogue; oases_debug_gemm runs exactly the kernel
 * the block uses for such a product.
 */
#ifndef OASES_DEBUG_H
#define OASES_DEBUG_H

#include <stdint.h>

#include "oases.h"

#ifdef __cplusplus
extern "C" {
#endif

/* D[m, n] = sum_k A(m, k) * B(n, k) for m < M, n < N, k < K, then epilogue:
 *   0 Store      C = D
 *   1 Bias       C = D + bias[n]
 *   2 BiasGelu   C = gelu(D + bias[n]); C2 = gelu'(D + bias[n]) (if C2 != NULL)
 *   3 BiasResid  C = D + bias[n] + aux[m * ld_aux + n]
 *   4 Mul        C = D * aux[m * ld_aux + n]  (GeLU backward: aux = the stored gelu')
 *   5 Accum      C (fp32) += D
 * A(m, k) = a_kmajor ? A[m * lda + k] : A[k * lda + m]; B(n, k) likewise with
 * b_kmajor / ldb.  A, B, bias and aux have type in_dtype (oases_dtype); C and
 * C2 have type c_dtype, leading dimension ldc.  All pointers are device
 * memory.  path: 0 = the block's own choice, 1 = CUDA-core kernel,
 * 2 = tensor-core kernel (OASES_ERR_UNSUPPORTED if the operands do not meet
 * its rules: bf16, K > 0, lda and ldb multiples of 8, 16-byte aligned A, B).
 * Asynchronous on stream. */
oases_status oases_debug_gemm(int M, int N, int K, int in_dtype, const void *A, int64_t lda,
                              int a_kmajor, const void *B, int64_t ldb, int b_kmajor, int epilogue,
                              void *C, int64_t ldc, int c_dtype, void *C2, const void *bias,
                              const void *aux, int64_t ld_aux, int path, void *stream);

/* Causal softmax attention of the attention segment's F_i (Oases §IV-A: the
 * column-parallel attention layer; each shard owns heads, and heads are
 * independent, so all shards' heads run in one call):
 *   O_h = softmax(Q_h K_h^T / sqrt(d) + mask) V_h, LSE_h = log sum exp
 * per sequence and head, mask: key j visible from query i iff j <= i when
 * causal.  qkv: device [batch*seq, 3*heads*head_dim], rows of one sequence
 * contiguous, Q of head h at column h*d, K at H + h*d, V at 2H + h*d
 * (H = heads*head_dim).  o: [batch*seq, H]; lse: fp32 [heads, batch*seq].
 * backward = 1: from d_o ([batch*seq, H]) and the forward's o and lse, writes
 * delta (fp32 [heads, batch*seq], rowsum(d_o * o)) and dqkv ([batch*seq, 3H],
 * gradients of Q, K, V in qkv's layout).  dtype: oases_dtype of qkv, o, d_o,
 * dqkv.  path: 0 = the block's choice, 1 = CUDA-core kernels, 2 = tensor-core
 * kernels (bf16, head_dim 128; OASES_ERR_UNSUPPORTED otherwise).
 * Asynchronous on stream. */
oases_status oases_debug_attention(const void *qkv, void *o, float *lse, const void *d_o,
                                   float *delta, void *dqkv, int batch, int seq, int heads,
                                   int head_dim, int causal, int dtype, int backward, int path,
                                   void *stream);

/* Debugging aids for the tensor-core attention kernels.
 * oases_debug_attention_progress: host_mapped is a device-accessible host
 * buffer of 768 ints (pinned) or NULL; when set, thread 0 of CTA c of kernel k
 * (0 forward, 1 dQ, 2 dK/dV) writes its current stage to host_mapped[256k + c]
 * as it goes, which lets a host watchdog see where a stalled kernel stands.
 * oases_debug_attention_error_word: reads and clears the code of the first
 * bounded wait that gave up (kernel * 100 + site; 0 = none, -1 = unreadable). */
oases_status oases_debug_attention_progress(int *host_mapped);
/* Timeline of the tensor-core attention kernels (debugging aid): device_buffer
 * holds uint64 %globaltimer stamps, written by every following launch.
 * Backward: for the persistent dQ kernel, the start (first S and dP MMAs
 * issued) and end (dQ stored) of each work item i < 4096 (128 queries of one
 * sequence and head, numbered heaviest first) at [2i]; entry and exit of each
 * dK/dV CTA c < 4096 at [8192 + 2c]; for CTA 0 (dQ: its first item) and
 * block j < 64, four stamps at
 * [16384 + 4j] (dQ) and [16640 + 4j] (dK/dV): S and dP MMAs issued,
 * accumulation MMAs issued, element-wise warp 2 saw S and dP, and handed over
 * its rows.  Forward (persistent; an item is 256 queries of one sequence and
 * head, items numbered heaviest first): for the first item of CTA 0, query
 * tile t (0, 1) and key block j < 64, eight stamps at [16896 + 8 (64 t + j)]:
 * S_t(j) issued, the softmax warp of lane quarter 2 saw S_t(j), the warps of
 * lane quarters 0..3 published P_t(j), PV_t(j) issued, PV_t(j) about to be
 * issued (its P and V ready); for every item
 * i < 4096, eight stamps at [17920 + 8i]: its CTA's entry, its CTA set up, Q
 * and K_0 of the item landed, tile 0's softmax saw S_0(0), tile 0's and tile
 * 1's last PV complete, tile 1's O stored, its CTA's exit; at [50688 ..
 * 50691] CTA 0's globaltimer and clock64 at its entry and exit (their deltas
 * give the SM clock).  The buffer then holds 50692 stamps.  NULL switches it
 * off. */
oases_status oases_debug_attention_timeline(unsigned long long *device_buffer);
/* Timeline of the tensor-core GEMM (debugging aid): device_buffer holds 16
 * uint64 %globaltimer stamps per CTA of every following launch (entry,
 * prologue done, first stage landed, then per local tile t < 5 its last MMA
 * issued and its epilogue done, exit); NULL switches it off. */
oases_status oases_debug_gemm_timeline(unsigned long long *device_buffer);
int oases_debug_attention_error_word(void);
/* Failure-detection probe: launches one thread that waits, with the bounded
 * mbarrier wait the tensor-core kernels use, on a barrier nothing arrives on.
 * The wait gives up after limit_cycles SM clocks (1 .. 2^32; about 2 ms at
 * 2^22) and records error site 999, so the next oases_check_device on that
 * stream returns OASES_ERR_TIMEOUT while the CUDA context stays usable.
 * Returns OASES_ERR_INVALID_ARG for a limit out of range (nothing launched). */
oases_status oases_debug_wait_probe(uint64_t limit_cycles, void *stream);

/* Per-operator timeline of the block scheduler (debugging aid).  With
 * tracing on (a process-wide switch), every following block call records a
 * timing event before and after each scheduled step (Algorithm 1 operator of
 * one sub-batch) on that sub-batch's stream.  oases_debug_trace_read
 * synchronizes the events of the calling thread's last block call and writes
 * 6 doubles per step into out: event, operator, segment, sub-batch, start and
 * end in microseconds from the first step's start; it returns the number of
 * steps of that call (entries beyond cap are not written), or -1 on a CUDA
 * error.  Tracing adds two event records per step. */
void oases_debug_trace_enable(int on);
int oases_debug_trace_read(double *out, int cap);

/* Bias gradient of a linear layer, as the block takes it: by Oases §IV,
 * Eq. (1) every shard's partial receives the same output gradient dY, and the
 * row-parallel bias (added once after the shard sum) gets
 *   out[n] += sum_{m < M} in[m * ld + n],   n < N,
 * (also used for the column-parallel bias with in = dA).  Deterministic:
 * blocks of 32 rows are summed into partial rows in scratch, then the partial
 * rows are added in a fixed order.  in: device, type dtype (oases_dtype), leading
 * dimension ld >= N.  out: device fp32 [N], accumulated.  scratch: device,
 * at least oases_debug_bias_grad_scratch_bytes(M, N) bytes, owned by the
 * caller.  Asynchronous on stream. */
size_t oases_debug_bias_grad_scratch_bytes(int M, int N);
oases_status oases_debug_bias_grad(const void *in, int64_t ld, int M, int N, int dtype, float *out,
                                   void *scratch, size_t scratch_bytes, void *stream);

/* LayerNorm forward of a pre-LN segment (the normalisation in front of F_i;
 * under fine-grained recomputation it is part of R_i, Oases §IV-A, Fig. 4):
 *   u[m, h] = (x[m, h] - mean[m]) * rstd[m] * gamma[h] + beta[h],
 *   mean[m] = (1/H) sum_h x[m, h], rstd[m] = 1 / sqrt((1/H) sum_h (x[m, h] - mean[m])^2 + eps).
 * x, u: device [M, H] row-major (pitch H), type dtype (oases_dtype); gamma,
 * beta: device [H], type dtype; mean, rstd: device fp32 [M], written.  Every
 * pointer 16-byte aligned (OASES_ERR_INVALID_ARG otherwise).  Asynchronous on
 * stream. */
oases_status oases_debug_layer_norm(const void *x, const void *gamma, const void *beta, void *u,
                                    float *mean, float *rstd, int M, int H, float eps, int dtype,
                                    void *stream);

/* LayerNorm backward, the last step of the block's C_i(B) (Oases §IV-A,
 * Fig. 4d: the input gradient of a segment flows through its LayerNorm):
 * with xhat = (x - mean) * rstd and gg = du * gamma per row,
 *   dx[m, h] = rstd[m] * (gg[m, h] - mean_h(gg) - xhat[m, h] * mean_h(gg * xhat)) (+ dres[m, h]),
 *   dgamma[h] += sum_m du[m, h] * xhat[m, h],  dbeta[h] += sum_m du[m, h].
 * du: device fp32 [M, H]; x, gamma, dres (NULL: no residual term), dx: type
 * dtype; mean, rstd: the forward's fp32 [M]; dgamma, dbeta: device fp32 [H],
 * accumulated in a fixed order (bit-reproducible).  scratch: device, at least
 * oases_debug_layer_norm_bwd_scratch_bytes(M, H) bytes, owned by the caller
 * (OASES_ERR_WORKSPACE otherwise).  Every pointer 16-byte aligned.
 * Asynchronous on stream. */
size_t oases_debug_layer_norm_bwd_scratch_bytes(int M, int H);
oases_status oases_debug_layer_norm_bwd(const float *du, const void *x, const float *mean,
                                        const float *rstd, const void *gamma, const void *dres,
                                        void *dx, float *dgamma, float *dbeta, int M, int H,
                                        int dtype, void *scratch, size_t scratch_bytes,
                                        void *stream);

/* The shard sum C_i(F) of the separate-reduction mode (Oases §IV, Eq. (1):
 * the row-parallel output is the sum of the w shards' partial outputs):
 *   out[m, n] = sum_{k < w} part[k * pstride + m * N + n] (+ bias[n]) (+ resid[m * N + n]),
 * shards added in the order k = 0, 1, ..., then the bias, then the residual.
 * part: device fp32, w slabs of [M, N] with pstride >= M * N floats between
 * them; bias [N], resid [M, N] (either may be NULL) and out [M, N]: type
 * dtype.  Every pointer 16-byte aligned.  Asynchronous on stream. */
oases_status oases_debug_shard_sum(const float *part, int64_t pstride, int w, const void *bias,
                                   const void *resid, void *out, int M, int N, int dtype,
                                   void *stream);

/* The bias-gradient sum above for callers that cannot allocate device memory.
 * The paper has no counterpart to this entry point; it exists for callers such
 * as a plugin inside a host framework that owns every device allocation, a
 * real-time loop where cudaMalloc's implicit device synchronisation is not
 * acceptable, or code that must not grow its memory footprint after start-up.
 *
 * Same arguments and result as oases_debug_bias_grad, without the scratch
 * argument: the partial rows live in a static device array of
 * OASES_NOALLOC_SCRATCH_FLOATS fp32 values (4 MiB) that every GPU which loads
 * the library keeps until the process exits.  Sizes whose partial rows do not
 * fit, ceil(M / 32) * N > OASES_NOALLOC_SCRATCH_FLOATS, are rejected with
 * OASES_ERR_UNSUPPORTED before anything is enqueued (oases_last_error() says
 * how many floats were needed).  Nothing is allocated or freed, by this call
 * or by any library routine it uses.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture.  The address is kept per device together with the CUDA
 * context it belongs to: after a cudaDeviceReset (or after oases_shutdown())
 * the next call looks it up again, so that call too should come before any
 * capture.  All calls on a device share the one array, which keeps
 * the previous call's contents (every value it reads is written first by the
 * same call): calls whose executions overlap on the GPU (for instance on two
 * streams without ordering between them) race on the array and give wrong
 * results.  Asynchronous on stream. */
#define OASES_NOALLOC_SCRATCH_FLOATS (1u << 20)
oases_status oases_bias_grad_noalloc(const void *in, int64_t ld, int M, int N, int dtype,
                                     float *out, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* OASES_DEBUG_H */
