/*
 * oases_mx.h — MX-FP8 variant of the block's GEMMs (liboases.so).
 *
 * The column-parallel F_i and row-parallel F_j of a segment and their backward
 * products (Oases, arXiv 2305.16121, §IV-A, Fig. 4a) are GEMMs; the pages give
 * them in the training precision only and describe no 8-bit form.  This is
 * that GEMM with both operands in the OCP Microscaling (MX) FP8 format (OCP
 * Microscaling Formats Specification v1.0): E4M3 elements (1 sign, 4 exponent
 * bits with bias 7, 3 mantissa bits; largest finite 448, no infinity) and one
 * UE8M0 power-of-two scale per 32 consecutive elements along the contraction,
 * multiplied on the 5th-generation tensor cores (tcgen05.mma kind::mxf8f6f4
 * with block scaling) and accumulated in fp32.
 *
 * Operand layout.  An MX operand with `rows` rows and contraction length K is
 *   codes  [rows, K] uint8 E4M3 codes, row-major, leading dimension ldq bytes
 *          (a multiple of 16, >= K), 16-byte aligned;
 *   scales oases_mx_scale_bytes(rows, K) bytes of UE8M0 scale bytes (value
 *          2^(byte - 127)) in 512-byte tiles: tile (rb, kg) covers rows
 *          128 rb .. +127 and K blocks 4 kg .. +3 and starts at byte
 *          (rb * ceil(K / 128) + kg) * 512; inside it, row r and block j sit
 *          at byte (r % 32) * 16 + (r / 32) * 4 + j.  Rows and blocks past the
 *          matrix hold 127.  16-byte aligned.
 * All pointers are device memory owned by the caller; nothing is allocated.
 * Calls are asynchronous on `stream`; argument errors are returned before
 * anything is enqueued.
 */
#ifndef OASES_MX_H
#define OASES_MX_H

#include <stddef.h>
#include <stdint.h>

#include "oases.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of the scale tiles of an MX operand with `rows` rows and contraction
 * length K (0 for a negative argument). */
size_t oases_mx_scale_bytes(int rows, int K);

/* Quantises to an MX operand (codes + scales as above).
 * transpose = 0: x is [rows, K] (leading dimension ld elements) and row r of
 *                the operand is row r of x;
 * transpose = 1: x is [K, rows] (leading dimension ld) and the operand is its
 *                transpose, for products that contract over x's rows (the
 *                weight gradients dW = dY^T H contract over the batch rows).
 * Per block v of 32 consecutive operand elements along K (the last one
 * shorter when K % 32 != 0): X = 2^(floor(log2 max|v|) - 8), clamped to
 * [2^-127, 2^127], X = 1 for an all-zero block; codes E4M3(v / X), nearest
 * value with ties to the even code, magnitudes above 448 saturated to 448.
 * dtype: oases_dtype of x (OASES_F32 or OASES_BF16).
 * Errors: OASES_ERR_INVALID_ARG for negative sizes, a bad dtype, NULL or
 * misaligned pointers (q, scales 16-byte aligned; ldq a multiple of 16 and at
 * least K); rows == 0 or K == 0 does nothing. */
oases_status oases_mx_quantize(const void *x, int64_t ld, int rows, int K, int dtype,
                               int transpose, uint8_t *q, int64_t ldq, uint8_t *scales,
                               void *stream);

/* D[m, n] = sum over 32-blocks b of X_A[m, b] X_B[n, b] sum_{k in b} A[m, k] B[n, k]
 * for MX operands A ([M, K]: codes a, leading dimension lda, scales a_scales)
 * and B ([N, K]: b, ldb, b_scales), fp32 accumulation, then the epilogue of
 * oases_debug_gemm (0 Store, 1 Bias, 2 BiasGelu (+ C2 = gelu'), 3 BiasResid,
 * 4 Mul, 5 Accum (fp32 C += D)).  bias ([N]) and aux ([M, ld_aux]) are bf16;
 * C and C2 have type c_dtype (OASES_F32 or OASES_BF16; fp32 for Accum),
 * leading dimension ldc.  One CTA per 128 x 128 output tile, persistent.
 * Errors: OASES_ERR_INVALID_ARG for bad sizes, codes or NULL pointers;
 * OASES_ERR_UNSUPPORTED when the operands miss the alignment rules (lda, ldb
 * multiples of 16 and >= K; codes, scales, C, C2, bias, aux 16-byte aligned). */
oases_status oases_mx_gemm(int M, int N, int K, const uint8_t *a, int64_t lda,
                           const uint8_t *a_scales, const uint8_t *b, int64_t ldb,
                           const uint8_t *b_scales, int epilogue, void *C, int64_t ldc,
                           int c_dtype, void *C2, const void *bias, const void *aux,
                           int64_t ld_aux, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* OASES_MX_H */
