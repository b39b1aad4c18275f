/*
 * rmsnorm_matmul.h -- C ABI of the fused RMSNorm + matmul (GB300, sm_103a).
 *
 * The operation (matmul_rms_norm.wgsl, meganeura 0.2.0: the header comment,
 * C = RmsNorm(X, W_norm) x W_proj, and the entry point's row-scale prologue
 * and normalised A-tile load):
 *
 *     C[i, j] = sum over t of  X[i, t] * r[i] * W_norm[t] * W_proj[t, j]
 *     r[i]    = 1 / sqrt( (sum over t of X[i, t]^2) / K + eps )
 *
 * with X [M][K], W_norm [K], W_proj [K][N] and C [M][N], all row-major and
 * dense (row pitch = row length).  The page passes eps bit-cast in a u32;
 * here it is a float field.
 *
 * Arguments: device pointers (the caller owns every buffer; nothing is
 * allocated, kept or freed).  X, W_norm and W_proj are read and have the
 * element type `dtype` (dgrad_dtype of conv2d_grad_input.h); C is float32 and
 * overwritten.  `stream` may be NULL (the legacy default stream); the call
 * only enqueues work on it.
 *
 * Arithmetic: DGRAD_BF16 / DGRAD_F16 run on the tensor cores when the
 * tensor-core kernel applies (see rmsnorm_matmul_select_kernel): each
 * element X[i, t] * W_norm[t] is formed in float32 and rounded to the input
 * type for the tcgen05 product (exact products, float32 accumulation), the
 * row's sum of squares is accumulated in float32 from the same X elements as
 * they stream through, and r[i] scales row i of the float32 accumulator in
 * the epilogue -- X is read once.  DGRAD_F32, and 16-bit shapes the
 * tensor-core kernel does not take, run a CUDA-core kernel in float32
 * throughout.
 *
 * Errors (dgrad_status, conv2d_grad_input.h), checked on the host before any
 * work is enqueued, C untouched: DGRAD_ERR_INVALID_ARG for a NULL pointer or
 * params, an unknown dtype or a non-finite or negative eps;
 * DGRAD_ERR_SHAPE for m, n or k equal to 0; DGRAD_ERR_ALIGNMENT for a
 * pointer not aligned to its element size; DGRAD_ERR_UNSUPPORTED for a
 * matrix of more than 2^31 - 1 elements, or a forced kernel
 * (rmsnorm_matmul_set_kernel) that does not apply; DGRAD_ERR_CUDA when a
 * launch fails.  A device-side wait that runs out of time ends the kernel
 * early and raises this library's error flag, read (and cleared) by
 * rmsnorm_matmul_check_errors as DGRAD_ERR_TIMEOUT.
 */
#ifndef RMSNORM_MATMUL_H
#define RMSNORM_MATMUL_H

#include <stdint.h>

#include "conv2d_grad_input.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct rmsnorm_matmul_params {
    uint32_t m;  /* rows of X and C */
    uint32_t n;  /* columns of W_proj and C */
    uint32_t k;  /* columns of X, rows of W_proj, length of W_norm */
    float eps;   /* added to the mean square of each row of X */
} rmsnorm_matmul_params;

/* C = RmsNorm(X, W_norm) x W_proj as defined above. */
int rmsnorm_matmul(const void *x, const void *w_norm, const void *w_proj, float *c,
                   const rmsnorm_matmul_params *p, int dtype, struct CUstream_st *stream);

/* Which kernel rmsnorm_matmul runs for these arguments: DGRAD_KERNEL_TC or
 * DGRAD_KERNEL_SIMT, or a negative dgrad_status for invalid arguments.  The
 * tensor-core kernel takes DGRAD_BF16 / DGRAD_F16 with k a multiple of 8, n a
 * multiple of 64 and X, W_proj and C 16-byte aligned (its TMA tensor maps);
 * host logic only, no device access. */
int rmsnorm_matmul_select_kernel(const void *x, const void *w_norm, const void *w_proj,
                                 const float *c, const rmsnorm_matmul_params *p, int dtype);

/* Process-wide kernel choice for rmsnorm_matmul: DGRAD_KERNEL_AUTO (default),
 * DGRAD_KERNEL_TC or DGRAD_KERNEL_SIMT.  Returns the previous choice, or
 * DGRAD_ERR_INVALID_ARG for another value (the choice is then unchanged). */
int rmsnorm_matmul_set_kernel(int kernel);

/* Synchronises `stream`, then reports and clears the tensor-core kernel's
 * timeout flag (DGRAD_ERR_TIMEOUT) or a pending CUDA error (DGRAD_ERR_CUDA). */
int rmsnorm_matmul_check_errors(struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* RMSNORM_MATMUL_H */
