/*
 * mha_grad_v.h -- C ABI of the attention gradient with respect to V (GB300, sm_103a).
 *
 * The operation (mha_grad_v.wgsl, meganeura 0.2.0: Params struct and entry
 * point), with Q and dO [q_seq][num_heads][head_dim], K [kv][num_kv_heads]
 * [head_dim], LSE [q_seq][num_heads][2] and dV [kv][num_kv_heads][head_dim],
 * all row-major and dense:
 *
 *   kv     = kv_seq, or q_seq when kv_seq == 0 (causal self-attention);
 *   for key position t, KV head g and the heads h = g * (num_heads /
 *   num_kv_heads) + r of its group,
 *   dV[t][g][:] = sum over pos in [start, end) and r of  P * dO[pos][h][:],
 *   start = t if causal else 0,  end = min(q_seq, t + window_size) if
 *   window_size > 0 else q_seq,
 *   P = exp(min(s - LSE[pos][h][0], 0) - LSE[pos][h][1]),
 *   s = (Q[pos][h][:] . K[t][g][:]) / sqrt(head_dim).
 *
 * LSE holds the forward pass's statistics of each query and head: the maximum
 * score and the log of the sum of exp(score - maximum) over the keys it
 * attended.  The page binds V and the forward output O as well; the dV
 * computation reads neither, so they are not arguments here.  The page packs
 * num_heads and num_kv_heads into one u32; here they are separate fields.
 *
 * Arguments: device pointers owned by the caller (nothing allocated or kept).
 * Q, K and dO have the element type `dtype` (dgrad_dtype of conv2d_grad_input.h);
 * LSE and dV are float32; dV is overwritten.  `stream` may be NULL.
 *
 * Arithmetic: the CUDA-core kernel (every dtype and shape) computes in
 * float32: scores, exponentials and the sums.  The tensor-core kernel
 * (bf16 / fp16, head_dim 64, an even num_heads, 16-byte aligned pointers; see
 * mha_grad_v_select_kernel) forms the scores with tcgen05 (exact products,
 * float32 sums), P in float32, rounds P to the input type for the second
 * product (with dO) and sums in float32.
 *
 * Errors (dgrad_status), checked on the host before any work, dV untouched:
 * DGRAD_ERR_INVALID_ARG for a NULL pointer or params, or an unknown dtype;
 * DGRAD_ERR_SHAPE for q_seq, num_heads, num_kv_heads or head_dim equal to 0, or
 * num_heads not a multiple of num_kv_heads; DGRAD_ERR_ALIGNMENT for a pointer
 * not aligned to its element size; DGRAD_ERR_UNSUPPORTED for a tensor of more
 * than 2^31 - 1 elements, head_dim above 256, or a forced kernel
 * (mha_grad_v_set_kernel) that does not apply; DGRAD_ERR_CUDA when a launch
 * fails.  A device-side wait that runs out of time ends the tensor-core
 * kernel early and raises the flag mha_grad_v_check_errors reports as
 * DGRAD_ERR_TIMEOUT.
 */
#ifndef MHA_GRAD_V_H
#define MHA_GRAD_V_H

#include <stdint.h>

#include "conv2d_grad_input.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct mha_grad_v_params {
    uint32_t q_seq;        /* query positions */
    uint32_t kv_seq;       /* key/value positions; 0: causal self-attention with kv = q_seq */
    uint32_t num_heads;    /* query heads */
    uint32_t num_kv_heads; /* key/value heads; num_heads is a multiple of it */
    uint32_t head_dim;     /* elements per head */
    uint32_t window_size;  /* > 0: query pos reaches key t only when pos < t + window_size */
} mha_grad_v_params;

/* dV as defined above. */
int mha_grad_v(const void *q, const void *k, const void *d_out, const float *lse, float *dv,
               const mha_grad_v_params *p, int dtype, struct CUstream_st *stream);

/* Which kernel mha_grad_v runs for these arguments: DGRAD_KERNEL_TC or
 * DGRAD_KERNEL_SIMT, or a negative dgrad_status for invalid arguments.  The
 * tensor-core kernel takes DGRAD_BF16 / DGRAD_F16 with head_dim 64, an even
 * num_heads (its statistics view needs rows of a multiple of 16 bytes) and Q,
 * K, dO, LSE and dV 16-byte aligned; host logic only. */
int mha_grad_v_select_kernel(const void *q, const void *k, const void *d_out, const float *lse,
                             const float *dv, const mha_grad_v_params *p, int dtype);

/* Process-wide kernel choice for mha_grad_v: DGRAD_KERNEL_AUTO (default),
 * DGRAD_KERNEL_TC or DGRAD_KERNEL_SIMT.  Returns the previous choice, or
 * DGRAD_ERR_INVALID_ARG for another value. */
int mha_grad_v_set_kernel(int kernel);

/* Synchronises `stream`, then reports and clears the tensor-core kernel's
 * timeout flag (DGRAD_ERR_TIMEOUT) or a pending CUDA error (DGRAD_ERR_CUDA). */
int mha_grad_v_check_errors(struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* MHA_GRAD_V_H */
