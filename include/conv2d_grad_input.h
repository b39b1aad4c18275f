/*
 * conv2d_grad_input.h -- C ABI of the GB300 (sm_103a) conv2d input-gradient library.
 *
 * What it computes (the page "conv2d_grad_input_gemm_coop.wgsl", meganeura
 * 0.2.0: header comment, Params struct and strided staging branch; the
 * semantics are those of the exact adjoint of the forward convolution):
 *
 *   grad_in[n,ci,ih,iw] = sum over co < Co, kh < kH, kw < kW of
 *                         grad_out[n,co,oh,ow] * weight[co,ci,kh,kw]
 *   over the taps with ih + padding_h - kh = stride*oh, iw + padding_w - kw =
 *   stride*ow, 0 <= oh < out_h, 0 <= ow < out_w.
 *
 * That is, per batch item, C[Ci, H*W] = A[Ci, K] x B[K, H*W] with
 * K = Co*kH*kW, A the transposed weights and B the im2col matrix of
 * grad_out.  It is the gradient of out[n,co,oh,ow] = sum x[n,ci,oh*s-ph+kh,
 * ow*s-pw+kw] * w[co,ci,kh,kw] (x zero outside the image) with respect to x.
 * Pixels that no tap reaches get 0.
 *
 * Layouts (all dense, row-major, no padding between rows):
 *   grad_out  [batch, out_channels, out_h, out_w]        dtype
 *   weight    [out_channels, in_channels, kernel_h, kernel_w] dtype
 *   grad_in   [batch, in_channels, in_h, in_w]           float32, overwritten
 * dtype is DGRAD_BF16 or DGRAD_F16 (tensor-core products exact, float32
 * accumulate) or DGRAD_F32 (operands rounded to TF32, float32 accumulate).
 *
 * Ownership: the caller owns every buffer.  The library keeps no pointer
 * after a call returns; the work it enqueued reads and writes them
 * asynchronously on `stream`, so they must stay alive until that work is done.
 *
 * Streams and devices: `stream` is a cudaStream_t (NULL = the legacy default
 * stream) of the current device, the kernels run on the current device, and
 * every buffer must be memory of that device (the library does not check
 * which device a pointer belongs to; the Python binding does).  Every entry point that takes one is asynchronous with
 * respect to the host, except conv2d_grad_input_check_errors.
 *
 * Errors: every entry point returns a dgrad_status (0 = success) and never
 * aborts or throws.  Arguments are checked on the host before anything is
 * enqueued; on an argument error nothing is enqueued and grad_in is left
 * untouched.  DGRAD_ERR_CUDA means a CUDA call failed (the CUDA error is
 * cleared and not left for the caller).  A device-side wait that exceeds its
 * time limit makes the kernel stop early, set a device flag and return; the
 * flag is reported as DGRAD_ERR_TIMEOUT by conv2d_grad_input_check_errors.
 */
#ifndef CONV2D_GRAD_INPUT_H
#define CONV2D_GRAD_INPUT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* the same opaque type cudaStream_t points to */

/* The twelve fields and their order follow the Params struct of
 * conv2d_grad_input_gemm_coop.wgsl.  One stride serves both axes; the two
 * paddings are separate.  out_h/out_w must equal
 * floor((in + 2*padding - kernel) / stride) + 1 (checked). */
typedef struct conv2d_grad_input_params {
    uint32_t batch;
    uint32_t in_channels;
    uint32_t in_h;
    uint32_t in_w;
    uint32_t out_channels;
    uint32_t kernel_h;
    uint32_t kernel_w;
    uint32_t stride;
    uint32_t padding_h;
    uint32_t out_h;
    uint32_t out_w;
    uint32_t padding_w;
} conv2d_grad_input_params;

typedef enum dgrad_dtype {
    DGRAD_F32 = 0,  /* float32 in, TF32 tensor-core products */
    DGRAD_BF16 = 1, /* bfloat16 in */
    DGRAD_F16 = 2   /* float16 in */
} dgrad_dtype;

typedef enum dgrad_status {
    DGRAD_OK = 0,
    DGRAD_ERR_INVALID_ARG = 1, /* NULL pointer, unknown dtype or kernel id */
    DGRAD_ERR_SHAPE = 2,       /* zero or inconsistent sizes, out_h/out_w off the formula */
    DGRAD_ERR_ALIGNMENT = 3,   /* a pointer is not aligned to its element size */
    DGRAD_ERR_UNSUPPORTED = 4, /* a size beyond the library's limits (e.g. > 2^31-1 per index) */
    DGRAD_ERR_CUDA = 5,        /* a CUDA runtime call failed */
    DGRAD_ERR_TIMEOUT = 6,     /* a device-side wait ran out of time (kernel returned early) */
    DGRAD_ERR_WORKSPACE = 7    /* the packed-weight buffer is too small: the one passed in, or the
                                  fixed 8 MiB internal array of conv2d_grad_input_noalloc */
} dgrad_status;

typedef enum dgrad_kernel {
    DGRAD_KERNEL_AUTO = 0, /* tensor-core kernel where it applies, else the CUDA-core kernel */
    DGRAD_KERNEL_TC = 1,   /* tcgen05 implicit GEMM (weights pre-packed, or packed by the kernel itself) */
    DGRAD_KERNEL_SIMT = 2, /* direct CUDA-core kernel, one thread per grad_in element */
    /* tcgen05 implicit GEMM with the output positions on the MMA M side and
     * the kW taps of a kernel row side by side on N, for stride 1, bf16 or
     * fp16, in_channels and out_channels <= 64, kernel_w <= 3, in_w and
     * out_w <= 56 with 16-byte grad_out rows; other shapes run as
     * DGRAD_KERNEL_TC.  Weights pre-packed by conv2d_grad_input_pack_weight.  Opt-in:
     * its epilogue writes grad_in with plain stores from the epilogue warps. */
    DGRAD_KERNEL_TC_POSM = 3
} dgrad_kernel;

/* The whole operation: packs the weights into a stream-ordered temporary
 * buffer (cudaMallocAsync / cudaFreeAsync on `stream`) and runs the dgrad
 * kernel; when conv2d_grad_input_workspace_size is 0 the kernel reads the
 * weights as they are (one launch, no allocation).  grad_out and weight are
 * read, grad_in is overwritten. */
int conv2d_grad_input(const void *grad_out, const void *weight, float *grad_in,
                      const conv2d_grad_input_params *p, int dtype, struct CUstream_st *stream);

/* Bytes of the packed-weight buffer that conv2d_grad_input_pack_weight
 * writes and conv2d_grad_input_prepacked reads for these params and dtype,
 * for the kernel that the current selection would run.  0 when the
 * selected kernel reads the weights unpacked -- the CUDA-core kernel, and the
 * tensor-core kernel on 16-bit stride-1 layers whose packed weights stay
 * resident in shared memory (its epilogue warps pack them there while the
 * first grad_out tile loads) -- or when the arguments are invalid. */
size_t conv2d_grad_input_workspace_size(const conv2d_grad_input_params *p, int dtype);

/* The weight pre-pack: transposes weight [Co,Ci,kH,kW] into per-phase,
 * K-major [Ci, Co*taps] tiles (for stride s > 1 each of the s*s sub-pixel
 * phases keeps only its own taps), zero-padded to whole tiles, and for
 * DGRAD_F32 rounds to TF32 (nearest, ties away from zero).  `packed` is a
 * device buffer of at least packed_bytes >= conv2d_grad_input_workspace_size
 * bytes, 16-byte aligned.  A pack depends only on weight, p and dtype, so it
 * can be reused across calls with the same weights.  When
 * conv2d_grad_input_workspace_size is 0 there is nothing to pack: the call
 * returns DGRAD_OK and launches nothing. */
int conv2d_grad_input_pack_weight(const void *weight, void *packed, size_t packed_bytes,
                                  const conv2d_grad_input_params *p, int dtype,
                                  struct CUstream_st *stream);

/* The dgrad kernel alone, reading weights packed by
 * conv2d_grad_input_pack_weight with the same p and dtype (and the same
 * kernel selection).  When conv2d_grad_input_workspace_size is 0 (the
 * CUDA-core kernel, or a kernel that packs in shared memory), `packed` must be
 * the original weight tensor instead, aligned to its element size. */
int conv2d_grad_input_prepacked(const void *grad_out, const void *packed, float *grad_in,
                                const conv2d_grad_input_params *p, int dtype,
                                struct CUstream_st *stream);

/* Synchronizes `stream`, then reports and clears the device-side timeout
 * flag of this device (DGRAD_ERR_TIMEOUT) or a pending CUDA error
 * (DGRAD_ERR_CUDA).  Returns DGRAD_OK when neither occurred. */
int conv2d_grad_input_check_errors(struct CUstream_st *stream);

/* A static, human-readable name for a dgrad_status value. */
const char *conv2d_grad_input_status_string(int status);

/* Which kernel a call with these arguments runs: DGRAD_KERNEL_TC,
 * DGRAD_KERNEL_TC_POSM or DGRAD_KERNEL_SIMT, or a negative dgrad_status for
 * invalid arguments. */
int conv2d_grad_input_select_kernel(const conv2d_grad_input_params *p, int dtype);

/* Process-wide kernel choice (DGRAD_KERNEL_AUTO by default).  Forcing
 * DGRAD_KERNEL_TC for a shape the tensor-core kernel cannot run makes calls
 * return DGRAD_ERR_UNSUPPORTED.  Returns the previous choice, or
 * -DGRAD_ERR_INVALID_ARG for an unknown id. */
int conv2d_grad_input_set_kernel(int kernel);

/* Device-wait time limit in nanoseconds for later launches (default
 * 2,000,000,000 = 2 s; 0 restores the default).  Returns the previous value. */
uint64_t conv2d_grad_input_set_wait_limit_ns(uint64_t ns);

/* Failure-injection switch for tests of the timeout path (0 = off, the
 * default).  DGRAD_DEBUG_SKIP_ARRIVE makes the tensor-core kernel's first
 * gather warp withhold its first "stage full" signal, so the MMA warp's wait
 * runs out of time; the kernel then returns early and
 * conv2d_grad_input_check_errors reports DGRAD_ERR_TIMEOUT.  grad_in is left
 * partly written.  Returns the previous value. */
#define DGRAD_DEBUG_SKIP_ARRIVE 1
int conv2d_grad_input_set_debug(int flags);

/* The forward convolution of the same layer:
 *
 *   out[n,co,oh,ow] = sum over ci < Ci, kh < kH, kw < kW of
 *                     x[n,ci,stride*oh-padding_h+kh, stride*ow-padding_w+kw] * weight[co,ci,kh,kw]
 *
 * (x zero outside the image) -- the convolution whose input gradient
 * conv2d_grad_input computes (the page's header comment defines the
 * gradient as its adjoint).  `p` describes the layer exactly as for
 * conv2d_grad_input: x is [batch, in_channels, in_h, in_w] of dtype, weight
 * [out_channels, in_channels, kernel_h, kernel_w] of dtype, out [batch,
 * out_channels, out_h, out_w] float32, overwritten.
 *  - Stride 1: the input gradient of a layer with the roles of the channel
 *    axes swapped, the kernel flipped and padding kernel - 1 - padding; the
 *    call flips and transposes the weights into a stream-ordered temporary
 *    buffer and runs the same kernels.  A padding above kernel - 1 returns
 *    DGRAD_ERR_UNSUPPORTED.
 *  - Stride s from 2 to 8: one stride-1 correlation without padding of a
 *    space-to-depth copy of x (one channel group per residue r of kh -
 *    padding_h and c of kw - padding_w modulo s that a tap reaches:
 *    [batch][(r, c, ci)][out_h + KH - 1][out_w + KW - 1], KH = floor((kH - 1
 *    - padding_h) / s) - floor(-padding_h / s) + 1) with the weights
 *    rearranged to match ([out_channels][(r, c, ci)][KH][KW], zero where a
 *    residue has no tap); both go to one stream-ordered temporary buffer and
 *    the stride-1 path runs on them.  Stride above 8 returns
 *    DGRAD_ERR_UNSUPPORTED.
 * Nothing is enqueued on an error; other argument errors as for
 * conv2d_grad_input. */
int conv2d_forward(const void *x, const void *weight, float *out, const conv2d_grad_input_params *p,
                   int dtype, struct CUstream_st *stream);

/* conv2d_grad_input without any device allocation.  The pages have no
 * counterpart to this entry point; it exists for callers that cannot
 * allocate device memory where they need the gradient -- code recorded into
 * a CUDA graph whose capture mode forbids allocation calls, runtimes whose
 * own memory arena owns the device and bans cudaMalloc/cudaMallocAsync on
 * their execution path, and latency-critical loops that cannot afford an
 * allocation's synchronisation.  Same arguments, semantics and results as
 * conv2d_grad_input, but the packed weights live in a fixed 8 MiB device
 * array inside the library instead of a temporary allocation:
 *  - the 8 MiB are device memory of the library's module: they are
 *    committed on a device when the module is loaded there -- under CUDA's
 *    lazy module loading (the default) at the first conv2d_grad_input_noalloc
 *    call on that device, whose address lookup loads it -- and stay until the
 *    process exits;
 *  - a problem whose packed weights exceed 8 MiB
 *    (conv2d_grad_input_workspace_size > 8388608) is rejected with
 *    DGRAD_ERR_WORKSPACE before anything is enqueued;
 *  - all calls share the array: calls whose GPU work can overlap (unordered
 *    streams, concurrent host threads) race on it and must be ordered by
 *    the caller; nothing from an earlier call needs clearing, since each
 *    call rewrites every byte its kernel reads;
 *  - the first call on a device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture.
 * Calls no cudaMalloc, cudaFree or other allocating routine. */
int conv2d_grad_input_noalloc(const void *grad_out, const void *weight, float *grad_in,
                              const conv2d_grad_input_params *p, int dtype,
                              struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* CONV2D_GRAD_INPUT_H */
