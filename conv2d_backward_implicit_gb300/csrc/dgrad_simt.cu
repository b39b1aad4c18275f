// dgrad_simt.cu -- direct CUDA-core dgrad, one thread per grad_in element.
//
// The fallback for shapes outside the tensor-core kernel's limits and a
// second, independent GPU path for cross-checks.  Each thread visits only the
// taps of its own sub-pixel phase: kh runs over th, th + s, ... with
// th = (ih + ph) mod s, so oh = (ih + ph - kh) / s is always exact (the
// divisibility test of the page's strided staging branch,
// conv2d_grad_input_gemm_coop.wgsl, taken out of the loop).  Products and
// sums in float32; bf16/fp16 inputs are widened exactly.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "conv2d_grad_input.h"
#include "dgrad_internal.h"

namespace dgrad {
namespace {

__device__ __forceinline__ float widen(float x) { return x; }
__device__ __forceinline__ float widen(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float widen(__half x) { return __half2float(x); }

template <typename T>
__global__ void __launch_bounds__(256) dgrad_simt_kernel(const T *__restrict__ g,
                                                         const T *__restrict__ w,
                                                         float *__restrict__ gi,
                                                         const SimtParams p) {
    const int64_t total = (int64_t)p.N * p.Ci * p.H * p.W;
    const int64_t plane_o = (int64_t)p.OH * p.OW;
    const int64_t step = (int64_t)gridDim.x * blockDim.x;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += step) {
        int64_t r = idx;
        const int iw = (int)(r % p.W); r /= p.W;
        const int ih = (int)(r % p.H); r /= p.H;
        const int ci = (int)(r % p.Ci); r /= p.Ci;
        const int n = (int)r;
        const int yh = ih + p.ph, yw = iw + p.pw;
        float acc = 0.f;
        for (int kh = yh % p.stride; kh < p.kH && kh <= yh; kh += p.stride) {
            const int oh = (yh - kh) / p.stride;
            if (oh >= p.OH) continue;
            for (int kw = yw % p.stride; kw < p.kW && kw <= yw; kw += p.stride) {
                const int ow = (yw - kw) / p.stride;
                if (ow >= p.OW) continue;
                const T *gp = g + (int64_t)n * p.Co * plane_o + (int64_t)oh * p.OW + ow;
                const T *wp = w + ((int64_t)ci * p.kH + kh) * p.kW + kw;
                const int64_t wstride = (int64_t)p.Ci * p.kH * p.kW;
                for (int co = 0; co < p.Co; ++co)
                    acc = fmaf(widen(gp[co * plane_o]), widen(wp[co * wstride]), acc);
            }
        }
        gi[idx] = acc;
    }
}

}  // namespace

int launch_simt(const Plan &plan, const void *grad_out, const void *weight, float *grad_in,
                void *stream) {
    NvtxRange range("conv2d_grad_input: dgrad (CUDA cores)");
    const SimtParams &p = plan.simt;
    const int64_t total = (int64_t)p.N * p.Ci * p.H * p.W;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    if (blocks > 65536) blocks = 65536;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (plan.dtype) {
    case DGRAD_F32:
        dgrad_simt_kernel<float><<<(int)blocks, threads, 0, st>>>(
            static_cast<const float *>(grad_out), static_cast<const float *>(weight), grad_in, p);
        break;
    case DGRAD_BF16:
        dgrad_simt_kernel<__nv_bfloat16><<<(int)blocks, threads, 0, st>>>(
            static_cast<const __nv_bfloat16 *>(grad_out), static_cast<const __nv_bfloat16 *>(weight),
            grad_in, p);
        break;
    default:
        dgrad_simt_kernel<__half><<<(int)blocks, threads, 0, st>>>(
            static_cast<const __half *>(grad_out), static_cast<const __half *>(weight), grad_in, p);
        break;
    }
    return (int)cudaGetLastError();
}

}  // namespace dgrad
