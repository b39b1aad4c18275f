// pack.cu -- the weight pre-pack kernel.
//
// The page's shader (conv2d_grad_input_gemm_coop.wgsl, weight staging of the
// A tiles) re-gathers A[ci, k] = weight[co, ci, kh, kw] with K ordered
// (co, kh, kw) for every output tile and every batch item.  Here that gather
// runs once per call and writes the exact shared-memory image the
// tensor-core kernel consumes, so the kernel moves it with plain bulk copies:
//
//   for each phase (rh, rw) with taps kh = s*j + th, kw = s*i + tw,
//     for each Ci tile mt, grad_out channel chunk cc, tap j, tap i:
//       m_tile rows (ci) of 128 bytes (kc consecutive co), 128-byte swizzled
//
// (stacked-phase mode: for each channel chunk cc and window tap t, st_n rows
// n = phase * Ci + ci of 128 bytes, zero where that phase has no such tap)
// i.e. K-major [Ci, K] operand tiles in the 128-byte swizzle layout of the
// tcgen05 shared-memory descriptors: within each group of 8 rows, the 16-byte
// chunk c of row r is stored at chunk position c ^ (r mod 8).  Rows ci >= Ci
// and channels co >= Co are zero.  For float32 input the values are rounded
// to TF32 (nearest, ties away from zero), the operand precision of kind::tf32.
#include <cuda_runtime.h>

#include "conv2d_grad_input.h"
#include "dgrad_internal.h"

namespace dgrad {
namespace {

__device__ __forceinline__ uint32_t to_tf32_rna(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

template <typename T>
__global__ void __launch_bounds__(256) pack_weight_kernel(const T *__restrict__ w,
                                                          T *__restrict__ out,
                                                          const __grid_constant__ PackParams k) {
    // Launched with programmatic stream serialization: let the next kernel
    // start its prologue, and wait for the previous kernel (which may still
    // read `out` or produce `w`) before touching global memory.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t stride_all = (int64_t)gridDim.x * blockDim.x;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < k.total_elems;
         idx += stride_all) {
        if (k.stacked) {
            // [chunk cc][tap t][row n][kc], rows 128-byte swizzled.
            const int E = k.elems16;
            int64_t r = idx;
            const int pos = (int)(r % k.kc); r /= k.kc;
            const int n = (int)(r % k.st_n); r /= k.st_n;
            const int taps = k.st_th * k.st_tw;
            const int t = (int)(r % taps);
            const int cc = (int)(r / taps);
            const int chunk = (pos / E) ^ (n & 7);
            const int co = cc * k.kc + chunk * E + pos % E;
            const int ph = n / k.Ci, ci = n - ph * k.Ci;
            T v = T(0);
            if (co < k.Co && ph < k.stride * k.stride) {
                const int j = k.qh[ph] - (k.st_dy0 + t / k.st_tw);
                const int i = k.qw[ph] - (k.st_dx0 + t % k.st_tw);
                if (j >= 0 && j < k.Jh[ph] && i >= 0 && i < k.Jw[ph]) {
                    const int kh = k.stride * j + k.th[ph], kw = k.stride * i + k.tw[ph];
                    v = w[(((int64_t)co * k.Ci + ci) * k.kH + kh) * k.kW + kw];
                }
            }
            if constexpr (sizeof(T) == 4) {
                out[idx] = __uint_as_float(to_tf32_rna(v));
            } else {
                out[idx] = v;
            }
            continue;
        }
        int ph = 0;
        while (ph + 1 < k.n_phases && idx >= k.elem_begin[ph + 1]) ++ph;
        int64_t r = idx - k.elem_begin[ph];
        const int E = k.elems16;                 // elements per 16-byte chunk
        const int row_elems = k.kc;              // elements per 128-byte row
        const int pos = (int)(r % row_elems);    // physical element slot within the row
        r /= row_elems;
        const int row = (int)(r % k.m_tile); r /= k.m_tile;
        const int i = (int)(r % k.Jw[ph]); r /= k.Jw[ph];
        const int j = (int)(r % k.Jh[ph]); r /= k.Jh[ph];
        const int cc = (int)(r % k.n_cchunks); r /= k.n_cchunks;
        const int mt = (int)r;
        const int chunk = (pos / E) ^ (row & 7);  // logical chunk stored at this slot
        const int co = cc * k.kc + chunk * E + pos % E;
        const int ci = mt * k.m_tile + row;
        const int kh = k.stride * j + k.th[ph];
        const int kw = k.stride * i + k.tw[ph];
        T v;
        if (co < k.Co && ci < k.Ci) {
            v = w[(((int64_t)co * k.Ci + ci) * k.kH + kh) * k.kW + kw];
        } else {
            v = T(0);
        }
        if constexpr (sizeof(T) == 4) {
            out[idx] = __uint_as_float(to_tf32_rna(v));
        } else {
            out[idx] = v;
        }
    }
}

// wt[ci][co][kh][kw] = w[co][ci][kH-1-kh][kW-1-kw]: the weights of a layer
// seen from the other side (channel axes swapped, kernel flipped).
template <typename T>
__global__ void __launch_bounds__(256) flip_transpose_kernel(const T *__restrict__ w, T *__restrict__ wt,
                                                             int Co, int Ci, int kH, int kW, int64_t total) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = idx;  // idx enumerates wt = [Ci][Co][kH][kW]
        const int kw = (int)(r % kW); r /= kW;
        const int kh = (int)(r % kH); r /= kH;
        const int co = (int)(r % Co);
        const int ci = (int)(r / Co);
        wt[idx] = w[(((int64_t)co * Ci + ci) * kH + (kH - 1 - kh)) * kW + (kW - 1 - kw)];
    }
}

// X''[n][(pr, pc, ci)][a][b] of a FwdSplit, one element per thread (writes
// coalesced along b; the reads stride by s along x's rows).
template <typename T>
__global__ void __launch_bounds__(256) space_to_depth_kernel(const T *__restrict__ x, T *__restrict__ xs,
                                                             const __grid_constant__ FwdSplit f,
                                                             int64_t total) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = idx;
        const int b = (int)(r % f.Wx); r /= f.Wx;
        const int a = (int)(r % f.Hx); r /= f.Hx;
        const int ch = (int)(r % ((int64_t)f.nr * f.nc * f.Ci));
        const int n = (int)(r / ((int64_t)f.nr * f.nc * f.Ci));
        const int ci = ch % f.Ci, pc = (ch / f.Ci) % f.nc, pr = ch / (f.Ci * f.nc);
        const int ih = f.s * (a + f.jmin) + f.R[pr], iw = f.s * (b + f.imin) + f.C[pc];
        xs[idx] = (ih >= 0 && ih < f.H && iw >= 0 && iw < f.W)
                      ? x[(((int64_t)n * f.Ci + ci) * f.H + ih) * f.W + iw]
                      : T(0);
    }
}

// W''[co][(pr, pc, ci)][j][i] of a FwdSplit.
template <typename T>
__global__ void __launch_bounds__(256) split_weights_kernel(const T *__restrict__ w, T *__restrict__ ws,
                                                            const __grid_constant__ FwdSplit f,
                                                            int64_t total) {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        int64_t r = idx;
        const int i = (int)(r % f.KW); r /= f.KW;
        const int j = (int)(r % f.KH); r /= f.KH;
        const int ch = (int)(r % ((int64_t)f.nr * f.nc * f.Ci));
        const int co = (int)(r / ((int64_t)f.nr * f.nc * f.Ci));
        const int ci = ch % f.Ci, pc = (ch / f.Ci) % f.nc, pr = ch / (f.Ci * f.nc);
        const int kh = f.s * (j + f.jmin) + f.R[pr] + f.ph, kw = f.s * (i + f.imin) + f.C[pc] + f.pw;
        ws[idx] = (kh >= 0 && kh < f.kH && kw >= 0 && kw < f.kW)
                      ? w[(((int64_t)co * f.Ci + ci) * f.kH + kh) * f.kW + kw]
                      : T(0);
    }
}

// One launch of an elementwise kernel over `total` elements with programmatic
// stream serialization (the next kernel's prologue may overlap this one).
template <typename K, typename... A>
int launch_elementwise(K kern, int64_t total, void *stream, A... args) {
    if (total == 0) return (int)cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 8192) blocks = 8192;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, args..., total);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

}  // namespace

int launch_space_to_depth(const FwdSplit &f, const void *x, void *xs, int esize, void *stream) {
    NvtxRange range("conv2d_forward: space-to-depth of x");
    const int64_t total = (int64_t)f.N * f.nr * f.nc * f.Ci * f.Hx * f.Wx;
    if (esize == 4)
        return launch_elementwise(space_to_depth_kernel<float>, total, stream, static_cast<const float *>(x),
                                  static_cast<float *>(xs), f);
    return launch_elementwise(space_to_depth_kernel<unsigned short>, total, stream,
                              static_cast<const unsigned short *>(x), static_cast<unsigned short *>(xs), f);
}

int launch_split_weights(const FwdSplit &f, const void *w, void *ws, int esize, void *stream) {
    NvtxRange range("conv2d_forward: split weights");
    const int64_t total = (int64_t)f.Co * f.nr * f.nc * f.Ci * f.KH * f.KW;
    if (esize == 4)
        return launch_elementwise(split_weights_kernel<float>, total, stream, static_cast<const float *>(w),
                                  static_cast<float *>(ws), f);
    return launch_elementwise(split_weights_kernel<unsigned short>, total, stream,
                              static_cast<const unsigned short *>(w), static_cast<unsigned short *>(ws), f);
}

int launch_flip_transpose(const void *w, void *wt, int Co, int Ci, int kH, int kW, int esize,
                          void *stream) {
    NvtxRange range("conv2d_forward: flip weights");
    const int64_t total = (int64_t)Co * Ci * kH * kW;
    if (total == 0) return (int)cudaSuccess;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = static_cast<cudaStream_t>(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (esize == 4)
        e = cudaLaunchKernelEx(&cfg, flip_transpose_kernel<float>, static_cast<const float *>(w),
                               static_cast<float *>(wt), Co, Ci, kH, kW, total);
    else
        e = cudaLaunchKernelEx(&cfg, flip_transpose_kernel<unsigned short>, static_cast<const unsigned short *>(w),
                               static_cast<unsigned short *>(wt), Co, Ci, kH, kW, total);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

int launch_pack(const Plan &plan, const void *weight, void *packed, void *stream) {
    NvtxRange range("conv2d_grad_input: pack weights");
    const PackParams &k = plan.pack;
    if (k.total_elems == 0) return (int)cudaSuccess;
    const int threads = 256;
    int64_t blocks = (k.total_elems + threads - 1) / threads;
    if (blocks > 4096) blocks = 4096;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(threads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    if (plan.esize == 4) {
        e = cudaLaunchKernelEx(&cfg, pack_weight_kernel<float>, static_cast<const float *>(weight),
                               static_cast<float *>(packed), k);
    } else {
        e = cudaLaunchKernelEx(&cfg, pack_weight_kernel<unsigned short>,
                               static_cast<const unsigned short *>(weight),
                               static_cast<unsigned short *>(packed), k);
    }
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

}  // namespace dgrad
