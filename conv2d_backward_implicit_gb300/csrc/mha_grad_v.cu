// mha_grad_v.cu -- the attention gradient with respect to V (mha_grad_v.wgsl,
// meganeura 0.2.0: Params struct and entry point), declared in
// include/mha_grad_v.h.
//
// CUDA-core kernel (every dtype, any head_dim up to 256): one block per 32 key
// positions of one KV head.  The block keeps its K rows in shared memory and
// walks the query positions that can reach them (from t0 when causal, up to
// the window's end) 32 at a time, for each head of the group: the 32 x 32
// scores from shared-memory Q and K rows, P from the forward statistics with
// the page's clamp and mask, then dV += P^T dO with each thread owning one key
// row and every 8th element of it.  Float32 throughout.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdint>

#include "mha_grad_v.h"
#include "nvtx_range.h"

namespace mhadv {

__device__ unsigned int g_mha_error_word = 0;

namespace {

constexpr int kT = 32, kP = 32;  // key rows per block, query rows per step
constexpr int kMaxHd = 256;

template <typename T>
__device__ __forceinline__ float to_f(T v) {
    if constexpr (sizeof(T) == 4) {
        return v;
    } else {
        return (float)v;
    }
}

struct SimtArgs {
    int q_seq, kv, nh, nkv, hd, window, causal;
    float scale;
};

template <typename T>
__global__ void __launch_bounds__(256) mha_grad_v_simt_kernel(const T *__restrict__ q, const T *__restrict__ k,
                                                              const T *__restrict__ d_out,
                                                              const float *__restrict__ lse, float *__restrict__ dv,
                                                              const SimtArgs a) {
    extern __shared__ float sm[];
    const int hd = a.hd, hdp = hd + 1;  // padded rows
    float *k_s = sm;                     // [kT][hdp]
    float *q_s = k_s + kT * hdp;         // [kP][hdp]
    float *o_s = q_s + kP * hdp;         // [kP][hdp] dO rows
    float *p_s = o_s + kP * hdp;         // [kT][kP + 1]
    float *st_s = p_s + kT * (kP + 1);   // [kP][2]
    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * kT, g = blockIdx.y;
    const int hpk = a.nh / a.nkv;
    const int64_t q_dim = (int64_t)a.nh * hd, kv_dim = (int64_t)a.nkv * hd;
    for (int e = tid; e < kT * hd; e += 256) {
        const int tr = e / hd, d = e - tr * hd, t = t0 + tr;
        k_s[tr * hdp + d] = t < a.kv ? to_f(k[(int64_t)t * kv_dim + (int64_t)g * hd + d]) : 0.f;
    }
    // This thread's outputs: key row tr, elements d = dl + 8 j.
    const int tr = tid >> 3, dl = tid & 7;
    const int t = t0 + tr;
    const int nd = (hd - dl + 7) / 8;
    float acc[kMaxHd / 8];
#pragma unroll
    for (int j = 0; j < kMaxHd / 8; ++j) acc[j] = 0.f;
    // Query positions that reach some key of this block.
    const int t_last = (t0 + kT - 1 < a.kv ? t0 + kT - 1 : a.kv - 1);
    const int lo = a.causal ? t0 : 0;
    int hi = a.q_seq;
    if (a.window > 0 && t_last + a.window < hi) hi = t_last + a.window;
    for (int p0 = lo; p0 < hi; p0 += kP)
        for (int r = 0; r < hpk; ++r) {
            const int h = g * hpk + r;
            __syncthreads();  // previous step's readers are done
            for (int e = tid; e < kP * hd; e += 256) {
                const int pr = e / hd, d = e - pr * hd, pos = p0 + pr;
                const bool ok = pos < a.q_seq;
                const int64_t off = (int64_t)pos * q_dim + (int64_t)h * hd + d;
                q_s[pr * hdp + d] = ok ? to_f(q[off]) : 0.f;
                o_s[pr * hdp + d] = ok ? to_f(d_out[off]) : 0.f;
            }
            if (tid < 2 * kP) {
                const int pr = tid >> 1, pos = p0 + pr;
                st_s[tid] = pos < a.q_seq ? lse[((int64_t)pos * a.nh + h) * 2 + (tid & 1)] : 0.f;
            }
            __syncthreads();
            // Scores and P: thread -> key row tid / 8, query rows (tid % 8) + 8 i.
            {
                const int kr = tid >> 3, tk = t0 + kr;
                const int start = a.causal ? tk : 0;
                int end = a.q_seq;
                if (a.window > 0 && tk + a.window < end) end = tk + a.window;
#pragma unroll
                for (int i = 0; i < kP / 8; ++i) {
                    const int pr = (tid & 7) + 8 * i, pos = p0 + pr;
                    float s = 0.f;
                    for (int d = 0; d < hd; ++d) s = fmaf(k_s[kr * hdp + d], q_s[pr * hdp + d], s);
                    float p = 0.f;
                    if (tk < a.kv && pos >= start && pos < end) {
                        const float e = fminf(s * a.scale - st_s[2 * pr], 0.f);
                        p = expf(e - st_s[2 * pr + 1]);
                    }
                    p_s[kr * (kP + 1) + pr] = p;
                }
            }
            __syncthreads();
            // dV rows: acc[j] (element dl + 8 j of key row tr) += sum over pr of P * dO.
            for (int pr = 0; pr < kP; ++pr) {
                const float p = p_s[tr * (kP + 1) + pr];
#pragma unroll
                for (int j = 0; j < kMaxHd / 8; ++j)
                    if (j < nd) acc[j] = fmaf(p, o_s[pr * hdp + dl + 8 * j], acc[j]);
            }
        }
    if (t < a.kv) {
#pragma unroll
        for (int j = 0; j < kMaxHd / 8; ++j)
            if (j < nd) dv[(int64_t)t * kv_dim + (int64_t)g * hd + dl + 8 * j] = acc[j];
    }
}

std::atomic<int> g_kernel_choice{DGRAD_KERNEL_AUTO};

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) & (a - 1)) == 0; }

int validate(const void *q, const void *k, const void *go, const float *lse, const float *dv,
             const mha_grad_v_params *p, int dtype) {
    if (!q || !k || !go || !lse || !dv || !p) return DGRAD_ERR_INVALID_ARG;
    if (dtype != DGRAD_F32 && dtype != DGRAD_BF16 && dtype != DGRAD_F16) return DGRAD_ERR_INVALID_ARG;
    if (p->q_seq == 0 || p->num_heads == 0 || p->num_kv_heads == 0 || p->head_dim == 0 ||
        p->num_heads % p->num_kv_heads != 0)
        return DGRAD_ERR_SHAPE;
    const int64_t kv = p->kv_seq == 0 ? p->q_seq : p->kv_seq, lim = INT32_MAX;
    if ((int64_t)p->q_seq * p->num_heads * p->head_dim > lim || kv * p->num_kv_heads * p->head_dim > lim ||
        p->head_dim > (uint32_t)kMaxHd || (kv + kT - 1) / kT > lim || p->num_kv_heads > 65535u)
        return DGRAD_ERR_UNSUPPORTED;
    const uintptr_t e = dtype == DGRAD_F32 ? 4 : 2;
    if (!aligned(q, e) || !aligned(k, e) || !aligned(go, e) || !aligned(lse, 4) || !aligned(dv, 4))
        return DGRAD_ERR_ALIGNMENT;
    return DGRAD_OK;
}

bool tc_applies(const void *q, const void *k, const void *go, const float *lse, const float *dv,
                const mha_grad_v_params *p, int dtype);

int select(const void *q, const void *k, const void *go, const float *lse, const float *dv,
           const mha_grad_v_params *p, int dtype) {
    const int v = validate(q, k, go, lse, dv, p, dtype);
    if (v != DGRAD_OK) return -v;
    const int choice = g_kernel_choice.load();
    const bool tc = tc_applies(q, k, go, lse, dv, p, dtype);
    if (choice == DGRAD_KERNEL_SIMT) return DGRAD_KERNEL_SIMT;
    if (choice == DGRAD_KERNEL_TC) return tc ? DGRAD_KERNEL_TC : -DGRAD_ERR_UNSUPPORTED;
    return tc ? DGRAD_KERNEL_TC : DGRAD_KERNEL_SIMT;
}

template <typename T>
int launch_simt(const void *q, const void *k, const void *go, const float *lse, float *dv,
                const mha_grad_v_params *p, cudaStream_t st) {
    SimtArgs a;
    a.q_seq = (int)p->q_seq;
    a.causal = p->kv_seq == 0;
    a.kv = a.causal ? a.q_seq : (int)p->kv_seq;
    a.nh = (int)p->num_heads;
    a.nkv = (int)p->num_kv_heads;
    a.hd = (int)p->head_dim;
    a.window = (int)p->window_size;
    a.scale = 1.0f / sqrtf((float)a.hd);
    const size_t smem = sizeof(float) * ((size_t)(kT + 2 * kP) * (a.hd + 1) + kT * (kP + 1) + 2 * kP);
    auto kern = mha_grad_v_simt_kernel<T>;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return DGRAD_ERR_CUDA;
    const dim3 grid((a.kv + kT - 1) / kT, a.nkv);
    kern<<<grid, 256, smem, st>>>(static_cast<const T *>(q), static_cast<const T *>(k),
                                  static_cast<const T *>(go), lse, dv, a);
    return cudaGetLastError() == cudaSuccess ? DGRAD_OK : DGRAD_ERR_CUDA;
}

int launch_tc(const void *q, const void *k, const void *go, const float *lse, float *dv, const mha_grad_v_params *p,
              int dtype, cudaStream_t st);

}  // namespace
}  // namespace mhadv

#include "mha_grad_v_tc.cuh"

extern "C" {

int mha_grad_v(const void *q, const void *k, const void *d_out, const float *lse, float *dv,
               const mha_grad_v_params *p, int dtype, struct CUstream_st *stream) {
    using namespace mhadv;
    dgrad::NvtxRange range("mha_grad_v");
    const int kern = select(q, k, d_out, lse, dv, p, dtype);
    if (kern < 0) return -kern;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (kern == DGRAD_KERNEL_TC) return launch_tc(q, k, d_out, lse, dv, p, dtype, st);
    if (dtype == DGRAD_F32) return launch_simt<float>(q, k, d_out, lse, dv, p, st);
    if (dtype == DGRAD_BF16) return launch_simt<__nv_bfloat16>(q, k, d_out, lse, dv, p, st);
    return launch_simt<__half>(q, k, d_out, lse, dv, p, st);
}

int mha_grad_v_select_kernel(const void *q, const void *k, const void *d_out, const float *lse, const float *dv,
                             const mha_grad_v_params *p, int dtype) {
    return mhadv::select(q, k, d_out, lse, dv, p, dtype);
}

int mha_grad_v_set_kernel(int kernel) {
    if (kernel != DGRAD_KERNEL_AUTO && kernel != DGRAD_KERNEL_TC && kernel != DGRAD_KERNEL_SIMT)
        return DGRAD_ERR_INVALID_ARG;
    return mhadv::g_kernel_choice.exchange(kernel);
}

int mha_grad_v_check_errors(struct CUstream_st *stream) {
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    unsigned int word = 0;
    const unsigned int zero = 0;
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(&word, mhadv::g_mha_error_word, sizeof(word));
    if (e == cudaSuccess && word) e = cudaMemcpyToSymbol(mhadv::g_mha_error_word, &zero, sizeof(zero));
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return DGRAD_ERR_CUDA;
    }
    return word ? DGRAD_ERR_TIMEOUT : DGRAD_OK;
}

}  // extern "C"
