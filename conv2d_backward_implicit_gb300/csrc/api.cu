// api.cu -- the extern "C" entry points declared in include/conv2d_grad_input.h.
//
// Argument checks happen on the host before anything is enqueued; nothing
// here aborts, throws across the ABI or leaves a CUDA error pending.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>

#include "conv2d_grad_input.h"
#include "dgrad_internal.h"

namespace {

std::atomic<int> g_kernel_choice{DGRAD_KERNEL_AUTO};
std::atomic<int> g_debug_flags{0};
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
std::atomic<uint64_t> g_wait_limit_ns{kDefaultWaitNs};

int cuda_status(int err) {
    if (err == (int)cudaSuccess) return DGRAD_OK;
    (void)cudaGetLastError();  // do not leave a (non-sticky) error for the caller
    return DGRAD_ERR_CUDA;
}

bool aligned(const void *ptr, uintptr_t a) { return (reinterpret_cast<uintptr_t>(ptr) % a) == 0; }

int plan_for(const conv2d_grad_input_params *p, int dtype, dgrad::Plan *plan) {
    int rc = dgrad::make_plan(p, dtype, g_kernel_choice.load(), plan);
    if (rc != DGRAD_OK) return rc;
    plan->tc.debug_flags = plan->tc_alt.debug_flags = g_debug_flags.load();
    plan->tc.wait_limit_ns = plan->tc_alt.wait_limit_ns = g_wait_limit_ns.load();
    return DGRAD_OK;
}

int run_main(const dgrad::Plan &plan, const void *grad_out, const void *packed_or_weight,
             float *grad_in, cudaStream_t stream) {
    if (plan.kernel == DGRAD_KERNEL_SIMT)
        return cuda_status(dgrad::launch_simt(plan, grad_out, packed_or_weight, grad_in, stream));
    return cuda_status(dgrad::launch_tc(plan, grad_out, packed_or_weight, grad_in, stream));
}

// The stride-1 forward convolution of layer p (padding at most kernel - 1):
// the input gradient of the layer with the channel axes swapped, the kernel
// flipped and padding k - 1 - p, so out plays grad_in and x plays grad_out.
// The weights are flipped and transposed into a stream-ordered temporary
// buffer (and packed there unless the kernel packs them itself).
int forward_stride1(const void *x, const void *weight, float *out, const conv2d_grad_input_params *p,
                    int dtype, cudaStream_t st) {
    conv2d_grad_input_params q;
    q.batch = p->batch;
    q.in_channels = p->out_channels;
    q.in_h = p->out_h;
    q.in_w = p->out_w;
    q.out_channels = p->in_channels;
    q.kernel_h = p->kernel_h;
    q.kernel_w = p->kernel_w;
    q.stride = 1;
    q.padding_h = p->kernel_h - 1 - p->padding_h;
    q.out_h = p->in_h;
    q.out_w = p->in_w;
    q.padding_w = p->kernel_w - 1 - p->padding_w;
    dgrad::Plan plan;
    int rc = plan_for(&q, dtype, &plan);
    if (rc != DGRAD_OK) return rc;
    const size_t wt_bytes = ((size_t)p->out_channels * p->in_channels * p->kernel_h * p->kernel_w *
                                 plan.esize + 255) / 256 * 256;
    void *ws = nullptr;
    cudaError_t e = cudaMallocAsync(&ws, wt_bytes + plan.workspace, st);
    if (e != cudaSuccess) return cuda_status((int)e);
    void *packed = static_cast<char *>(ws) + wt_bytes;
    int le = dgrad::launch_flip_transpose(weight, ws, (int)p->out_channels, (int)p->in_channels,
                                          (int)p->kernel_h, (int)p->kernel_w, plan.esize, st);
    if (le == (int)cudaSuccess && plan.kernel == DGRAD_KERNEL_TC && plan.workspace > 0)
        le = dgrad::launch_pack(plan, ws, packed, st);
    const bool prepacked = plan.kernel == DGRAD_KERNEL_TC && plan.workspace > 0;
    rc = le == (int)cudaSuccess ? run_main(plan, x, prepacked ? packed : ws, out, st) : cuda_status(le);
    e = cudaFreeAsync(ws, st);
    if (rc == DGRAD_OK && e != cudaSuccess) rc = cuda_status((int)e);
    return rc;
}

// The split of a stride > 1 forward convolution (FwdSplit): false when the
// stride is above kMaxFwdStride.
bool forward_split(const conv2d_grad_input_params *p, dgrad::FwdSplit *f) {
    const int s = (int)p->stride;
    if (s < 2 || s > dgrad::kMaxFwdStride) return false;
    f->N = (int)p->batch; f->Ci = (int)p->in_channels; f->H = (int)p->in_h; f->W = (int)p->in_w;
    f->Co = (int)p->out_channels; f->kH = (int)p->kernel_h; f->kW = (int)p->kernel_w;
    f->s = s; f->ph = (int)p->padding_h; f->pw = (int)p->padding_w;
    f->OH = (int)p->out_h; f->OW = (int)p->out_w;
    auto floor_div = [](int a, int b) { return a >= 0 ? a / b : -((-a + b - 1) / b); };
    bool rh[dgrad::kMaxFwdStride] = {}, rw[dgrad::kMaxFwdStride] = {};
    for (int t = 0; t < f->kH; ++t) rh[((t - f->ph) % s + s) % s] = true;
    for (int t = 0; t < f->kW; ++t) rw[((t - f->pw) % s + s) % s] = true;
    f->nr = f->nc = 0;
    for (int r = 0; r < s; ++r) {
        if (rh[r]) f->R[f->nr++] = r;
        if (rw[r]) f->C[f->nc++] = r;
    }
    f->jmin = floor_div(-f->ph, s);
    f->imin = floor_div(-f->pw, s);
    f->KH = floor_div(f->kH - 1 - f->ph, s) - f->jmin + 1;
    f->KW = floor_div(f->kW - 1 - f->pw, s) - f->imin + 1;
    f->Hx = f->OH + f->KH - 1;
    f->Wx = f->OW + f->KW - 1;
    return true;
}

}  // namespace

namespace dgrad {
int plan_with_settings(const void *params, int dtype, Plan *out) {
    return plan_for(static_cast<const conv2d_grad_input_params *>(params), dtype, out);
}
}  // namespace dgrad

extern "C" {

int conv2d_grad_input(const void *grad_out, const void *weight, float *grad_in,
                      const conv2d_grad_input_params *p, int dtype, struct CUstream_st *stream) {
    if (!grad_out || !weight || !grad_in || !p) return DGRAD_ERR_INVALID_ARG;
    dgrad::Plan plan;
    int rc = plan_for(p, dtype, &plan);
    if (rc != DGRAD_OK) return rc;
    if (!aligned(grad_out, plan.esize) || !aligned(weight, plan.esize) || !aligned(grad_in, 4))
        return DGRAD_ERR_ALIGNMENT;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (plan.kernel == DGRAD_KERNEL_SIMT) return run_main(plan, grad_out, weight, grad_in, st);

    void *ws = nullptr;
    if (plan.workspace > 0) {
        cudaError_t e = cudaMallocAsync(&ws, plan.workspace, st);
        if (e != cudaSuccess) return cuda_status((int)e);
        int le = dgrad::launch_pack(plan, weight, ws, st);
        if (le != (int)cudaSuccess) {
            (void)cudaFreeAsync(ws, st);
            return cuda_status(le);
        }
    }
    rc = run_main(plan, grad_out, ws ? ws : weight, grad_in, st);  // no workspace: the kernel packs
    if (ws) {
        cudaError_t e = cudaFreeAsync(ws, st);
        if (rc == DGRAD_OK && e != cudaSuccess) rc = cuda_status((int)e);
    }
    return rc;
}

int conv2d_forward(const void *x, const void *weight, float *out, const conv2d_grad_input_params *p,
                   int dtype, struct CUstream_st *stream) {
    if (!x || !weight || !out || !p) return DGRAD_ERR_INVALID_ARG;
    // The layer itself must be valid (same checks as its input gradient).
    dgrad::Plan layer;
    int rc = plan_for(p, dtype, &layer);
    if (rc != DGRAD_OK) return rc;
    if (!aligned(x, layer.esize) || !aligned(weight, layer.esize) || !aligned(out, 4)) return DGRAD_ERR_ALIGNMENT;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (p->stride == 1) {
        if (p->padding_h > p->kernel_h - 1 || p->padding_w > p->kernel_w - 1) return DGRAD_ERR_UNSUPPORTED;
        return forward_stride1(x, weight, out, p, dtype, st);
    }
    // Stride s > 1: the same output as a stride-1 valid correlation of the
    // space-to-depth copy X'' of x with the rearranged weights W'' (FwdSplit
    // in dgrad_internal.h): with kh - ph = s j + r, input row s oh - ph + kh
    // is row oh + j - jmin of residue r's decimated image.
    dgrad::FwdSplit f;
    if (!forward_split(p, &f)) return DGRAD_ERR_UNSUPPORTED;
    conv2d_grad_input_params q;
    q.batch = p->batch;
    q.in_channels = (uint32_t)(f.nr * f.nc) * p->in_channels;
    q.in_h = (uint32_t)f.Hx;
    q.in_w = (uint32_t)f.Wx;
    q.out_channels = p->out_channels;
    q.kernel_h = (uint32_t)f.KH;
    q.kernel_w = (uint32_t)f.KW;
    q.stride = 1;
    q.padding_h = 0;
    q.out_h = p->out_h;
    q.out_w = p->out_w;
    q.padding_w = 0;
    dgrad::Plan inner;
    rc = plan_for(&q, dtype, &inner);
    if (rc != DGRAD_OK) return rc;
    const size_t es = (size_t)layer.esize;
    const size_t xs_bytes = ((size_t)q.batch * q.in_channels * q.in_h * q.in_w * es + 255) / 256 * 256;
    const size_t ws_bytes = ((size_t)q.out_channels * q.in_channels * q.kernel_h * q.kernel_w * es + 255) / 256 * 256;
    void *buf = nullptr;
    cudaError_t e = cudaMallocAsync(&buf, xs_bytes + ws_bytes, st);
    if (e != cudaSuccess) return cuda_status((int)e);
    void *xs = buf, *wsplit = static_cast<char *>(buf) + xs_bytes;
    int le = dgrad::launch_space_to_depth(f, x, xs, layer.esize, st);
    if (le == (int)cudaSuccess) le = dgrad::launch_split_weights(f, weight, wsplit, layer.esize, st);
    rc = le == (int)cudaSuccess ? forward_stride1(xs, wsplit, out, &q, dtype, st) : cuda_status(le);
    e = cudaFreeAsync(buf, st);
    if (rc == DGRAD_OK && e != cudaSuccess) rc = cuda_status((int)e);
    return rc;
}

size_t conv2d_grad_input_workspace_size(const conv2d_grad_input_params *p, int dtype) {
    if (!p) return 0;
    dgrad::Plan plan;
    if (plan_for(p, dtype, &plan) != DGRAD_OK) return 0;
    return plan.kernel == DGRAD_KERNEL_TC ? plan.workspace : 0;
}

int conv2d_grad_input_pack_weight(const void *weight, void *packed, size_t packed_bytes,
                                  const conv2d_grad_input_params *p, int dtype,
                                  struct CUstream_st *stream) {
    if (!weight || !p) return DGRAD_ERR_INVALID_ARG;
    dgrad::Plan plan;
    int rc = plan_for(p, dtype, &plan);
    if (rc != DGRAD_OK) return rc;
    if (plan.kernel != DGRAD_KERNEL_TC || plan.workspace == 0) return DGRAD_OK;  // nothing to pack
    if (!packed) return DGRAD_ERR_INVALID_ARG;
    if (packed_bytes < plan.workspace) return DGRAD_ERR_WORKSPACE;
    if (!aligned(weight, plan.esize) || !aligned(packed, 16)) return DGRAD_ERR_ALIGNMENT;
    return cuda_status(dgrad::launch_pack(plan, weight, packed, reinterpret_cast<cudaStream_t>(stream)));
}

int conv2d_grad_input_prepacked(const void *grad_out, const void *packed, float *grad_in,
                                const conv2d_grad_input_params *p, int dtype,
                                struct CUstream_st *stream) {
    if (!grad_out || !grad_in || !p) return DGRAD_ERR_INVALID_ARG;
    dgrad::Plan plan;
    int rc = plan_for(p, dtype, &plan);
    if (rc != DGRAD_OK) return rc;
    if (!packed) return DGRAD_ERR_INVALID_ARG;  // packed weights, or the weights themselves
    const uintptr_t pa = plan.workspace > 0 ? 16 : (uintptr_t)plan.esize;
    if (!aligned(grad_out, plan.esize) || !aligned(grad_in, 4) || !aligned(packed, pa))
        return DGRAD_ERR_ALIGNMENT;
    return run_main(plan, grad_out, packed, grad_in, reinterpret_cast<cudaStream_t>(stream));
}

int conv2d_grad_input_check_errors(struct CUstream_st *stream) {
    cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_status((int)e);
    unsigned int flag = 0;
    int le = dgrad::tc_read_and_clear_error(&flag);
    if (le != (int)cudaSuccess) return cuda_status(le);
    return flag ? DGRAD_ERR_TIMEOUT : DGRAD_OK;
}

const char *conv2d_grad_input_status_string(int status) {
    switch (status) {
    case DGRAD_OK: return "ok";
    case DGRAD_ERR_INVALID_ARG: return "invalid argument";
    case DGRAD_ERR_SHAPE: return "invalid or inconsistent shape";
    case DGRAD_ERR_ALIGNMENT: return "misaligned pointer";
    case DGRAD_ERR_UNSUPPORTED: return "unsupported size or kernel choice";
    case DGRAD_ERR_CUDA: return "CUDA runtime error";
    case DGRAD_ERR_TIMEOUT: return "device wait timed out";
    case DGRAD_ERR_WORKSPACE: return "packed-weight buffer too small (the one passed in, or the 8 MiB array of the no-alloc entry point)";
    default: return "unknown status";
    }
}

int conv2d_grad_input_select_kernel(const conv2d_grad_input_params *p, int dtype) {
    if (!p) return -DGRAD_ERR_INVALID_ARG;
    dgrad::Plan plan;
    int rc = plan_for(p, dtype, &plan);
    if (rc != DGRAD_OK) return -rc;
    return plan.kernel == DGRAD_KERNEL_TC && plan.tc.pos_m ? DGRAD_KERNEL_TC_POSM : plan.kernel;
}

int conv2d_grad_input_set_kernel(int kernel) {
    if (kernel != DGRAD_KERNEL_AUTO && kernel != DGRAD_KERNEL_TC && kernel != DGRAD_KERNEL_SIMT &&
        kernel != DGRAD_KERNEL_TC_POSM)
        return -DGRAD_ERR_INVALID_ARG;
    return g_kernel_choice.exchange(kernel);
}

uint64_t conv2d_grad_input_set_wait_limit_ns(uint64_t ns) {
    return g_wait_limit_ns.exchange(ns ? ns : kDefaultWaitNs);
}

int conv2d_grad_input_set_debug(int flags) { return g_debug_flags.exchange(flags); }

}  // extern "C"
