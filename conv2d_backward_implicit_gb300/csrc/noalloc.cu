// noalloc.cu -- conv2d_grad_input_noalloc: the one-call dgrad without any
// device allocation.
//
// Some callers cannot allocate device memory at the point where they need the
// gradient: code recorded into a CUDA graph whose capture mode forbids
// allocation calls, runtimes whose own arena owns all device memory and bans
// cudaMalloc/cudaMallocAsync on their execution path, and latency-critical
// loops where an allocation's implicit synchronisation is not acceptable.
// This entry point serves them: it keeps the packed weights (the only scratch
// the tensor-core path needs, unless its kernel packs the weights itself) in a
// fixed, file-scope device array instead of a stream-ordered allocation.  The caller still owns and passes grad_out,
// weight and grad_in.
//
// Costs and rules:
//  * The array is device memory of this library's module: kNoAllocScratchBytes
//    (8 MiB) are committed on a device when the module is loaded there.
//    Under CUDA's lazy module loading (the default) that is the first call of
//    this entry point on the device (its cudaGetSymbolAddress loads the
//    module); the memory then stays until the process exits.
//  * All calls share the one array.  Calls whose work overlaps on the GPU
//    (different streams without ordering, or several host threads) race on
//    it; order such calls on one stream or serialise them.
//  * The array keeps the previous call's contents.  Nothing needs clearing:
//    the pack kernel writes every byte that the dgrad kernel then reads,
//    zero padding included.
//  * The device address of the array is looked up with cudaGetSymbolAddress
//    the first time the entry point runs on a device (with that device
//    current) and cached; make that first call before any stream capture.
#include <cuda_runtime.h>

#include <mutex>

#include "conv2d_grad_input.h"
#include "dgrad_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set-up once per device).
int scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return (int)e;
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return (int)cudaSuccess;
}

int cuda_status(int err) {
    if (err == (int)cudaSuccess) return DGRAD_OK;
    (void)cudaGetLastError();
    return DGRAD_ERR_CUDA;
}

}  // namespace

extern "C" int conv2d_grad_input_noalloc(const void *grad_out, const void *weight, float *grad_in,
                                         const conv2d_grad_input_params *p, int dtype,
                                         struct CUstream_st *stream) {
    if (!grad_out || !weight || !grad_in || !p) return DGRAD_ERR_INVALID_ARG;
    dgrad::Plan plan;
    int rc = dgrad::plan_with_settings(p, dtype, &plan);
    if (rc != DGRAD_OK) return rc;
    const uintptr_t es = (uintptr_t)plan.esize;
    if ((uintptr_t)grad_out % es || (uintptr_t)weight % es || (uintptr_t)grad_in % 4)
        return DGRAD_ERR_ALIGNMENT;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (plan.kernel == DGRAD_KERNEL_SIMT)  // reads the weights unpacked: no scratch at all
        return cuda_status(dgrad::launch_simt(plan, grad_out, weight, grad_in, st));
    if (plan.workspace > kNoAllocScratchBytes) return DGRAD_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (plan.workspace > 0) {
        int e = scratch_address(&scratch);
        if (e != (int)cudaSuccess) return cuda_status(e);
        e = dgrad::launch_pack(plan, weight, scratch, st);
        if (e != (int)cudaSuccess) return cuda_status(e);
    }
    // No workspace: the kernel packs the weights itself from the weight tensor.
    return cuda_status(dgrad::launch_tc(plan, grad_out, scratch ? scratch : weight, grad_in, st));
}
