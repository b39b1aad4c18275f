// tma_store_rate.cu -- measures TMA tensor-store throughput on this GPU:
// [chans][rows][cols] float32 boxes of a [32][64][56][56] float32 tensor (the
// ResNet grad_in size), every SM storing 64 boxes from shared memory with
// `inflight` stores outstanding per issuing thread.  A measurement aid of
// bench.py (--probe tma_store); not part of the library.
#include <cstdio>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
struct Cfg { int reps, chans, rows, cols, inflight; };
__global__ void __launch_bounds__(32, 1) kst(const __grid_constant__ CUtensorMap map, Cfg c, long long *out, int H, int C, int N) {
  extern __shared__ __align__(1024) uint8_t sm[];
  uint8_t *base = (uint8_t *)(((uintptr_t)sm + 1023) & ~(uintptr_t)1023);
  for (int i = threadIdx.x; i < c.chans * c.rows * c.cols; i += 32) ((float *)base)[i] = (float)i;
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  __syncwarp();
  if (threadIdx.x != 0) return;
  long long t0 = clock64();
  for (int i = 0; i < c.reps; ++i) {
    const int b = (int)((blockIdx.x * 7919LL + i * 13) % 100000);
    const int n = b % N, cg = (b / N) % (C / c.chans), rg = (b / N / (C / c.chans)) % (H / c.rows);
    asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];"
                 :: "l"((uint64_t)&map), "r"(0), "r"(rg * c.rows), "r"(cg * c.chans), "r"(n), "r"(su32(base)) : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    if (c.inflight == 1) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    else if (c.inflight == 2) asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
    else asm volatile("cp.async.bulk.wait_group.read 3;" ::: "memory");
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
  long long t1 = clock64();
  if (blockIdx.x == 0) out[0] = t1 - t0;
}
int main() {
  const int N = 32, C = 64, H = 56, W = 56;
  size_t bytes = (size_t)N * C * H * W * 4;
  float *dst; cudaMalloc(&dst, bytes);
  long long *dout; cudaMalloc(&dout, 8);
  void *fnp = nullptr; cudaDriverEntryPointQueryResult q;
  cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault, &q);
  auto fn = (PFN_cuTensorMapEncodeTiled_v12000)fnp;
  int sms; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  cudaFuncSetAttribute(kst, cudaFuncAttributeMaxDynamicSharedMemorySize, 100 * 1024);
  Cfg cs[] = {{64, 16, 1, 56, 1}, {64, 16, 1, 56, 2}, {64, 16, 1, 56, 4}, {64, 16, 4, 56, 1}, {64, 16, 4, 56, 4}, {64, 64, 1, 56, 1}, {64, 64, 4, 56, 1}, {64, 8, 1, 56, 4}};
  for (auto c : cs) {
    CUtensorMap map;
    cuuint64_t dims[4] = {(cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)C, (cuuint64_t)N};
    cuuint64_t str[3] = {(cuuint64_t)W * 4, (cuuint64_t)H * W * 4, (cuuint64_t)C * H * W * 4};
    cuuint32_t box[4] = {(cuuint32_t)c.cols, (cuuint32_t)c.rows, (cuuint32_t)c.chans, 1}, es[4] = {1, 1, 1, 1};
    CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dst, dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { printf("encode failed %d\n", (int)r); continue; }
    const int box_bytes = c.chans * c.rows * c.cols * 4;
    float best = 1e30f; long long cyc = 0;
    for (int rep = 0; rep < 3; ++rep) {
      cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
      cudaEventRecord(e0);
      kst<<<sms, 32, box_bytes + 1024>>>(map, c, dout, H, C, N);
      cudaEventRecord(e1);
      cudaError_t e = cudaEventSynchronize(e1);
      if (e != cudaSuccess) { printf("error %s\n", cudaGetErrorString(e)); return 1; }
      float ms; cudaEventElapsedTime(&ms, e0, e1);
      cudaMemcpy(&cyc, dout, 8, cudaMemcpyDeviceToHost);
      if (ms < best) best = ms;
    }
    printf("store box %dch x %drows x %dcols (%d B) inflight %d: cta0 %.0f cycles/box, all SMs %.1f GB/s\n", c.chans, c.rows, c.cols, box_bytes, c.inflight,
           cyc / (double)c.reps, (double)sms * c.reps * box_bytes / (best * 1e-3) / 1e9);
  }
  return 0;
}
