// mma_rate.cu -- measures how long back-to-back tcgen05.mma instructions of one
// shape take on this GPU: one CTA, zero operands in shared memory (K-major,
// 128-byte swizzled), one accumulator or two alternating, 512 MMAs issued by
// one thread, timed with clock64 until their commit lands (a bounded wait).
// Prints cycles per MMA for the shapes the dgrad kernels use.  A measurement
// aid of bench.py (--probe mma); not part of the library.
#include <cstdio>
#include <cstdint>
#include <cuda_runtime.h>
__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ uint64_t desc(uint32_t addr) {
  uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
  d |= (uint64_t)1 << 16; d |= (uint64_t)(1024 >> 4) << 32; d |= (uint64_t)1 << 46; d |= (uint64_t)2 << 61;
  return d;
}
template <bool TF32>
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  if (TF32) asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n}" :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
  else asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\ntcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" :: "r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
struct Cfg { int tf32, M, N, n, alt; };
__global__ void __launch_bounds__(128, 1) kmb(Cfg c, long long *out) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar; __shared__ uint32_t tbase;
  uint8_t *base = (uint8_t *)(((uintptr_t)sm + 1023) & ~(uintptr_t)1023);
  for (int i = threadIdx.x; i < 65536 / 4; i += 128) ((uint32_t *)base)[i] = 0;
  if (threadIdx.x == 0) { asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(su32(&bar))); asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
  if (threadIdx.x < 32) { asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" :: "r"(su32(&tbase)) : "memory"); asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tm = tbase;
  if (threadIdx.x == 0) {
    const uint32_t fmt = c.tf32 ? 2u : 1u;
    const uint32_t idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(c.N >> 3) << 17) | ((uint32_t)(c.M >> 4) << 24);
    const uint64_t a0 = desc(su32(base)), b0 = desc(su32(base + 32768));
    long long t0 = clock64();
    for (int i = 0; i < c.n; ++i) {
      const uint32_t d = tm + (c.alt ? (uint32_t)((i & 1) * 256) : 0u);
      const uint64_t adv = (uint64_t)(2 * (i & 3));
      if (c.tf32) mma<true>(d, a0 + adv, b0 + adv, idesc, i >= 2 ? 1u : 0u);
      else mma<false>(d, a0 + adv, b0 + adv, idesc, i >= 2 ? 1u : 0u);
    }
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(su32(&bar)) : "memory");
    uint32_t ok = 0;
    for (long long spin = 0; spin < 50000000LL && !ok; ++spin)
      asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\nselp.u32 %0, 1, 0, p;\n}" : "=r"(ok) : "r"(su32(&bar)) : "memory");
    long long t1 = clock64();
    out[0] = ok ? (t1 - t0) : -1;
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (threadIdx.x < 32) { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" :: "r"(tm) : "memory"); }
}
int main() {
  cudaFuncSetAttribute(kmb, cudaFuncAttributeMaxDynamicSharedMemorySize, 66560 + 1024);
  long long *dout; cudaMalloc(&dout, 8);
  Cfg cs[] = {{1,128,16,512,0},{1,128,32,512,0},{1,128,64,512,0},{1,128,64,512,1},{1,128,128,512,0},{1,128,256,512,0},
              {0,128,64,512,0},{0,128,64,512,1},{0,128,128,512,0},{0,128,192,512,0},{0,128,256,512,0},{0,64,256,512,0},{0,64,128,512,0}};
  for (auto c : cs) {
    long long best = -1;
    for (int r = 0; r < 3; ++r) {
      kmb<<<1, 128, 66560 + 1024>>>(c, dout);
      cudaError_t e = cudaDeviceSynchronize();
      if (e != cudaSuccess) { printf("error %s\n", cudaGetErrorString(e)); return 1; }
      long long v; cudaMemcpy(&v, dout, 8, cudaMemcpyDeviceToHost);
      if (best < 0 || (v >= 0 && v < best)) best = v;
    }
    printf("%s M%d N%d %s: %.1f cycles/mma\n", c.tf32 ? "tf32 K8 " : "bf16 K16", c.M, c.N, c.alt ? "2 acc" : "1 acc", best / (double)c.n);
  }
  return 0;
}
