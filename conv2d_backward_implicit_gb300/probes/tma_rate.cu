// tma_rate.cu -- measures TMA load throughput on this GPU: every SM loads 64
// boxes of one shape from an L2-resident 12.8 MB source (the ResNet grad_out
// size) into a ring of slots, the copies issued by one or several warps (or
// lanes of one warp), each issuer waiting (bounded) for its own slot before
// reusing it.  Prints cycles per copy on CTA 0 and the aggregate rate.  Mode
// 0 = 4-D tensor box, 1 = one bulk copy per channel, 2 = one bulk copy of the
// box's bytes.  A measurement aid of bench.py (--probe tma); not part of the
// library.
#include <cstdio>
#include <cstdint>
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ void expect(uint32_t bar, uint32_t bytes) { asm volatile("{\n.reg .b64 s;\nmbarrier.arrive.expect_tx.shared::cta.b64 s, [%0], %1;\n}" :: "r"(bar), "r"(bytes) : "memory"); }
__device__ __forceinline__ bool trywait(uint32_t bar, uint32_t ph) { uint32_t ok; asm volatile("{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\nselp.u32 %0, 1, 0, p;\n}" : "=r"(ok) : "r"(bar), "r"(ph) : "memory"); return ok; }
struct Cfg { int mode; int reps; int nbox_src; int chans; int rows; int cols; int esize; int slots; int issuers; int lanes; };
// mode 0: 4-D tensor box [cols][rows][chans] of a [N][C][H][W] tensor; mode 1: one bulk copy per channel (rows*cols contiguous);
// mode 2: one bulk copy of the whole box bytes
__global__ void __launch_bounds__(256, 1) ktma(const __grid_constant__ CUtensorMap map, const uint8_t *src, Cfg c, long long *out, int H, int W, int C, int N) {
  extern __shared__ __align__(1024) uint8_t sm[];
  __shared__ uint64_t bar[8];
  uint8_t *base = (uint8_t *)(((uintptr_t)sm + 1023) & ~(uintptr_t)1023);
  const uint32_t box_bytes = (uint32_t)(c.chans * c.rows * c.cols * c.esize);
  const uint32_t slot_bytes = (box_bytes + 1023) / 1024 * 1024;
  if (threadIdx.x == 0) {
    for (int s = 0; s < 8; ++s) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" :: "r"(su32(&bar[s])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  // issuers: lane 0 of warps 0..issuers-1, or (lanes) lanes 0..issuers-1 of warp 0
  const int who = c.lanes ? (int)threadIdx.x : (int)(threadIdx.x >> 5);
  if (c.lanes ? (threadIdx.x >= (unsigned)c.issuers) : ((threadIdx.x & 31) != 0 || who >= c.issuers)) return;
  const int per = c.slots / c.issuers;  // slots of this issuer: who*per .. +per-1
  long long t0 = clock64();
  uint32_t ok = 1;
  for (int i = 0; i < c.reps / c.issuers && ok; ++i) {
    const int s = who * per + i % per;
    const uint32_t ph = (uint32_t)((i / per) & 1);
    if (i >= per) {  // wait for the slot's previous load
      ok = 0;
      for (long long sp = 0; sp < 20000000LL && !ok; ++sp) ok = trywait(su32(&bar[s]), ph ^ 1u);
      if (!ok) break;
    }
    const int b = (int)((blockIdx.x * 7919LL + i * 4 + who) % c.nbox_src);  // which box of the source
    const uint32_t dst = su32(base + s * slot_bytes);
    const uint32_t mb = su32(&bar[s]);
    expect(mb, box_bytes);
    const int n = b % N, cg = (b / N) % (C / c.chans), rg = (b / N / (C / c.chans)) % (H / c.rows);
    if (c.mode == 0) {
      asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];"
                   :: "r"(dst), "l"((uint64_t)&map), "r"(0), "r"(rg * c.rows), "r"(cg * c.chans), "r"(n), "r"(mb) : "memory");
    } else if (c.mode == 1) {
      const uint32_t per = (uint32_t)(c.rows * c.cols * c.esize);
      for (int k = 0; k < c.chans; ++k) {
        const uint8_t *g = src + ((((size_t)n * C + cg * c.chans + k) * H + rg * c.rows) * W) * c.esize;
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" :: "r"(dst + k * per), "l"(g), "r"(per), "r"(mb) : "memory");
      }
    } else {
      const uint8_t *g = src + (size_t)b * box_bytes % ((size_t)N * C * H * W * c.esize - box_bytes) / 16 * 16;
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" :: "r"(dst), "l"(g), "r"(box_bytes), "r"(mb) : "memory");
    }
  }
  const int myreps = c.reps / c.issuers;
  for (int s = 0; s < per && ok; ++s) {  // drain
    const int i = myreps - per + s; if (i < 0) continue;
    const uint32_t ph = (uint32_t)((i / per) & 1);
    ok = 0; for (long long sp = 0; sp < 20000000LL && !ok; ++sp) ok = trywait(su32(&bar[who * per + i % per]), ph);
  }
  long long t1 = clock64();
  if (blockIdx.x == 0 && who == 0) out[0] = ok ? t1 - t0 : -1;
}
int main() {
  const int N = 32, C = 64, H = 56, W = 56, E = 2;
  size_t bytes = (size_t)N * C * H * W * E;  // 12.8 MB: the ResNet grad_out
  uint8_t *src; cudaMalloc(&src, bytes); cudaMemset(src, 1, bytes);
  long long *dout; cudaMalloc(&dout, 8);
  void *fnp = nullptr; cudaDriverEntryPointQueryResult q;
  cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault, &q);
  auto fn = (PFN_cuTensorMapEncodeTiled_v12000)fnp;
  int sms; cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  cudaFuncSetAttribute(ktma, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
  // mode, reps, source boxes, channels, rows, columns, element size, slots, issuers, lanes
  Cfg cs[] = {{0, 64, 100000, 16, 7, 56, 2, 4, 1, 0}, {0, 64, 100000, 64, 7, 56, 2, 2, 1, 0},
              {2, 64, 100000, 16, 7, 56, 2, 4, 1, 0}, {1, 64, 100000, 16, 7, 56, 2, 4, 1, 0},
              {0, 64, 100000, 16, 7, 56, 2, 4, 2, 0}, {0, 64, 100000, 16, 7, 56, 2, 4, 4, 0},
              {0, 64, 100000, 16, 7, 56, 2, 4, 4, 1}, {2, 64, 100000, 16, 7, 56, 2, 8, 8, 0}};
  for (auto c : cs) {
    CUtensorMap map;
    cuuint64_t dims[4] = {(cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)C, (cuuint64_t)N};
    cuuint64_t str[3] = {(cuuint64_t)W * E, (cuuint64_t)H * W * E, (cuuint64_t)C * H * W * E};
    cuuint32_t box[4] = {(cuuint32_t)c.cols, (cuuint32_t)c.rows, (cuuint32_t)c.chans, 1}, es[4] = {1, 1, 1, 1};
    CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 4, src, dims, str, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { printf("encode failed %d\n", (int)r); continue; }
    const int box_bytes = c.chans * c.rows * c.cols * c.esize;
    const int smem = c.slots * ((box_bytes + 1023) / 1024 * 1024) + 1024;
    const int threads = 32 * c.issuers;
    if (smem > 200 * 1024) { printf("skip\n"); continue; }
    float best = 1e30f; long long cyc = 0;
    for (int rep = 0; rep < 3; ++rep) {
      cudaEvent_t e0, e1; cudaEventCreate(&e0); cudaEventCreate(&e1);
      cudaEventRecord(e0);
      ktma<<<sms, threads, smem>>>(map, src, c, dout, H, W, C, N);
      cudaEventRecord(e1);
      cudaError_t e = cudaEventSynchronize(e1);
      if (e != cudaSuccess) { printf("error %s\n", cudaGetErrorString(e)); return 1; }
      float ms; cudaEventElapsedTime(&ms, e0, e1);
      cudaMemcpy(&cyc, dout, 8, cudaMemcpyDeviceToHost);
      if (ms < best) best = ms;
    }
    const double total = (double)sms * c.reps * box_bytes;
    printf("%s issuers %d mode %d box %dch x %drows x %dcols (%d B) slots %d: cta0 %.0f cycles/box, all SMs %.1f GB/s (%.1f us)\n", c.lanes ? "lane" : "warp", c.issuers, c.mode, c.chans, c.rows, c.cols,
           box_bytes, c.slots, cyc / (double)(c.reps / c.issuers), total / (best * 1e-3) / 1e9, best * 1e3);
  }
  return 0;
}
