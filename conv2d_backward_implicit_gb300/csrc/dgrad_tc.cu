// dgrad_tc.cu -- the sm_103a tensor-core dgrad kernel (tcgen05 + TMEM + mbarrier).
//
// What it computes is the page's implicit GEMM (conv2d_grad_input_gemm_coop.wgsl,
// header comment): per batch item C[Ci, H*W] = A[Ci, K] x B[K, H*W], K =
// Co*kH*kW, with the exact-adjoint index map of its strided staging branch.
// How it computes it is GB300-first rather than the shader's 2x2 grid of
// cooperative-matrix tiles with two workgroup barriers per K step:
//
//  * The stride's sub-pixel phases (dgrad_internal.h) make every phase a
//    dense stride-1 correlation: structural-zero products are never issued.
//  * The im2col operand is never materialised per tap: raw grad_out slices
//    (TMA tensor loads or 1-D bulk copies) are turned by gather warps into one
//    frame window per stage, 128-byte K-major swizzled rows in shared memory,
//    and every tap is that window read through a descriptor whose start is
//    shifted by the tap's offset.  For 1x1 problems the window is kept
//    MN-major (channel rows of positions) and only regrouped.
//  * The weights come pre-packed (pack.cu) in exactly their shared-memory
//    image and move with bulk copies: resident when they fit, otherwise a
//    ring of per-(chunk, tap group) stages.
//  * One thread issues tcgen05.mma (kind::f16 for bf16/fp16, kind::tf32 for
//    fp32) into double-buffered TMEM accumulators; epilogue warps drain one
//    buffer with tcgen05.ld while the next tile's MMAs fill the other, and
//    store float32 NCHW grad_in through TMA tensor stores (whole rows or
//    planes) or predicated stores.  Persistent grid: one CTA per SM.
//
// Kernel variants (one compiled kernel each, see Roles): General (input
// channels on M -- 64 or 128 rows -- and up to 256 positions on N), Frame64
// (stride 1, 16-bit, rows up to 56: a 64-wide frame filled by ldmatrix
// transposes), PosM (opt-in: positions on M, kernel-row taps on N), Pair
// (stride 2: the two column phases of the same rows from one window into two
// accumulators, stored as whole rows) and Stacked (few input channels:
// positions on M, every phase's channels stacked on N).
//
// Every mbarrier wait is bounded by a wall-clock limit (globaltimer).  On
// expiry the CTA raises an abort flag in shared memory, sets bit 0 of the
// device error word, drains copies and MMAs it has in flight, releases TMEM
// and returns; no wait is unbounded and nothing traps.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <atomic>

#include "conv2d_grad_input.h"
#include "dgrad_internal.h"

namespace dgrad {

__device__ unsigned int g_dgrad_error_word = 0;

namespace {

// Kernel variants.  Pair and Stacked are the general mode with its paired
// column-phase epilogue or its stacked-phase MMA and epilogue compiled in
// (separate variants keep the general one's register allocation lean).
constexpr int kVarGeneral = 0, kVarFrame64 = 1, kVarPosM = 2, kVarPair = 3, kVarStacked = 4, kVarMN = 5;
__host__ __device__ constexpr bool is_general(int v) {
    return v == kVarGeneral || v == kVarPair || v == kVarStacked || v == kVarMN;
}

// Warp roles of each variant: epilogue warps first, then the MMA warp, the
// producer warp(s) and the gather warps.  w2_warp >= 0: a second producer
// warp -- with streamed weights and raw slices, one warp issues the raw
// slices and the other the weight stages, because one thread's bulk copies
// run one after another (each about 1.1K cycles, whatever its size) while
// copies issued by different warps overlap.
template <int V>
struct Roles {
    static constexpr int epi_warps = kEpiWarps, mma_warp = kMmaWarp, w_warp = kWWarp, w2_warp = -1;
    static constexpr int g_warp0 = kGWarp0, g_warps = kGWarps, threads = kThreads;
};
// Paired column phases and the MN-major 1x1 mode stream their weights: two
// producer warps and five gather warps.
template <>
struct Roles<kVarPair> {
    static constexpr int epi_warps = kEpiWarps, mma_warp = kMmaWarp, w_warp = kWWarp, w2_warp = kWWarp + 1;
    static constexpr int g_warp0 = kGWarp0 + 1, g_warps = kGWarps - 1, threads = kThreads;
};
template <>
struct Roles<kVarMN> {
    static constexpr int epi_warps = kEpiWarps, mma_warp = kMmaWarp, w_warp = kWWarp, w2_warp = kWWarp + 1;
    static constexpr int g_warp0 = kGWarp0 + 1, g_warps = kGWarps - 1, threads = kThreads;
};
// Stacked-phase mode: a short epilogue (one TMEM read and s^2 Ci stores per
// position) and a long gather, so four epilogue warps (one per TMEM lane
// quadrant) and ten gather warps.
template <>
struct Roles<kVarStacked> {
    static constexpr int epi_warps = 4, mma_warp = 4, w_warp = 5, w2_warp = -1;
    static constexpr int g_warp0 = 6, g_warps = 10, threads = 512;
};
template <>
struct Roles<kVarPosM> {
    static constexpr int epi_warps = kPmEpiWarps, mma_warp = kPmMmaWarp, w_warp = kPmWWarp, w2_warp = -1;
    static constexpr int g_warp0 = kPmGWarp0, g_warps = kPmGWarps, threads = kPmThreads;
};


struct Shared {
    uint64_t full_g[4], empty_g[4], full_w[kMaxW], empty_w[kMaxW], full_raw[kMaxRaw],
        empty_raw[kMaxRaw];
    uint64_t acc_full[2], acc_empty[2];
    uint64_t x_full[16], x_empty[16];  // positions-on-M epilogue boundary exchange
    uint64_t full_early[kMaxEarly];    // raw slices parked in G stage 1
    uint64_t early_free;               // every gather warp is done with them
    uint64_t w_full, mma_done;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(Shared) <= kBarrierBytes, "barrier block too large");

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar)
        : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile(
        "{\n\t.reg .b64 st;\n\t"
        "mbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
        "r"(bytes)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probe of a phase (no suspend window, unlike try_wait).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch: wait until the preceding kernel of the
// stream has completed and its writes are visible; let the next kernel of the
// stream start its own prologue.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                         uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// TMA tensor load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            int z, int w, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes "
        "[%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
        : "memory");
}

// TMA tensor prefetch of one box into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap *map, int x, int y, int z, int w) {
    asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}

// Four 8x8 16-bit matrices, transposed on the way into registers (rows of
// 16 bytes at the addresses lanes 8m..8m+7 give for matrix m).
__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr)
                 : "memory");
}

// Four 8x8 16-bit matrices from registers into rows of 16 bytes.
__device__ __forceinline__ void stmatrix_x4(uint32_t addr, const uint32_t (&r)[4]) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.shared.b16 [%0], {%1, %2, %3, %4};" ::"r"(addr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3])
                 : "memory");
}

__device__ __forceinline__ uint32_t ld_shared_u16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr) : "memory");
    return v;
}

// float32 bits rounded to TF32 (nearest, ties away from zero): the operand
// precision of kind::tf32.
__device__ __forceinline__ uint32_t to_tf32(uint32_t bits) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(__uint_as_float(bits)));
    return r;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ float4 ld_shared_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

__device__ __forceinline__ float ld_shared_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ldg_u16(const unsigned short *p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_b32(const float *p) {
    uint32_t v;
    asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// The MMA roles run on their whole warp (control flow and descriptor
// arithmetic warp-uniform, which issues the small MMAs faster than a lone
// divergent lane); the tcgen05 instructions themselves execute in lane 0 only.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred q;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 q, l, 0;\n\t"
        "@q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}

template <bool TF32>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    if constexpr (TF32) {
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 q, l, 0;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "@q tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p, q;\n\t.reg .u32 l;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 q, l, 0;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "@q tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}

// 32 lanes x 16 consecutive 32-bit columns of TMEM into registers.  The load
// is asynchronous: the registers are valid only after tmem_wait_ld(r).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

// Waits for this thread's outstanding TMEM loads; naming the destination
// registers as in-out operands keeps their uses after the wait.
__device__ __forceinline__ void tmem_wait_ld4(uint32_t (&r)[4][16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0][0]), "+r"(r[0][1]), "+r"(r[0][2]), "+r"(r[0][3]), "+r"(r[0][4]), "+r"(r[0][5]), "+r"(r[0][6]), "+r"(r[0][7]), "+r"(r[0][8]), "+r"(r[0][9]), "+r"(r[0][10]), "+r"(r[0][11]), "+r"(r[0][12]), "+r"(r[0][13]), "+r"(r[0][14]), "+r"(r[0][15]), "+r"(r[1][0]), "+r"(r[1][1]), "+r"(r[1][2]), "+r"(r[1][3]), "+r"(r[1][4]), "+r"(r[1][5]), "+r"(r[1][6]), "+r"(r[1][7]), "+r"(r[1][8]), "+r"(r[1][9]), "+r"(r[1][10]), "+r"(r[1][11]), "+r"(r[1][12]), "+r"(r[1][13]), "+r"(r[1][14]), "+r"(r[1][15]), "+r"(r[2][0]), "+r"(r[2][1]), "+r"(r[2][2]), "+r"(r[2][3]), "+r"(r[2][4]), "+r"(r[2][5]), "+r"(r[2][6]), "+r"(r[2][7]), "+r"(r[2][8]), "+r"(r[2][9]), "+r"(r[2][10]), "+r"(r[2][11]), "+r"(r[2][12]), "+r"(r[2][13]), "+r"(r[2][14]), "+r"(r[2][15]), "+r"(r[3][0]), "+r"(r[3][1]), "+r"(r[3][2]), "+r"(r[3][3]), "+r"(r[3][4]), "+r"(r[3][5]), "+r"(r[3][6]), "+r"(r[3][7]), "+r"(r[3][8]), "+r"(r[3][9]), "+r"(r[3][10]), "+r"(r[3][11]), "+r"(r[3][12]), "+r"(r[3][13]), "+r"(r[3][14]), "+r"(r[3][15])
                 :
                 : "memory");
}

// TMA tensor store of a [16 ch][1 row][W] float32 box from shared memory
// (bulk-group completion), and the waits on this thread's bulk groups.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap *map, uint32_t smem_src, int x,
                                             int y, int z, int w) {
    asm volatile(
        "cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4}], [%5];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(w), "r"(smem_src)
        : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// The same for a 3-D tensor map.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *map, uint32_t smem_src, int x, int y,
                                             int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(z), "r"(smem_src)
        : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// None of this thread's bulk groups may still be reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// All but the latest bulk group of this thread are done reading shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() {
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// 32 lanes x 8 / 4 consecutive 32-bit TMEM columns, asynchronous like tmem_ld16.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t *r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}

__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t *r) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
}

// 16 lanes x 64 columns (eight 16x256b blocks): thread t gets, for block b,
// r[4b], r[4b+1] = lane t/4, columns 8b + 2(t%4) + {0, 1} and r[4b+2],
// r[4b+3] = lane t/4 + 8, the same columns.  Asynchronous like tmem_ld16.
__device__ __forceinline__ void tmem_ld_16x256b_x8(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x256b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
        "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
        "%29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_wait_ld32(uint32_t (&r)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                   "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                   "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
                   "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
                   "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
                   "+r"(r[31])
                 :
                 : "memory");
}

__device__ __forceinline__ void st_shared_v2(uint32_t addr, uint32_t a, uint32_t b) {
    asm volatile("st.shared.v2.b32 [%0], {%1, %2};" ::"r"(addr), "r"(a), "r"(b) : "memory");
}

// Waits for this thread's outstanding TMEM loads into r[0..2][0..15].
__device__ __forceinline__ void tmem_wait_ld3(uint32_t (&r)[3][16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0][0]), "+r"(r[0][1]), "+r"(r[0][2]), "+r"(r[0][3]), "+r"(r[0][4]), "+r"(r[0][5]), "+r"(r[0][6]), "+r"(r[0][7]), "+r"(r[0][8]), "+r"(r[0][9]), "+r"(r[0][10]), "+r"(r[0][11]), "+r"(r[0][12]), "+r"(r[0][13]), "+r"(r[0][14]), "+r"(r[0][15]), "+r"(r[1][0]), "+r"(r[1][1]), "+r"(r[1][2]), "+r"(r[1][3]), "+r"(r[1][4]), "+r"(r[1][5]), "+r"(r[1][6]), "+r"(r[1][7]), "+r"(r[1][8]), "+r"(r[1][9]), "+r"(r[1][10]), "+r"(r[1][11]), "+r"(r[1][12]), "+r"(r[1][13]), "+r"(r[1][14]), "+r"(r[1][15]), "+r"(r[2][0]), "+r"(r[2][1]), "+r"(r[2][2]), "+r"(r[2][3]), "+r"(r[2][4]), "+r"(r[2][5]), "+r"(r[2][6]), "+r"(r[2][7]), "+r"(r[2][8]), "+r"(r[2][9]), "+r"(r[2][10]), "+r"(r[2][11]), "+r"(r[2][12]), "+r"(r[2][13]), "+r"(r[2][14]), "+r"(r[2][15])
                 :
                 : "memory");
}

// Waits for this thread's outstanding TMEM loads into r[0..3][0..15].
__device__ __forceinline__ void tmem_wait_ld16x4(uint32_t (&r)[4][16]) {
    tmem_wait_ld4(r);
}

// Waits for this thread's outstanding TMEM loads into r[0..1][0..15].
__device__ __forceinline__ void tmem_wait_ld16x2(uint32_t (&r)[2][16]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0][0]), "+r"(r[0][1]), "+r"(r[0][2]), "+r"(r[0][3]), "+r"(r[0][4]), "+r"(r[0][5]), "+r"(r[0][6]), "+r"(r[0][7]), "+r"(r[0][8]), "+r"(r[0][9]), "+r"(r[0][10]), "+r"(r[0][11]), "+r"(r[0][12]), "+r"(r[0][13]), "+r"(r[0][14]), "+r"(r[0][15]), "+r"(r[1][0]), "+r"(r[1][1]), "+r"(r[1][2]), "+r"(r[1][3]), "+r"(r[1][4]), "+r"(r[1][5]), "+r"(r[1][6]), "+r"(r[1][7]), "+r"(r[1][8]), "+r"(r[1][9]), "+r"(r[1][10]), "+r"(r[1][11]), "+r"(r[1][12]), "+r"(r[1][13]), "+r"(r[1][14]), "+r"(r[1][15])
                 :
                 : "memory");
}

// Waits for this thread's outstanding TMEM loads into r[0..63].
__device__ __forceinline__ void tmem_wait_ld64(uint32_t (&r)[64]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31]), "+r"(r[32]), "+r"(r[33]), "+r"(r[34]), "+r"(r[35]), "+r"(r[36]), "+r"(r[37]), "+r"(r[38]), "+r"(r[39]), "+r"(r[40]), "+r"(r[41]), "+r"(r[42]), "+r"(r[43]), "+r"(r[44]), "+r"(r[45]), "+r"(r[46]), "+r"(r[47]), "+r"(r[48]), "+r"(r[49]), "+r"(r[50]), "+r"(r[51]), "+r"(r[52]), "+r"(r[53]), "+r"(r[54]), "+r"(r[55]), "+r"(r[56]), "+r"(r[57]), "+r"(r[58]), "+r"(r[59]), "+r"(r[60]), "+r"(r[61]), "+r"(r[62]), "+r"(r[63])
                 :
                 : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format) for a K-major operand in
// the 128-byte swizzle layout: rows of 128 bytes, groups of 8 rows (1024 B)
// one after another, and within a group the 16-byte chunk c of row r stored
// at chunk position c ^ r.  The swizzle is applied to absolute shared-memory
// address bits (chunk bits 4-6 XOR row bits 7-9), so with the data written
// the same way and the ring 1024-byte aligned, `addr` may start at any
// 128-byte row -- a tap's shifted view of the frame window -- and at any
// 32-byte K step inside a row, with the base-offset field left at 0.
// (Setting that field to the row phase instead gives wrong results on
// sm_103a: checked against the oracle.)
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr) {
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)1 << 16;             // leading byte offset: unused for swizzled K-major
    d |= (uint64_t)(1024 >> 4) << 32;   // stride byte offset: next group of 8 rows
    d |= (uint64_t)1 << 46;             // descriptor version
    d |= (uint64_t)2 << 61;             // SWIZZLE_128B, base offset 0
    return d;
}

// Shared-memory matrix descriptor for an MN-major operand in the 128-byte
// swizzle layout: atoms of 8 K rows x 128 bytes (64 16-bit MN elements), the
// 16-byte chunk c of row r at chunk position c ^ r; lbo = bytes from one
// 64-element MN atom to the next, sbo = bytes from one 8-row K group to the
// next.
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// ----------------------------------------------------------- bounded waits
__device__ __forceinline__ bool abort_raised(Shared &sh) {
    return *reinterpret_cast<volatile int *>(&sh.abort_flag) != 0;
}

__device__ __noinline__ bool wait_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                       Shared &sh, bool honour_abort) {
    const uint64_t t0 = global_ns();
    // Backstop in case the timer does not advance: each poll takes well over
    // 16 ns, so this many polls outlast the time limit.
    const uint64_t max_spins = limit_ns / 16 + (1u << 20);
    for (uint64_t spin = 1;; ++spin) {
        if (mbar_try_wait(bar, parity)) return true;
        if (honour_abort && abort_raised(sh)) return false;
        if (((spin & 31u) == 0 && global_ns() - t0 > limit_ns) || spin > max_spins) {
            *reinterpret_cast<volatile int *>(&sh.abort_flag) = 1;
            atomicOr(&g_dgrad_error_word, 1u);
            return false;
        }
    }
}

// One thread waits; false means the CTA is aborting.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const TcParams &p,
                                         Shared &sh) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, p.wait_limit_ns, sh, true);
}

// Whole warp: every lane polls the barrier (no divergent branch around a lone
// polling lane) and one vote gives the warp a single verdict, also when the
// wait runs out.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const TcParams &p,
                                              Shared &sh, int lane) {
    (void)lane;
    const bool ok = wait_bar(bar, parity, p, sh);
    return __all_sync(0xffffffffu, ok) != 0;
}

// Waits that must end even while aborting (copies / MMAs already in flight).
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, const TcParams &p,
                                           Shared &sh) {
    if (mbar_try_wait(bar, parity)) return;
    wait_slow(bar, parity, p.wait_limit_ns, sh, false);
}

// ------------------------------------------------------------ tile decode
struct Tile {
    int phase, pt, mt;  // phase, 256-position tile, input-channel tile
};

// V: the kernel variant; only the general mode has interleaved phases.
template <int V = kVarGeneral>
__device__ __forceinline__ Tile decode_tile(const TcParams &p, int64_t t) {
    if (is_general(V) && p.interleave) {  // (position tile, phase, channel tile), phases side by side
        const int per = p.n_phases * p.n_mtiles;
        Tile r;
        r.pt = (int)(t / per);
        const int rem = (int)(t - (int64_t)r.pt * per);
        r.phase = rem / p.n_mtiles;
        r.mt = rem - r.phase * p.n_mtiles;
        return r;
    }
    int ph = 0;
    while (ph + 1 < p.n_phases && t >= p.ph[ph + 1].tile_begin) ++ph;
    const int64_t local = t - p.ph[ph].tile_begin;
    Tile r;
    r.phase = ph;
    r.pt = (int)(local / p.n_mtiles);
    r.mt = (int)(local - (int64_t)r.pt * p.n_mtiles);
    return r;
}

// First frame position of a position tile, and how many positions it owns:
// whole frame rows (stride 1) or tile_p consecutive positions.
__device__ __forceinline__ int tile_start(const TcParams &p, const PhaseDesc &d, int pt) {
    if (p.rows_per_tile > 0) {
        const int tpi = (d.Hr + p.rows_per_tile - 1) / p.rows_per_tile;  // tiles per image
        const int n = pt / tpi, g = pt - n * tpi;
        return (n * d.R + g * p.rows_per_tile) * d.X;
    }
    return pt * p.tile_p;
}

// The last row tile of an image owns only the rows left in it: positions past
// them continue into the next image's frame, which that image's own tiles
// write.
__device__ __forceinline__ int tile_own(const TcParams &p, const PhaseDesc &d, int pt) {
    if (p.rows_per_tile <= 0) return p.tile_p;
    const int tpi = (d.Hr + p.rows_per_tile - 1) / p.rows_per_tile;
    const int left = d.Hr - (pt % tpi) * p.rows_per_tile;
    return (left < p.rows_per_tile ? left : p.rows_per_tile) * d.X;
}

// This CTA's tiles: groups of tile_group consecutive tiles, the groups dealt
// round-robin over the grid (tile_group = 1: blockIdx.x, + gridDim.x, ...).
// Only the pair variant (V) takes groups of more than one tile.
template <int V = kVarGeneral>
__device__ __forceinline__ int64_t first_tile(const TcParams &p) {
    if constexpr (V != kVarPair && V != kVarGeneral) return (int64_t)blockIdx.x;
    return (int64_t)blockIdx.x * p.tile_group;
}
template <int V = kVarGeneral>
__device__ __forceinline__ int64_t next_tile(const TcParams &p, int64_t t) {
    if constexpr (V != kVarPair && V != kVarGeneral) return t + gridDim.x;
    if (p.tile_group == 1) return t + gridDim.x;
    return (t + 1) % p.tile_group ? t + 1 : t + 1 + (int64_t)(gridDim.x - 1) * p.tile_group;
}

// Byte offset, inside the packed weights, of (phase, ci tile, channel chunk).
__device__ __forceinline__ int64_t w_block_off(const TcParams &p, const PhaseDesc &d, int mt,
                                               int cc) {
    return d.pack_off + ((int64_t)mt * p.n_cchunks + cc) * (d.Jh * d.Jw) * p.w_unit_bytes;
}

// ------------------------------------------------------------------ roles
// First grad_out row of a whole-row tile's window, and its image.
__device__ __forceinline__ void row_tile_origin(const TcParams &p, const PhaseDesc &d, int pt,
                                                int &n, int &u_first) {
    const int tpi = (d.Hr + p.rows_per_tile - 1) / p.rows_per_tile;
    n = pt / tpi;
    u_first = (pt - n * tpi) * p.rows_per_tile - (d.Jh - 1) + d.qh;
}

// First grad_out row held by a raw slice whose window starts at row
// u_first: the window's own first row (tiled mode), that row rounded down to
// a multiple of raw_rowg (the copy must start 16-byte aligned), or row 0
// (planes mode: whole planes).
__device__ __forceinline__ int raw_row_origin(const TcParams &p, int u_first) {
    if (p.raw_mode == kRawPlanes) return 0;
    const int g = p.raw_rowg;
    if (g > 1) return u_first >= 0 ? u_first / g * g : -((-u_first + g - 1) / g) * g;
    return u_first;
}

// 1-D bulk prefetch of [src, src + bytes) into L2.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// The grad_out rows [r0, r1) of a rows-mode raw slice that lie inside the
// grid (r1 <= r0: none).
__device__ __forceinline__ void raw_rows_inside(const TcParams &p, int u_lo, int &r0, int &r1) {
    r0 = u_lo < 0 ? 0 : u_lo;
    r1 = u_lo + p.raw_br < p.OH ? u_lo + p.raw_br : p.OH;
}

// grad_out channels of the raw slice that starts at channel c0 (0 when c0 is
// past the last channel: slices come in whole channel chunks).
__device__ __forceinline__ int raw_slice_channels(const TcParams &p, int c0) {
    const int left = p.Co - c0;
    return left <= 0 ? 0 : (left < p.raw_cs ? left : p.raw_cs);
}

// Loads one raw slice -- raw_cs channels from c0 of image n, the window that
// starts at grad_out row u_first -- into shared memory at dst, completing on
// bar.  Tiled mode: one TMA box (rows and channels outside grad_out
// zero-filled).  Rows / planes modes: 1-D bulk copies of the rows inside the
// grid and the channels below Co; the gather never reads the rest.
__device__ __noinline__ void issue_raw_slice_bulk(const TcParams &p, uint32_t dst, int u_first,
                                                  int c0, int n, uint32_t bar);

__device__ __forceinline__ void issue_raw_slice(const TcParams &p, uint32_t dst, int u_first, int c0,
                                                int n, uint32_t bar) {
    if (p.raw_mode == kRawTiled) {  // box rows of raw_rowg grad_out rows
        mbar_arrive_expect_tx(bar, (uint32_t)(p.raw_cs * p.raw_br * p.raw_bw * p.esize));
        tma_load_4d(dst, &p.in_map, p.raw_x0, raw_row_origin(p, u_first) / p.raw_rowg, c0, n, bar);
        return;
    }
    issue_raw_slice_bulk(p, dst, u_first, c0, n, bar);
}

// The 1-D bulk-copy modes of issue_raw_slice.
__device__ __noinline__ void issue_raw_slice_bulk(const TcParams &p, uint32_t dst, int u_first,
                                                  int c0, int n, uint32_t bar) {
    const int64_t plane = (int64_t)p.OH * p.OW * p.esize;
    const uint8_t *img = static_cast<const uint8_t *>(p.grad_out) + (int64_t)n * p.Co * plane;
    const int chans = raw_slice_channels(p, c0);
    if (p.raw_mode == kRawPlanes) {
        const uint32_t bytes = (uint32_t)(chans * plane);
        mbar_arrive_expect_tx(bar, bytes);
        if (bytes) bulk_g2s(dst, img + (int64_t)c0 * plane, bytes, bar);
        return;
    }
    const int u_lo = raw_row_origin(p, u_first);
    int r0, r1;
    raw_rows_inside(p, u_lo, r0, r1);
    const uint32_t row_bytes = (uint32_t)(p.OW * p.esize);
    const uint32_t bytes = r1 > r0 ? (uint32_t)(r1 - r0) * row_bytes : 0u;
    mbar_arrive_expect_tx(bar, bytes * (uint32_t)chans);
    if (bytes == 0 || chans == 0) return;
    const uint32_t ch_bytes = row_bytes * (uint32_t)p.raw_br;
    const uint8_t *src = img + (int64_t)c0 * plane + (int64_t)r0 * row_bytes;
    const uint32_t d0 = dst + (uint32_t)(r0 - u_lo) * row_bytes;
    for (int c = 0; c < chans; ++c)
        bulk_g2s(d0 + (uint32_t)c * ch_bytes, src + (int64_t)c * plane, bytes, bar);
}

// L2 prefetch of one raw slice (same footprint as issue_raw_slice).
__device__ __noinline__ void prefetch_raw_slice(const TcParams &p, int u_first, int c0, int n) {
    if (p.raw_mode == kRawTiled) {
        tma_prefetch_4d(&p.in_map, p.raw_x0, raw_row_origin(p, u_first) / p.raw_rowg, c0, n);
        return;
    }
    const int64_t plane = (int64_t)p.OH * p.OW * p.esize;
    const uint8_t *img = static_cast<const uint8_t *>(p.grad_out) + (int64_t)n * p.Co * plane;
    const int chans = raw_slice_channels(p, c0);
    if (chans == 0) return;
    if (p.raw_mode == kRawPlanes) {
        bulk_prefetch_l2(img + (int64_t)c0 * plane, (uint32_t)(chans * plane));
        return;
    }
    int r0, r1;
    raw_rows_inside(p, raw_row_origin(p, u_first), r0, r1);
    if (r1 <= r0) return;
    const int64_t row_bytes = (int64_t)p.OW * p.esize;
    for (int c = 0; c < chans; ++c)
        bulk_prefetch_l2(img + (int64_t)(c0 + c) * plane + r0 * row_bytes,
                         (uint32_t)((r1 - r0) * row_bytes));
}

// Bulk copies of the resident packed weights, completing on w_full (none
// when the epilogue warps pack them: w_raw).
__device__ void issue_weights(const TcParams &p, Shared &sh, uint32_t w_base) {
    if (p.w_raw) return;
    const uint8_t *src = static_cast<const uint8_t *>(p.packed);
    const uint32_t bar = smem_u32(&sh.w_full);
    mbar_arrive_expect_tx(bar, (uint32_t)p.packed_bytes);
    for (int64_t off = 0; off < p.packed_bytes; off += 32768) {
        const int64_t left = p.packed_bytes - off;
        bulk_g2s(w_base + (uint32_t)off, src + off, (uint32_t)(left < 32768 ? left : 32768), bar);
    }
}

// Resident weights packed in the kernel (w_raw: p.packed is the weight tensor
// [Co][Ci][kH][kW], 16-bit, one stride-1 phase, so tap (j, i) is (kh, kw)).
// Threads tid < nt write the packed image that issue_weights would copy:
// per (Ci tile mt, channel chunk cc, tap j, tap i) m_tile rows ci of 128
// bytes (64 consecutive co), 16-byte chunk c of row r at chunk slot c ^ (r & 7),
// zero for ci >= Ci and co >= Co.  With 16-byte aligned weight rows each item
// is 8 co rows x one 16-byte column of the [Co][Ci*kH*kW] matrix: eight vector
// loads, an 8x8 transpose of 16-bit values in registers, and eight 16-byte
// stores, one per (ci, tap) of the column.  Otherwise every 16-byte chunk of
// the image takes eight scalar loads.  The writes are made visible to the
// tensor core (async proxy) before each warp's arrival on w_full.
__device__ void pack_resident_weights(const TcParams &p, Shared &sh, uint32_t w_base, int tid,
                                      int nt) {
    const uint16_t *w = static_cast<const uint16_t *>(p.packed);
    const PhaseDesc &d = p.ph[0];
    const int Ci = p.Ci, Co = p.Co, KK = d.Jh * d.Jw, kW = d.Jw;
    const int64_t row_elems = (int64_t)Ci * KK;  // elements per co row of the weight tensor
    const uint32_t base = w_base + (uint32_t)d.pack_off;
    // Byte offset of 16-byte chunk `chunk` (64 co per chunk row) of (ci, tap, cc).
    auto slot_off = [&](int ci, int t, int cc, int chunk) -> uint32_t {
        const int mt = ci / p.m_tile, row = ci - mt * p.m_tile;
        const int64_t r = (((int64_t)(mt * p.n_cchunks + cc) * KK + t) * p.m_tile + row);
        return (uint32_t)(r * 128 + ((chunk ^ (row & 7)) << 4));
    };
    const bool vec = (reinterpret_cast<uintptr_t>(w) & 15u) == 0 && row_elems % 8 == 0;
    if (vec) {
        const int cols = (int)(row_elems / 8);  // 16-byte columns per co row
        const int total = p.n_cchunks * 8 * cols;  // co groups of 8 (whole chunks) x columns
        const int mshift = p.m_tile == 128 ? 7 : 6;
        auto load = [&](uint4 (&v)[8], int it) {
            const int g8 = it / cols, c = it - g8 * cols;
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int co = g8 * 8 + e;
                v[e] = co < Co ? __ldg(reinterpret_cast<const uint4 *>(w + (int64_t)co * row_elems) + c)
                               : make_uint4(0u, 0u, 0u, 0u);
            }
        };
        // Items dealt round-robin; the next item's loads are in flight while
        // this one is transposed and stored.  Each CTA starts at its own
        // offset (the item order rotated by the CTA index), so the CTAs' first
        // reads of the usually cold weights ask for different lines.
        const int rot = (int)(((int64_t)blockIdx.x * total) / gridDim.x);
        auto item = [&](int i) { return i + rot < total ? i + rot : i + rot - total; };
        uint4 cur[8];
        if (tid < total) load(cur, item(tid));
        for (int i = tid; i < total; i += nt) {
            uint4 nxt[8];
            if (i + nt < total) load(nxt, item(i + nt));
            const int it = item(i);
            const int g8 = it / cols, c = it - g8 * cols;
            const int cc = g8 >> 3, chunk = g8 & 7;
            int ci = (c * 8) / KK, t = c * 8 - ci * KK;  // (ci, tap) of element 0 of the column
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                // Element k of each co row: the halves of word k / 2.
                const uint32_t sel = (k & 1) ? 0x7632u : 0x5410u;
                auto word = [&](const uint4 &u) -> uint32_t {
                    const int q = k >> 1;
                    return q == 0 ? u.x : q == 1 ? u.y : q == 2 ? u.z : u.w;
                };
                const uint32_t o0 = __byte_perm(word(cur[0]), word(cur[1]), sel);
                const uint32_t o1 = __byte_perm(word(cur[2]), word(cur[3]), sel);
                const uint32_t o2 = __byte_perm(word(cur[4]), word(cur[5]), sel);
                const uint32_t o3 = __byte_perm(word(cur[6]), word(cur[7]), sel);
                const int mt = ci >> mshift, row = ci & (p.m_tile - 1);
                const uint32_t r = (uint32_t)(((mt * p.n_cchunks + cc) * KK + t) * p.m_tile + row);
                st_shared_v4(base + r * 128u + (uint32_t)((chunk ^ (row & 7)) << 4), o0, o1, o2, o3);
                if (++t == KK) {
                    t = 0;
                    ++ci;
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) cur[e] = nxt[e];
        }
        // Rows of the last Ci tile past Ci: zero.
        const int pad0 = Ci, pad1 = p.n_mtiles * p.m_tile;
        const int per_row = p.n_cchunks * KK * 8;  // 16-byte chunks of one ci over (cc, tap)
        for (int it = tid; it < (pad1 - pad0) * per_row; it += nt) {
            const int ci = pad0 + it / per_row;
            int r = it % per_row;
            const int chunk = r & 7;
            r >>= 3;
            const int t = r % KK, cc = r / KK;
            st_shared_v4(base + slot_off(ci, t, cc, chunk), 0u, 0u, 0u, 0u);
        }
    } else {
        const int64_t chunks = p.packed_bytes / 16;
        for (int64_t it = tid; it < chunks; it += nt) {
            int64_t r = it;
            const int slot = (int)(r & 7); r >>= 3;
            const int row = (int)(r % p.m_tile); r /= p.m_tile;
            const int t = (int)(r % KK); r /= KK;
            const int cc = (int)(r % p.n_cchunks);
            const int mt = (int)(r / p.n_cchunks);
            const int ci = mt * p.m_tile + row, chunk = slot ^ (row & 7);
            const int kh = t / kW, kw = t - kh * kW;
            uint32_t o[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
                uint32_t lo = 0, hi = 0;
                const int co = cc * 64 + chunk * 8 + 2 * e2;
                if (ci < Ci && co < Co)
                    lo = w[(((int64_t)co * Ci + ci) * d.Jh + kh) * kW + kw];
                if (ci < Ci && co + 1 < Co)
                    hi = w[(((int64_t)(co + 1) * Ci + ci) * d.Jh + kh) * kW + kw];
                o[e2] = lo | (hi << 16);
            }
            st_shared_v4(base + (uint32_t)(it * 16), o[0], o[1], o[2], o[3]);
        }
    }
    fence_proxy_async();
    __syncwarp();
    if ((tid & 31) == 0) mbar_arrive(smem_u32(&sh.w_full));
}

// L2 prefetch of every raw slice of tile t (if it exists): the ring's TMA
// loads of that tile then hit L2.
constexpr int kRawLookahead = 2;  // general mode: tiles of this CTA prefetched ahead
template <int V>
__device__ void prefetch_raw_tile(const TcParams &p, int64_t t) {
    if (t >= p.total_tiles || (is_general(V) && p.pair_rw && (t & 1))) return;
    const Tile ti = decode_tile<V>(p, t);
    const PhaseDesc &d = p.ph[ti.phase];
    if (d.Jh == 0 || ti.mt != 0) return;  // channel tiles share the window
    int n, u_first;
    row_tile_origin(p, d, ti.pt, n, u_first);
    const int slices = p.kc / p.raw_cs;
    for (int cc = 0; cc < p.n_cchunks; ++cc)
        for (int sl = 0; sl < slices; ++sl) {
            if constexpr (!is_general(V))  // 64-wide frame / positions-on-M: plain tiled map
                tma_prefetch_4d(&p.in_map, p.raw_x0, u_first, cc * p.kc + sl * p.raw_cs, n);
            else
                prefetch_raw_slice(p, u_first, cc * p.kc + sl * p.raw_cs, n);
        }
}

// issue_raw_slice for the kernel variant V: the 64-wide frame and
// positions-on-M always load through the plain tiled map (kept lean: the
// producer's time per slice sits on the raw ring's turnaround).
template <int V>
__device__ __forceinline__ void issue_raw(const TcParams &p, uint32_t dst, int u_first, int c0,
                                          int n, uint32_t bar) {
    if constexpr (!is_general(V)) {
        mbar_arrive_expect_tx(bar, (uint32_t)(p.raw_cs * p.raw_br * p.raw_bw * p.esize));
        tma_load_4d(dst, &p.in_map, p.raw_x0, u_first, c0, n, bar);
    } else {
        issue_raw_slice(p, dst, u_first, c0, n, bar);
    }
}

// TMA gather producer (warp 9, lane 0): for every tile and channel chunk of
// this CTA, the raw grad_out slices of the tile's window -- raw_cs channels x
// raw_br rows x raw_bw columns from column raw_x0 -- into the raw ring.  Rows
// and columns outside grad_out are zero-filled by the TMA unit.  The resident
// weights go out first (bulk copies; none when the epilogue warps pack them in
// shared memory), then the first tile's slices, then slices into the remaining
// free slots.  Once those are all queued and the first tile's last
// slice has landed (earlier, prefetches would compete with it for DRAM), the
// L2 prefetch starts: general mode (a ring shorter than a tile) the next
// kRawLookahead tiles, then each later tile the one kRawLookahead after it;
// positions-on-M mode (the ring holds a whole tile) the tile after the ring's,
// then at each tile's end the next one.
template <int V>
__device__ void raw_producer(const TcParams &p, Shared &sh, uint32_t raw_base, uint32_t w_base,
                             uint32_t early_base) {
    const int slices = p.kc / p.raw_cs;
    const int64_t per_tile = (int64_t)slices * p.n_cchunks;
    const int64_t fill = p.raw_early + p.raw_nr;  // slices that need no free slot
    int slot = 0;
    uint32_t phase = 0;
    int64_t issued = 0;  // slices, parked ones included
    bool aborted = false, weights_issued = false, prefetching = false;
    // This thread reaches here before the grid dependency wait (the setup
    // below is cold code, run while the previous kernel finishes) and waits
    // right before its first global-memory access.
    bool waited = false;
    for (int64_t t = first_tile<V>(p); t < p.total_tiles && !aborted; t = next_tile<V>(p, t)) {
        if (is_general(V) && p.pair_rw && (t & 1)) continue;  // a pair shares its first tile's window
        const Tile ti = decode_tile<V>(p, t);
        const PhaseDesc &d = p.ph[ti.phase];
        if (d.Jh == 0) continue;
        int n, u_first;
        row_tile_origin(p, d, ti.pt, n, u_first);
        for (int cc = 0; cc < p.n_cchunks && !aborted; ++cc) {
            for (int sl = 0; sl < slices; ++sl) {
                // The weights first: every CTA reads the same packed weights,
                // so they mostly come from L2 while the first slices' DRAM reads
                // are in flight (issue_weights does nothing when the epilogue
                // warps pack them: w_raw).
                if (!weights_issued) {
                    if (!waited) {
                        grid_dependency_wait();
                        waited = true;
                    }
                    issue_weights(p, sh, w_base);
                    weights_issued = true;
                }
                // Once every free slot is filled and the first tile's last
                // slice has landed, later tiles go to L2 ahead of the ring.
                if (weights_issued && !prefetching && issued == fill) {
                    const int64_t last = (per_tile < fill ? per_tile : fill) - 1;
                    const int64_t j = last - p.raw_early;
                    const bool ok = last < p.raw_early
                                        ? wait_bar(smem_u32(&sh.full_early[last]), 0, p, sh)
                                        : wait_bar(smem_u32(&sh.full_raw[j % p.raw_nr]),
                                                   (uint32_t)((j / p.raw_nr) & 1), p, sh);
                    if (!ok) {
                        aborted = true;
                        break;
                    }
                    // From the tile this slice belongs to: kRawLookahead tiles
                    // beyond it (general) or itself (positions-on-M).
                    prefetching = true;
                    int64_t ahead = t;
                    for (int k = 0; k <= (p.pos_m ? 0 : kRawLookahead); ++k, ahead = next_tile<V>(p, ahead))
                        prefetch_raw_tile<V>(p, ahead);
                } else if (!p.pos_m && prefetching && cc == 0 && sl == 0) {
                    int64_t ahead = t;
                    for (int k = 0; k < kRawLookahead; ++k) ahead = next_tile<V>(p, ahead);
                    prefetch_raw_tile<V>(p, ahead);
                }
                if (!waited) {
                    grid_dependency_wait();
                    waited = true;
                }
                if (issued < p.raw_early) {  // parked in G stage 1: no slot to wait for
                    issue_raw<V>(p, early_base + (uint32_t)issued * p.raw_slice_bytes, u_first,
                                    cc * p.kc + sl * p.raw_cs, n, smem_u32(&sh.full_early[issued]));
                    ++issued;
                    continue;
                }
                if (!wait_bar(smem_u32(&sh.empty_raw[slot]), phase ^ 1u, p, sh)) {
                    aborted = true;
                    break;
                }
                issue_raw<V>(p, raw_base + (uint32_t)slot * p.raw_slice_bytes, u_first,
                                cc * p.kc + sl * p.raw_cs, n, smem_u32(&sh.full_raw[slot]));
                ++issued;
                if (++slot == p.raw_nr) {
                    slot = 0;
                    phase ^= 1u;
                }
            }
        }
        // Positions-on-M mode (the ring holds a whole tile): all of this
        // tile's slices are queued, the next tile's go to L2.
        if (p.pos_m && prefetching && !aborted) prefetch_raw_tile<V>(p, next_tile<V>(p, t));
    }
    if (!waited) grid_dependency_wait();
    if (!weights_issued) issue_weights(p, sh, w_base);  // fewer slices than free slots
    if (aborted) {
        const int64_t parked = issued < p.raw_early ? issued : p.raw_early;
        for (int64_t k = 0; k < parked; ++k) wait_drain(smem_u32(&sh.full_early[k]), 0, p, sh);
        const int64_t ring = issued - parked;
        const int64_t k_end = ring < p.raw_nr ? ring : p.raw_nr;
        for (int64_t k = 0; k < k_end; ++k) {
            const int64_t q = ring - 1 - k;
            wait_drain(smem_u32(&sh.full_raw[q % p.raw_nr]), (uint32_t)((q / p.raw_nr) & 1), p, sh);
        }
    }
}

// A walk over this CTA's tiles (first_tile, next_tile, ...) that skips
// phases no tap reaches.  Each tile is decoded once, when the walk reaches it,
// so the per-slice and per-stage work of the producer is a few additions.
struct TileWalk {
    int64_t t;
    const PhaseDesc *d;
    int mt, n, u_first;
};

__device__ __forceinline__ bool walk_load(const TcParams &p, TileWalk &w) {
    for (; w.t < p.total_tiles; w.t = next_tile(p, w.t)) {
        if (p.pair_rw && (w.t & 1)) continue;  // a pair is walked at its first tile
        const Tile ti = decode_tile(p, w.t);
        const PhaseDesc &d = p.ph[ti.phase];
        if (d.Jh == 0) continue;
        w.d = &d;
        w.mt = ti.mt;
        row_tile_origin(p, d, ti.pt, w.n, w.u_first);
        return true;
    }
    return false;
}

// Producer for streamed weights together with the raw-slice gather (warp 9,
// lane 0): two independent rings filled in the order the consumers drain
// them -- raw slices for each tile / channel chunk / slice, and weight stages
// for each tile / channel chunk / tap group -- by polling both "empty"
// barriers without blocking, so a full ring never holds up the other.  Gives
// up (abort flag, error word) when neither ring makes progress within the
// wait limit, then drains the copies still in flight.
__device__ __noinline__ void raw_w_producer(const TcParams &p, Shared &sh, uint32_t raw_base, uint32_t w_base) {
    const uint8_t *wsrc = static_cast<const uint8_t *>(p.packed);
    const int slices = p.kc / p.raw_cs;
    const uint32_t w_unit = (uint32_t)p.w_unit_bytes;
    // raw cursor: tile, chunk rcc, slice rsl; ring slot / phase
    TileWalk rw{first_tile(p), nullptr, 0, 0, 0};
    bool r_live = walk_load(p, rw);
    int rcc = 0, rsl = 0, rslot = 0, rc0 = 0;  // rc0: first channel of the next slice
    uint32_t rph = 0;
    int64_t r_issued = 0;
    // weight cursor: tile (a pair: member wk of it), chunk wcc, first tap wt0;
    // ring stage / phase.  A pair's weights go chunk by chunk, both members'
    // taps of a chunk together, the order the MMA consumes them in.
    TileWalk ww{first_tile(p), nullptr, 0, 0, 0};
    bool w_live = walk_load(p, ww);
    int wcc = 0, wk = 0, wt0 = 0, wstage = 0, wtaps = 0;
    const uint8_t *wblk = nullptr;  // packed weights of (tile, member, chunk wcc)
    if (w_live) {
        wtaps = ww.d->Jh * ww.d->Jw;
        wblk = wsrc + w_block_off(p, *ww.d, ww.mt, 0);
    }
    uint32_t wph = 0;
    int64_t w_issued = 0;
    bool aborted = false;
    uint64_t t_idle = 0, idle_spins = 0;
    const uint64_t max_spins = p.wait_limit_ns / 16 + (1u << 20);  // backstop, as in wait_slow
    while (r_live || w_live) {
        bool progress = false;
        if (r_live && mbar_test_wait(smem_u32(&sh.empty_raw[rslot]), rph ^ 1u)) {
            issue_raw_slice(p, raw_base + (uint32_t)rslot * p.raw_slice_bytes, rw.u_first, rc0, rw.n,
                            smem_u32(&sh.full_raw[rslot]));
            ++r_issued;
            if (++rslot == p.raw_nr) {
                rslot = 0;
                rph ^= 1u;
            }
            rc0 += p.raw_cs;
            if (++rsl == slices) {
                rsl = 0;
                if (++rcc == p.n_cchunks) {
                    rcc = 0;
                    rc0 = 0;
                    rw.t = next_tile(p, rw.t);
                    r_live = walk_load(p, rw);
                }
            }
            progress = true;
        }
        if (w_live && mbar_test_wait(smem_u32(&sh.empty_w[wstage]), wph ^ 1u)) {
            const int ng = wtaps - wt0 < p.taps_per_w ? wtaps - wt0 : p.taps_per_w;
            const uint32_t bytes = (uint32_t)ng * w_unit;
            const uint32_t full = smem_u32(&sh.full_w[wstage]);
            mbar_arrive_expect_tx(full, bytes);
            bulk_g2s(w_base + (uint32_t)wstage * p.w_stage_bytes, wblk + (size_t)wt0 * w_unit, bytes, full);
            ++w_issued;
            if (++wstage == p.nw) {
                wstage = 0;
                wph ^= 1u;
            }
            wt0 += p.taps_per_w;
            if (wt0 >= wtaps) {
                wt0 = 0;
                if (p.pair_rw && wk == 0) {
                    wk = 1;  // the pair's other column phase, same chunk
                } else {
                    wk = 0;
                    if (++wcc == p.n_cchunks) {
                        wcc = 0;
                        ww.t = next_tile(p, ww.t);
                        w_live = walk_load(p, ww);
                    }
                }
                if (w_live) {
                    const PhaseDesc &dk = ww.d[wk];  // a pair's phases are adjacent in ph[]
                    wtaps = dk.Jh * dk.Jw;
                    wblk = wsrc + w_block_off(p, dk, ww.mt, wcc);
                }
            }
            progress = true;
        }
        if (progress) {
            idle_spins = 0;
            continue;
        }
        if (abort_raised(sh)) {
            aborted = true;
            break;
        }
        if (idle_spins == 0) t_idle = global_ns();
        ++idle_spins;
        __nanosleep(32);  // both rings full: back off instead of hammering the barriers
        if (((idle_spins & 31u) == 0 && global_ns() - t_idle > p.wait_limit_ns) ||
            idle_spins > max_spins) {
            *reinterpret_cast<volatile int *>(&sh.abort_flag) = 1;
            atomicOr(&g_dgrad_error_word, 1u);
            aborted = true;
            break;
        }
    }
    if (aborted) {
        // Let every copy that may still be landing finish before the CTA exits.
        const int64_t rk = r_issued < p.raw_nr ? r_issued : p.raw_nr;
        for (int64_t k = 0; k < rk; ++k) {
            const int64_t q = r_issued - 1 - k;
            wait_drain(smem_u32(&sh.full_raw[q % p.raw_nr]), (uint32_t)((q / p.raw_nr) & 1), p, sh);
        }
        const int64_t wk = w_issued < p.nw ? w_issued : p.nw;
        for (int64_t k = 0; k < wk; ++k) {
            const int64_t q = w_issued - 1 - k;
            wait_drain(smem_u32(&sh.full_w[q % p.nw]), (uint32_t)((q / p.nw) & 1), p, sh);
        }
    }
}

// The two streams of raw_w_producer, each on its own producer warp (lane 0)
// for the variants with two (Roles::w2_warp): raw slices for each tile /
// channel chunk / slice, and weight stages for each tile / channel chunk /
// tap group (a pair: both members' taps of a chunk together), each in the
// order its consumers drain it.  Each gives up on the wait limit (abort flag,
// error word) and then waits for its own copies still in flight.
__device__ __noinline__ void raw_stream_producer(const TcParams &p, Shared &sh, uint32_t raw_base) {
    const int slices = p.kc / p.raw_cs;
    TileWalk rw{first_tile(p), nullptr, 0, 0, 0};
    bool live = walk_load(p, rw);
    int rcc = 0, rsl = 0, rc0 = 0, slot = 0;
    uint32_t ph = 0;
    int64_t issued = 0;
    bool aborted = false;
    while (live) {
        if (!wait_bar(smem_u32(&sh.empty_raw[slot]), ph ^ 1u, p, sh)) {
            aborted = true;
            break;
        }
        issue_raw_slice(p, raw_base + (uint32_t)slot * p.raw_slice_bytes, rw.u_first, rc0, rw.n,
                        smem_u32(&sh.full_raw[slot]));
        ++issued;
        if (++slot == p.raw_nr) {
            slot = 0;
            ph ^= 1u;
        }
        rc0 += p.raw_cs;
        if (++rsl == slices) {
            rsl = 0;
            if (++rcc == p.n_cchunks) {
                rcc = 0;
                rc0 = 0;
                rw.t = next_tile(p, rw.t);
                live = walk_load(p, rw);
            }
        }
    }
    if (aborted) {
        const int64_t k_end = issued < p.raw_nr ? issued : p.raw_nr;
        for (int64_t k = 0; k < k_end; ++k) {
            const int64_t q = issued - 1 - k;
            wait_drain(smem_u32(&sh.full_raw[q % p.raw_nr]), (uint32_t)((q / p.raw_nr) & 1), p, sh);
        }
    }
}

__device__ __noinline__ void weight_stream_producer(const TcParams &p, Shared &sh, uint32_t w_base) {
    const uint8_t *wsrc = static_cast<const uint8_t *>(p.packed);
    const uint32_t w_unit = (uint32_t)p.w_unit_bytes;
    TileWalk ww{first_tile(p), nullptr, 0, 0, 0};
    bool live = walk_load(p, ww);
    int wcc = 0, wk = 0, wt0 = 0, wtaps = 0, stage = 0;
    uint32_t ph = 0;
    const uint8_t *wblk = nullptr;  // packed weights of (tile, member, chunk wcc)
    if (live) {
        wtaps = ww.d->Jh * ww.d->Jw;
        wblk = wsrc + w_block_off(p, *ww.d, ww.mt, 0);
    }
    int64_t issued = 0;
    bool aborted = false;
    while (live) {
        if (!wait_bar(smem_u32(&sh.empty_w[stage]), ph ^ 1u, p, sh)) {
            aborted = true;
            break;
        }
        const int ng = wtaps - wt0 < p.taps_per_w ? wtaps - wt0 : p.taps_per_w;
        const uint32_t bytes = (uint32_t)ng * w_unit;
        const uint32_t full = smem_u32(&sh.full_w[stage]);
        mbar_arrive_expect_tx(full, bytes);
        bulk_g2s(w_base + (uint32_t)stage * p.w_stage_bytes, wblk + (size_t)wt0 * w_unit, bytes, full);
        ++issued;
        if (++stage == p.nw) {
            stage = 0;
            ph ^= 1u;
        }
        wt0 += p.taps_per_w;
        if (wt0 >= wtaps) {
            wt0 = 0;
            if (p.pair_rw && wk == 0) {
                wk = 1;  // the pair's other column phase, same chunk
            } else {
                wk = 0;
                if (++wcc == p.n_cchunks) {
                    wcc = 0;
                    ww.t = next_tile(p, ww.t);
                    live = walk_load(p, ww);
                }
            }
            if (live) {
                const PhaseDesc &dk = ww.d[wk];  // a pair's phases are adjacent in ph[]
                wtaps = dk.Jh * dk.Jw;
                wblk = wsrc + w_block_off(p, dk, ww.mt, wcc);
            }
        }
    }
    if (aborted) {
        const int64_t k_end = issued < p.nw ? issued : p.nw;
        for (int64_t k = 0; k < k_end; ++k) {
            const int64_t q = issued - 1 - k;
            wait_drain(smem_u32(&sh.full_w[q % p.nw]), (uint32_t)((q / p.nw) & 1), p, sh);
        }
    }
}

// Warp 9, lane 0: packed weights into shared memory with bulk copies.
template <int V>
__device__ void role_weights(const TcParams &p, Shared &sh, uint32_t w_base, uint32_t raw_base,
                             uint32_t early_base) {
    const uint8_t *src = static_cast<const uint8_t *>(p.packed);
    if constexpr (!is_general(V)) {  // resident weights, raw slices by TMA
        raw_producer<V>(p, sh, raw_base, w_base, early_base);
        wait_drain(smem_u32(&sh.w_full), 0, p, sh);
        return;
    }
    if (p.nw != 0 && p.gather_tma) {
        raw_w_producer(p, sh, raw_base, w_base);
        return;
    }
    if (p.nw == 0) {
        if (p.gather_tma) {
            raw_producer<V>(p, sh, raw_base, w_base, early_base);
        } else {
            issue_weights(p, sh, w_base);
        }
        wait_drain(smem_u32(&sh.w_full), 0, p, sh);  // never leave a copy in flight
        return;
    }
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool aborted = false;
    const int members = p.pair_rw ? 2 : 1;  // a pair: both column phases per chunk
    for (int64_t t = first_tile(p); t < p.total_tiles && !aborted; t = next_tile(p, t)) {
        if (p.pair_rw && (t & 1)) continue;
        const Tile ti = decode_tile(p, t);
        if (p.ph[ti.phase].Jh == 0) continue;
        for (int cc = 0; cc < p.n_cchunks && !aborted; ++cc)
        for (int k = 0; k < members && !aborted; ++k) {
            const PhaseDesc &d = p.ph[ti.phase + k];
            const int taps = d.Jh * d.Jw;
            const uint8_t *blk = src + w_block_off(p, d, ti.mt, cc);
            for (int t0 = 0; t0 < taps; t0 += p.taps_per_w) {
                if (!wait_bar(smem_u32(&sh.empty_w[stage]), phase ^ 1u, p, sh)) {
                    aborted = true;
                    break;
                }
                const int ng = taps - t0 < p.taps_per_w ? taps - t0 : p.taps_per_w;
                const uint32_t bytes = (uint32_t)(ng * p.w_unit_bytes);
                const uint32_t full = smem_u32(&sh.full_w[stage]);
                mbar_arrive_expect_tx(full, bytes);
                bulk_g2s(w_base + (uint32_t)stage * p.w_stage_bytes,
                         blk + (int64_t)t0 * p.w_unit_bytes, bytes, full);
                ++issued;
                if (++stage == p.nw) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }
    if (aborted) {
        // Let every copy that may still be landing finish before the CTA exits.
        const int64_t k_end = issued < p.nw ? issued : p.nw;
        for (int64_t k = 0; k < k_end; ++k) {
            const int64_t q = issued - 1 - k;
            wait_drain(smem_u32(&sh.full_w[q % p.nw]), (uint32_t)((q / p.nw) & 1), p, sh);
        }
    }
}

// Warp 8 (converged; lane 0 issues): tcgen05.mma.  D[ci, pos] (TMEM, 256 columns per
// buffer) += W_tap[ci, co] (A: packed weights) x G[co, pos + shift(tap)]
// (B: the frame window seen from the tap's start row).
template <bool TF32, int V>
__device__ void role_mma(const TcParams &p, Shared &sh, uint32_t g_base, uint32_t w_base,
                         uint32_t tmem) {
    // Paired column phases: both members of a pair (adjacent phases) consume
    // each G stage, into the pair's two accumulators of the TMEM buffer.
    constexpr int kMembers = V == kVarPair ? 2 : 1;
    int gs = 0, ws = 0, acc = 0;
    uint32_t gph = 0, wph = 0, accph = 0;
    bool aborted = false;
    if (p.nw == 0 && !wait_bar(smem_u32(&sh.w_full), 0, p, sh)) aborted = true;
    for (int64_t t = first_tile<V>(p); t < p.total_tiles && !aborted; t = next_tile<V>(p, t)) {
        if (V == kVarPair && (t & 1)) continue;
        const Tile ti = decode_tile<V>(p, t);
        const PhaseDesc &d = p.ph[ti.phase];
        if (d.Jh == 0) continue;
        if (!wait_bar(smem_u32(&sh.acc_empty[acc]), accph ^ 1u, p, sh)) {
            aborted = true;
            break;
        }
        tc_fence_after();
        uint32_t accum[kMembers];
#pragma unroll
        for (int k = 0; k < kMembers; ++k) accum[k] = 0;
        for (int cc = 0; cc < p.n_cchunks; ++cc) {
            if (!wait_bar(smem_u32(&sh.full_g[gs]), gph, p, sh)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const uint32_t g_stage = g_base + (uint32_t)gs * p.g_stage_bytes;
#pragma unroll
            for (int mb = 0; mb < kMembers; ++mb) {
            const PhaseDesc &dk = p.ph[ti.phase + mb];
            const uint32_t d_tmem = tmem + (uint32_t)((acc * kMembers + mb) * p.tile_p);
            const int taps = dk.Jh * dk.Jw;
            uint32_t accumulate = accum[mb];
            const uint32_t w_res = w_base + (uint32_t)w_block_off(p, dk, ti.mt, cc);
            for (int t0 = 0; t0 < taps && !aborted; t0 += p.taps_per_w) {
                const int t1 = taps - t0 < p.taps_per_w ? taps : t0 + p.taps_per_w;
                uint32_t w_grp;
                if (p.nw == 0) {
                    w_grp = w_res + (uint32_t)(t0 * p.w_unit_bytes);
                } else {
                    if (!wait_bar(smem_u32(&sh.full_w[ws]), wph, p, sh)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    w_grp = w_base + (uint32_t)ws * p.w_stage_bytes;
                }
                // Descriptors are linear in the address (start field = addr >> 4,
                // far from overflowing inside shared memory): a tap's view or a
                // 32-byte K step is an add to a base descriptor.
                const uint64_t wd0 = sw128_desc(w_grp);
                // MN-major grad_out: a 16-channel K step is two 8-row groups.
                const bool mn = (V == kVarGeneral || V == kVarMN) && p.mn_b;
                const uint32_t mn_sbo = (uint32_t)p.mn_atoms * 1024u;
                const uint64_t gd0 = mn ? sw128_mn_desc(g_stage, 1024u, mn_sbo)
                                        : sw128_desc(g_stage + (uint32_t)(p.view0 * 128));
                const uint32_t b_kstep = mn ? (2u * mn_sbo) >> 4 : 2u;
                const uint32_t w_step = (uint32_t)(p.w_unit_bytes >> 4);
                int j = t0 / dk.Jw, i = t0 - j * dk.Jw;
                for (int tap = t0; tap < t1; ++tap) {
                    const uint64_t bd = gd0 + (uint64_t)(((dk.Jh - 1 - j) * dk.X + (dk.Jw - 1 - i)) * 8);
                    const uint64_t ad = wd0 + (uint64_t)((tap - t0) * w_step);
#pragma unroll
                    for (int k = 0; k < 4; ++k) {  // four 32-byte K steps per 128-byte row
                        tc_mma<TF32>(d_tmem, ad + 2u * k, bd + (uint64_t)(b_kstep * k), p.idesc, accumulate);
                        accumulate = 1;
                    }
                    if (++i == dk.Jw) {
                        i = 0;
                        ++j;
                    }
                }
                if (p.nw != 0) {
                    tc_commit(smem_u32(&sh.empty_w[ws]));
                    if (++ws == p.nw) {
                        ws = 0;
                        wph ^= 1u;
                    }
                }
            }
            accum[mb] = accumulate;
            }
            if (aborted) break;
            tc_commit(smem_u32(&sh.empty_g[gs]));
            if (++gs == p.ng) {
                gs = 0;
                gph ^= 1u;
            }
        }
        if (aborted) break;
        tc_commit(smem_u32(&sh.acc_full[acc]));
        if (++acc == ((V == kVarPair && p.acc_single) ? 1 : 2)) {
            acc = 0;
            accph ^= 1u;
        }
    }
    // No MMA may still be running when TMEM is released.
    tc_commit(smem_u32(&sh.mma_done));
    wait_drain(smem_u32(&sh.mma_done), 0, p, sh);
}

// Accumulator columns of one stacked-mode M-block: st_n, or st_tw x st_n with
// the column taps on N.
__device__ __forceinline__ int st_cols(const TcParams &p) {
    return p.st_qhalo ? p.st_tw * p.st_n : p.st_n;
}

// Warp 8 (converged; lane 0 issues), stacked-phase mode: D[position, (phase, ci)] (TMEM, st_n
// columns per buffer) += G[position + shift(tap), co] (A: the frame window
// seen from the tap's start row) x W_tap[(phase, ci), co] (B: resident packed
// weights of the chunk and tap).
template <bool TF32>
__device__ void role_mma_stacked(const TcParams &p, Shared &sh, uint32_t g_base, uint32_t w_base,
                                 uint32_t tmem) {
    int gs = 0, ws = 0, acc = 0;
    uint32_t gph = 0, wph = 0, accph = 0;
    bool aborted = p.nw == 0 && !wait_bar(smem_u32(&sh.w_full), 0, p, sh);
    const int X = p.ph[0].X;
    const int taps = p.st_th * p.st_tw;
    const int mblocks = p.st_mblocks;  // 128-position M-blocks of a tile, one accumulator each
    const uint32_t w_step = (uint32_t)(p.w_unit_bytes >> 4);
    const uint32_t ncols = (uint32_t)st_cols(p);
    if (p.st_qhalo) {
        // Column taps on N: for each grad_out chunk and row tap dy, one MMA
        // group per M-block (frame row mb of the tile) with A = the window
        // from frame row mb + dy (row taps are whole 128-element frame rows)
        // and B = the st_tw taps (dy, 0..st_tw-1) of the chunk, st_tw x st_n
        // rows; weights streamed one row tap per stage, or resident.
        for (int64_t t = first_tile<kVarStacked>(p); t < p.total_tiles && !aborted;
             t = next_tile<kVarStacked>(p, t)) {
            if (!wait_bar(smem_u32(&sh.acc_empty[acc]), accph ^ 1u, p, sh)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)acc * (uint32_t)mblocks * ncols;
            uint32_t accumulate = 0;
            for (int cc = 0; cc < p.n_cchunks && !aborted; ++cc) {
                if (!wait_bar(smem_u32(&sh.full_g[gs]), gph, p, sh)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint64_t ad0 = sw128_desc(g_base + (uint32_t)gs * p.g_stage_bytes);
                for (int dy = 0; dy < p.st_th; ++dy) {
                    uint32_t w_grp;  // taps (dy, 0 .. st_tw - 1) of this chunk
                    if (p.nw == 0) {
                        w_grp = w_base + (uint32_t)(cc * taps + dy * p.st_tw) * (uint32_t)p.w_unit_bytes;
                    } else {
                        if (!wait_bar(smem_u32(&sh.full_w[ws]), wph, p, sh)) {
                            aborted = true;
                            break;
                        }
                        tc_fence_after();
                        w_grp = w_base + (uint32_t)ws * p.w_stage_bytes;
                    }
                    const uint64_t bd = sw128_desc(w_grp);
                    for (int mb = 0; mb < mblocks; ++mb) {
                        const uint64_t ad = ad0 + (uint64_t)((mb + dy) * X * 8);  // frame rows of 128 B rows
#pragma unroll
                        for (int k = 0; k < 4; ++k)  // four 32-byte K steps per 128-byte row
                            tc_mma<TF32>(d_tmem + (uint32_t)mb * ncols, ad + 2u * k, bd + 2u * k, p.idesc,
                                         accumulate | (uint32_t)(k > 0));
                    }
                    accumulate = 1;
                    if (p.nw != 0) {
                        tc_commit(smem_u32(&sh.empty_w[ws]));
                        if (++ws == p.nw) {
                            ws = 0;
                            wph ^= 1u;
                        }
                    }
                }
                if (aborted) break;
                tc_commit(smem_u32(&sh.empty_g[gs]));
                if (++gs == p.ng) {
                    gs = 0;
                    gph ^= 1u;
                }
            }
            if (aborted) break;
            tc_commit(smem_u32(&sh.acc_full[acc]));
            if (++acc == 2) {
                acc = 0;
                accph ^= 1u;
            }
        }
        tc_commit(smem_u32(&sh.mma_done));
        wait_drain(smem_u32(&sh.mma_done), 0, p, sh);
        return;
    }
    for (int64_t t = first_tile<kVarStacked>(p); t < p.total_tiles && !aborted;
         t = next_tile<kVarStacked>(p, t)) {
        if (!wait_bar(smem_u32(&sh.acc_empty[acc]), accph ^ 1u, p, sh)) {
            aborted = true;
            break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * mblocks * p.st_n);
        uint32_t accumulate = 0;
        for (int cc = 0; cc < p.n_cchunks && !aborted; ++cc) {
            if (!wait_bar(smem_u32(&sh.full_g[gs]), gph, p, sh)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const uint64_t ad0 = sw128_desc(g_base + (uint32_t)gs * p.g_stage_bytes);
            int dy = 0, dx = 0;
            for (int t0 = 0; t0 < taps && !aborted; t0 += p.taps_per_w) {
                const int t1 = taps - t0 < p.taps_per_w ? taps : t0 + p.taps_per_w;
                uint32_t w_grp;  // weights of taps t0 .. t1 - 1 of this chunk
                if (p.nw == 0) {
                    w_grp = w_base + (uint32_t)(cc * taps + t0) * (uint32_t)p.w_unit_bytes;
                } else {
                    if (!wait_bar(smem_u32(&sh.full_w[ws]), wph, p, sh)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    w_grp = w_base + (uint32_t)ws * p.w_stage_bytes;
                }
                const uint64_t bd0 = sw128_desc(w_grp);
                for (int tap = t0; tap < t1; ++tap) {
                    const uint64_t ad = ad0 + (uint64_t)((dy * X + dx) * 8);  // 128-byte rows, in 16-byte units
                    const uint64_t bd = bd0 + (uint64_t)((tap - t0) * w_step);
                    for (int mb = 0; mb < mblocks; ++mb) {
                        const uint64_t adm = ad + (uint64_t)(mb * 128 * 8);  // the next 128 frame rows
#pragma unroll
                        for (int k = 0; k < 4; ++k)  // four 32-byte K steps per 128-byte row
                            tc_mma<TF32>(d_tmem + (uint32_t)(mb * p.st_n), adm + 2u * k, bd + 2u * k, p.idesc,
                                         accumulate | (uint32_t)(k > 0));
                    }
                    accumulate = 1;
                    if (++dx == p.st_tw) {
                        dx = 0;
                        ++dy;
                    }
                }
                if (p.nw != 0) {
                    tc_commit(smem_u32(&sh.empty_w[ws]));
                    if (++ws == p.nw) {
                        ws = 0;
                        wph ^= 1u;
                    }
                }
            }
            if (aborted) break;
            tc_commit(smem_u32(&sh.empty_g[gs]));
            if (++gs == p.ng) {
                gs = 0;
                gph ^= 1u;
            }
        }
        if (aborted) break;
        tc_commit(smem_u32(&sh.acc_full[acc]));
        if (++acc == 2) {
            acc = 0;
            accph ^= 1u;
        }
    }
    // No MMA may still be running when TMEM is released.
    tc_commit(smem_u32(&sh.mma_done));
    wait_drain(smem_u32(&sh.mma_done), 0, p, sh);
}

// Consumer side of the raw slices (gather warps): the first raw_early come
// from G stage 1, the rest through the ring.  After its last parked slice a
// warp arrives on early_free; a warp waits for it before it first writes
// G stage 1.
struct RawCursor {
    int64_t k = 0;  // slices consumed
    int rs = 0;
    uint32_t rph = 0;
};

__device__ __forceinline__ bool raw_acquire(const TcParams &p, Shared &sh, const RawCursor &c,
                                            uint32_t raw_base, uint32_t early_base, int lane,
                                            uint32_t &addr) {
    if (c.k < p.raw_early) {
        if (!wait_bar_warp(smem_u32(&sh.full_early[c.k]), 0, p, sh, lane)) return false;
        addr = early_base + (uint32_t)c.k * p.raw_slice_bytes;
    } else {
        if (!wait_bar_warp(smem_u32(&sh.full_raw[c.rs]), c.rph, p, sh, lane)) return false;
        addr = raw_base + (uint32_t)c.rs * p.raw_slice_bytes;
    }
    return true;
}

__device__ __forceinline__ void raw_release(const TcParams &p, Shared &sh, RawCursor &c,
                                            int lane) {
    __syncwarp();
    if (c.k < p.raw_early) {
        if (c.k == p.raw_early - 1 && lane == 0) mbar_arrive(smem_u32(&sh.early_free));
    } else {
        if (lane == 0) mbar_arrive(smem_u32(&sh.empty_raw[c.rs]));
        if (++c.rs == p.raw_nr) {
            c.rs = 0;
            c.rph ^= 1u;
        }
    }
    ++c.k;
}

// Before a warp first writes G stage `stage`: stage 1 may still hold parked
// raw slices that other gather warps read.
__device__ __forceinline__ bool stage_writable(const TcParams &p, Shared &sh, int stage,
                                               bool &early_done, int lane) {
    if (stage != 1 || early_done || p.raw_early == 0) return true;
    early_done = true;
    return wait_bar_warp(smem_u32(&sh.early_free), 0, p, sh, lane);
}

// Gather warps, TMA variant: the frame window of each stage is assembled
// from raw slices (raw_cs channels of whole grad_out rows) by a transpose in
// shared memory: frame element h, channel c comes from slice row h / X,
// column (h mod X) + vmin - raw_x0.  Each slice fills raw_cs / E 16-byte
// chunks of every 128-byte window row.  A thread owns the window rows
// h = 32 gw + lane + 32 GW k (GW gather warps); their places in a slice are
// worked out once per tile.
template <int ESIZE, int GW>
__device__ void gather_from_raw(const TcParams &p, Shared &sh, uint32_t g_base,
                                uint32_t raw_base, uint32_t early_base, int gw, int lane) {
    constexpr int E = 16 / ESIZE;  // channels per 16-byte chunk
    constexpr int kStep = GW * 32;
    const int slices = p.kc / p.raw_cs;
    const int groups = p.raw_cs / E;  // 16-byte chunks per slice and window row
    int stage = 0;
    uint32_t phase = 0;
    RawCursor rc;
    bool early_done = false;
    bool withhold = (p.debug_flags & DGRAD_DEBUG_SKIP_ARRIVE) && gw == 0;
    const uint32_t row_bytes = (uint32_t)(p.raw_bw * ESIZE);
    const uint32_t ch_bytes = row_bytes * (uint32_t)p.raw_br;
    const int h0 = gw * 32 + lane;
    const int nrows = h0 < p.hbp ? (p.hbp - 1 - h0) / kStep + 1 : 0;  // <= kMaxGatherRows (plan)
    for (int64_t t = first_tile(p); t < p.total_tiles; t = next_tile(p, t)) {
        if (p.pair_rw && (t & 1)) continue;  // a pair shares its first tile's window
        const Tile ti = decode_tile(p, t);
        const PhaseDesc &d = p.ph[ti.phase];
        if (d.Jh == 0) continue;
        const int X = d.X;
        const int xoff = -(d.Jw - 1) + d.qw - p.raw_x0;  // raw column of frame column 0
        int n_img, u_first;
        row_tile_origin(p, d, ti.pt, n_img, u_first);
        const int roff = u_first - raw_row_origin(p, u_first);  // raw row of frame row 0
        // Byte offset inside a slice of each owned row, or -1 (zero row or
        // column of the frame).
        int src[kMaxGatherRows];
        {
            int rho = h0 / X, x = h0 - rho * X;
            const int drho = kStep / X, dx = kStep - drho * X;
#pragma unroll
            for (int k = 0; k < kMaxGatherRows; ++k) {
                const int u = u_first + rho, xc = frame_column(x, p.st_qhalo) + xoff;
                const bool inside = xc >= 0 && xc < p.raw_bw && u >= 0 && u < p.OH;
                src[k] = inside ? (rho + roff) * (int)row_bytes + xc * ESIZE : -1;
                rho += drho;
                x += dx;
                if (x >= X) {
                    x -= X;
                    ++rho;
                }
            }
        }
        for (int cc = 0; cc < p.n_cchunks; ++cc) {
            if (!wait_bar_warp(smem_u32(&sh.empty_g[stage]), phase ^ 1u, p, sh, lane)) return;
            if (!stage_writable(p, sh, stage, early_done, lane)) return;
            const uint32_t s_base = g_base + (uint32_t)stage * p.g_stage_bytes;
            for (int sl = 0; sl < slices; ++sl) {
                // Channels of this slice inside grad_out (the bulk-copy modes
                // leave the slots of the others stale).
                const int cv = p.Co - (cc * p.kc + sl * p.raw_cs);
                uint32_t raw;
                if (!raw_acquire(p, sh, rc, raw_base, early_base, lane, raw)) return;
#pragma unroll
                for (int k = 0; k < kMaxGatherRows; ++k) {
                    if (k >= nrows) break;
                    const int h = h0 + k * kStep;
                    const uint32_t row = s_base + (uint32_t)h * 128u;
                    const int off = src[k];
                    // Batches of kGB 16-byte chunks: every shared-memory load
                    // of a batch is issued before any of them is used, so the
                    // loads overlap instead of each one waiting on the last.
                    constexpr int kGB = ESIZE == 2 ? 1 : 2;  // 16-bit: one chunk (measured faster on the paired mode)
                    for (int j0 = 0; j0 < groups; j0 += kGB) {
                        uint32_t v[kGB][E];  // raw elements: 16-bit values or float32 bits
#pragma unroll
                        for (int jj = 0; jj < kGB; ++jj) {
                            if (j0 + jj < groups && off >= 0) {
                                const uint32_t a = raw + (uint32_t)off + (uint32_t)((j0 + jj) * E) * ch_bytes;
#pragma unroll
                                for (int e = 0; e < E; ++e) {
                                    if constexpr (ESIZE == 2)
                                        v[jj][e] = ld_shared_u16(a + (uint32_t)e * ch_bytes);
                                    else
                                        v[jj][e] = __float_as_uint(ld_shared_f32(a + (uint32_t)e * ch_bytes));
                                }
                            }
                        }
#pragma unroll
                        for (int jj = 0; jj < kGB; ++jj) {
                            const int j = j0 + jj;
                            if (j >= groups) break;
                            uint32_t q[4] = {0u, 0u, 0u, 0u};
                            if (off >= 0) {
#pragma unroll
                                for (int e = 0; e < 4; ++e) {
                                    if constexpr (ESIZE == 2)
                                        q[e] = v[jj][2 * e] | (v[jj][2 * e + 1] << 16);
                                    else
                                        q[e] = to_tf32(v[jj][e]);
                                }
                                const int c0 = j * E;
                                if (c0 + E > cv) {  // ragged last slice: zero the missing channels
#pragma unroll
                                    for (int e = 0; e < 4; ++e) {
                                        constexpr int per = 4 / ESIZE;  // channels per 32-bit word
                                        const int c = c0 + e * per;
                                        if (c >= cv) q[e] = 0u;
                                        else if (per == 2 && c + 1 >= cv) q[e] &= 0xffffu;
                                    }
                                }
                            }
                            st_shared_v4(row + (uint32_t)(((sl * groups + j) ^ (h & 7)) << 4), q[0], q[1],
                                         q[2], q[3]);
                        }
                    }
                }
                raw_release(p, sh, rc, lane);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                if (withhold)
                    withhold = false;  // failure injection: this stage is never signalled
                else
                    mbar_arrive(smem_u32(&sh.full_g[stage]));
            }
            if (++stage == p.ng) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// Gather warps, MN-major operand (1x1 stride-1 tiles of whole images): a raw
// slice holds kc whole channel planes, [c][H*W] with a plane pitch of H*W
// elements; each 16-byte piece (8 consecutive positions of one channel) goes
// to its place in the stage's swizzled MN-major atoms.  Pieces past the end
// of a plane hold whatever follows it: those output columns are never stored.
// Channels past Co are zero.
template <int GW>
__device__ void gather_mn(const TcParams &p, Shared &sh, uint32_t g_base, uint32_t raw_base,
                          uint32_t early_base, int gw, int lane) {
    constexpr int kStep = GW * 32;
    const uint32_t plane = (uint32_t)(p.OH * p.OW) * 2u;  // bytes per channel plane (a multiple of 8)
    const int pieces = p.mn_atoms * 8;                     // 16-byte pieces per channel
    const int items = p.kc * pieces;
    const uint32_t sbo = (uint32_t)p.mn_atoms * 1024u;
    int stage = 0;
    uint32_t phase = 0;
    RawCursor rc;
    bool early_done = false;
    bool withhold = (p.debug_flags & DGRAD_DEBUG_SKIP_ARRIVE) && gw == 0;
    // This thread's first piece (channel c0, piece v0) and the stride between
    // its pieces, in channels and pieces.
    const int i0 = gw * 32 + lane;
    const int c0 = i0 / pieces, v0 = i0 - c0 * pieces;
    const int dc = kStep / pieces, dv = kStep - dc * pieces;
    for (int64_t t = first_tile(p); t < p.total_tiles; t = next_tile(p, t)) {
        for (int cc = 0; cc < p.n_cchunks; ++cc) {
            if (!wait_bar_warp(smem_u32(&sh.empty_g[stage]), phase ^ 1u, p, sh, lane)) return;
            if (!stage_writable(p, sh, stage, early_done, lane)) return;
            const uint32_t s_base = g_base + (uint32_t)stage * p.g_stage_bytes;
            const int cv = p.Co - cc * p.kc;  // channels of this chunk inside grad_out
            uint32_t raw;
            if (!raw_acquire(p, sh, rc, raw_base, early_base, lane, raw)) return;
            // All of this thread's pieces are loaded first, then stored, so the
            // loads overlap one another.
            uint32_t q[kMaxMnPieces][4], dst[kMaxMnPieces];
            int c = c0, v = v0;
#pragma unroll
            for (int k = 0; k < kMaxMnPieces; ++k) {
                q[k][0] = q[k][1] = q[k][2] = q[k][3] = 0u;
                dst[k] = ~0u;
                if (i0 + k * kStep < items) {
                    if (c < cv) {
                        const uint32_t a = raw + (uint32_t)c * plane + (uint32_t)v * 16u;
                        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(q[k][0]), "=r"(q[k][1]) : "r"(a) : "memory");
                        asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(q[k][2]), "=r"(q[k][3]) : "r"(a + 8u) : "memory");
                    }
                    const int r = c & 7;
                    dst[k] = s_base + (uint32_t)(c >> 3) * sbo + (uint32_t)(v >> 3) * 1024u + (uint32_t)r * 128u +
                             (uint32_t)(((v & 7) ^ r) << 4);
                }
                c += dc;
                v += dv;
                if (v >= pieces) {
                    v -= pieces;
                    ++c;
                }
            }
#pragma unroll
            for (int k = 0; k < kMaxMnPieces; ++k)
                if (dst[k] != ~0u) st_shared_v4(dst[k], q[k][0], q[k][1], q[k][2], q[k][3]);
            raw_release(p, sh, rc, lane);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                if (withhold)
                    withhold = false;  // failure injection: this stage is never signalled
                else
                    mbar_arrive(smem_u32(&sh.full_g[stage]));
            }
            if (++stage == p.ng) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// Gather warps: grad_out frame windows into 128-byte swizzled K-major rows
// (one row per frame element, 128 bytes of grad_out channels).
template <int ESIZE, int GW>
__device__ void role_gather(const TcParams &p, Shared &sh, uint32_t g_base, int gw, int lane) {
    const int64_t plane = (int64_t)p.OH * p.OW;
    int stage = 0;
    uint32_t phase = 0;
    bool withhold = (p.debug_flags & DGRAD_DEBUG_SKIP_ARRIVE) && gw == 0;
    for (int64_t t = first_tile(p); t < p.total_tiles; t = next_tile(p, t)) {
        if (p.pair_rw && (t & 1)) continue;  // a pair shares its first tile's window
        const Tile ti = decode_tile(p, t);
        const PhaseDesc &d = p.ph[ti.phase];
        if (d.Jh == 0) continue;
        const int L0 = tile_start(p, d, ti.pt);
        const int img = d.R * d.X;
        for (int cc = 0; cc < p.n_cchunks; ++cc) {
            if (!wait_bar_warp(smem_u32(&sh.empty_g[stage]), phase ^ 1u, p, sh, lane)) return;
            const uint32_t s_base = g_base + (uint32_t)stage * p.g_stage_bytes;
            const int co0 = cc * p.kc;
            const int cleft = p.Co - co0;
            // Rows of this thread in batches of RB: all loads of a batch are
            // issued before any is used, so many are in flight at once.
            constexpr int RB = ESIZE == 4 ? 2 : 1;  // rows per batch (64 registers of loads)
            constexpr int CHUNKS = 8;                // 16-byte chunks per 128-byte row
            constexpr int E = 16 / ESIZE;            // elements per chunk
            for (int h0 = gw * 32 + lane; h0 < p.hbp; h0 += RB * GW * 32) {
                int64_t off[RB];
                int cvalid[RB];
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const int h = h0 + r * GW * 32;
                    const int lam = L0 + h;
                    const int n = lam / img;
                    const int rem = lam - n * img;
                    const int rho = rem / d.X;
                    const int kap = rem - rho * d.X;
                    const int u = rho - (d.Jh - 1) + d.qh;
                    const int v = frame_column(kap, p.st_qhalo) - (d.Jw - 1) + d.qw;
                    const bool ok = h < p.hbp && n < p.N && u >= 0 && u < p.OH && v >= 0 && v < p.OW;
                    cvalid[r] = ok ? (cleft < p.kc ? cleft : p.kc) : 0;
                    off[r] = ok ? ((int64_t)n * p.Co + co0) * plane + (int64_t)u * p.OW + v : 0;
                }
                uint32_t x[RB][CHUNKS * E];  // raw elements: 16-bit values or float32 bits
#pragma unroll
                for (int r = 0; r < RB; ++r) {
#pragma unroll
                    for (int c = 0; c < CHUNKS * E; ++c) {
                        if constexpr (ESIZE == 2)
                            x[r][c] = c < cvalid[r]
                                          ? ldg_u16(static_cast<const unsigned short *>(p.grad_out) + off[r] + c * plane)
                                          : 0u;
                        else
                            x[r][c] = c < cvalid[r]
                                          ? ldg_b32(static_cast<const float *>(p.grad_out) + off[r] + c * plane)
                                          : 0u;
                    }
                }
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const int h = h0 + r * GW * 32;
                    if (h >= p.hbp) break;
                    const uint32_t row = s_base + (uint32_t)h * 128u;
#pragma unroll
                    for (int kc = 0; kc < CHUNKS; ++kc) {
                        uint32_t q[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            if constexpr (ESIZE == 2)
                                q[e] = x[r][kc * 8 + 2 * e] | (x[r][kc * 8 + 2 * e + 1] << 16);
                            else
                                q[e] = to_tf32(x[r][kc * 4 + e]);
                        }
                        st_shared_v4(row + (uint32_t)((kc ^ (h & 7)) << 4), q[0], q[1], q[2], q[3]);
                    }
                }
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                if (withhold)
                    withhold = false;  // failure injection: this stage is never signalled
                else
                    mbar_arrive(smem_u32(&sh.full_g[stage]));
            }
            if (++stage == p.ng) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// A position of the tile walked along the frame: (image, frame row, column).
struct FramePos {
    int n, a, b;
};

__device__ __forceinline__ FramePos frame_pos(const PhaseDesc &d, int lam) {
    const int img = d.R * d.X;
    FramePos f;
    f.n = lam / img;
    const int rem = lam - f.n * img;
    f.a = rem / d.X;
    f.b = rem - f.a * d.X;
    return f;
}

__device__ __forceinline__ void frame_advance(const PhaseDesc &d, FramePos &f, int step) {
    f.b += step;
    while (f.b >= d.X) {
        f.b -= d.X;
        if (++f.a == d.R) {
            f.a = 0;
            ++f.n;
        }
    }
}

// grad_in offset of channel 0 at a frame position, or -1 for frame padding
// and positions past the last image.
__device__ __forceinline__ int64_t out_offset(const TcParams &p, const PhaseDesc &d,
                                              const FramePos &f) {
    if (f.n >= p.N || f.a >= d.Hr || f.b >= d.Wr) return -1;
    return ((int64_t)f.n * p.Ci * p.H + (p.stride * f.a + d.rh)) * p.W + (p.stride * f.b + d.rw);
}

// Warps 0..7: TMEM accumulator -> float32 NCHW grad_in.  Warps q and q + 4
// share TMEM lane quadrant q: rows (input channels) 32q..32q+31 for a 128-row
// tile, or 16q..16q+15 (lanes 0..15 of the quadrant) for a 64-row tile; they
// split the tile's columns (positions) between them ("part" 0 and 1).
//
// Staged epilogue (any shape): a step takes 32 columns (positions); the values
// are turned around through a padded staging block in shared memory (row
// pitch 33 floats: conflict-free both ways) so that each store instruction
// writes 32 consecutive positions of one channel.  Part p takes the 32-column
// chunks whose index has parity p.
template <int ROWS>
__device__ void epilogue_staged(const TcParams &p, const PhaseDesc &d, const Tile &ti,
                                uint32_t taddr, uint32_t st_base, int q, int part, int lane) {
    const int64_t HW = (int64_t)p.H * p.W;
    const int ci_base = ti.mt * p.m_tile + q * ROWS;
    int ci_here = p.Ci - ci_base;  // channels of this warp that exist
    ci_here = ci_here < 0 ? 0 : (ci_here > ROWS ? ROWS : ci_here);
    const int L0 = tile_start(p, d, ti.pt), own = tile_own(p, d, ti.pt);
    FramePos f = frame_pos(d, L0 + part * kEpiChunk + lane);
    const uint32_t st_row = st_base + 4u * kEpiRowFloats * lane;  // row written by this lane
    const uint32_t st_col = st_base + 4u * lane;                  // column read by this lane
    for (int c0 = part * kEpiChunk; c0 < p.tile_p; c0 += 2 * kEpiChunk) {
        uint32_t v[2][16];
        tmem_ld16(taddr + (uint32_t)c0, v[0]);
        tmem_ld16(taddr + (uint32_t)(c0 + 16), v[1]);
        tmem_wait_ld16x2(v);
        if (lane < ROWS) {
#pragma unroll
            for (int e = 0; e < 32; ++e) st_shared_f32(st_row + 4u * e, v[e / 16][e % 16]);
        }
        __syncwarp();
        float val[ROWS];
#pragma unroll
        for (int r = 0; r < ROWS; ++r) val[r] = ld_shared_f32(st_col + 4u * kEpiRowFloats * r);
        __syncwarp();
        const int64_t o = c0 + lane < own ? out_offset(p, d, f) : -1;
        if (o >= 0) {
            float *out = p.grad_in + o + (int64_t)ci_base * HW;
#pragma unroll
            for (int r = 0; r < ROWS; ++r)
                if (r < ci_here) out[(int64_t)r * HW] = val[r];
        }
        frame_advance(d, f, 2 * kEpiChunk);
    }
}

// TMA-store epilogue (stride 1, tiles of whole frame rows, W a multiple of 4
// up to 64, grad_in 16-byte aligned): for each output row of the tile (part p
// takes the rows of parity p) and each group of 8 channels, the warp loads the
// row's W accumulator columns, copies them into a dense [8 channels][W] box in
// shared memory and one lane stores the box with a TMA tensor store, so
// grad_in is written in whole, aligned rows.
template <int V>
__device__ void epilogue_tma(const TcParams &p, const PhaseDesc &d, const Tile &ti,
                             uint32_t taddr, uint32_t box, int q, int part, int lane, int &bsel) {
    if ((V == kVarGeneral || V == kVarMN) && p.mn_b) {
        // Whole-image 1x1 tiles: accumulator column c is plane position c.
        // Per 32 positions the warp's channels go into a [channels][32]
        // float box, 128-byte swizzled (conflict-free writes; the box is
        // 1 KB aligned), stored with one TMA tensor store; positions past
        // the plane and channels past Ci are clipped by the TMA unit.
        const int rows = p.m_tile == 64 ? 16 : 32;
        const int ci0 = ti.mt * p.m_tile + q * rows;
        if (ci0 >= p.Ci) return;
        const int tpi = (d.Hr + p.rows_per_tile - 1) / p.rows_per_tile;
        const int n = ti.pt / tpi, own = tile_own(p, d, ti.pt);
        for (int b = part; b * 32 < own; b += 2) {
            uint32_t v[2][16];
            tmem_ld16(taddr + (uint32_t)(32 * b), v[0]);
            tmem_ld16(taddr + (uint32_t)(32 * b + 16), v[1]);
            tmem_wait_ld16x2(v);
            if (lane == 0) bulk_wait_read_all();  // the previous store has read the box
            __syncwarp();
            if (lane < rows) {
                const uint32_t row = box + (uint32_t)lane * 128u;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    st_shared_v4(row + (uint32_t)((k ^ (lane & 7)) << 4), v[k >> 2][4 * (k & 3)],
                                 v[k >> 2][4 * (k & 3) + 1], v[k >> 2][4 * (k & 3) + 2],
                                 v[k >> 2][4 * (k & 3) + 3]);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) tma_store_3d(&p.out_map, box, 32 * b, ci0, n);
        }
        return;
    }
    const int groups = p.m_tile == 64 ? 1 : 2;
    const int tpi = (d.Hr + p.rows_per_tile - 1) / p.rows_per_tile;
    const int n = ti.pt / tpi, a0 = (ti.pt - n * tpi) * p.rows_per_tile;
    const int W = p.W;
    if (p.epi_box_ci == 16) {
        // 64-row tile: the quadrant's 16 channels (TMEM lanes 0..15 of it) in
        // one [16][W] box per output row; thread t holds channels t/4 and
        // t/4 + 8 at two adjacent columns of each 8-column block.
        const int ci0 = ti.mt * p.m_tile + q * 16;
        if (ci0 >= p.Ci) return;
        const int ch = lane >> 2, c2 = 2 * (lane & 3);
        const uint32_t off_a = 4u * (uint32_t)(ch * W + c2), off_b = off_a + 4u * (uint32_t)(8 * W);
        for (int r = part; r < p.rows_per_tile && a0 + r < d.Hr; r += 2) {
            uint32_t v[32];
            tmem_ld_16x256b_x8(taddr + (uint32_t)(r * d.X), v);
            tmem_wait_ld32(v);
            if (lane == 0) bulk_wait_read_all();  // the previous store has read the box
            __syncwarp();
#pragma unroll
            for (int b = 0; b < 8; ++b) {
                if (8 * b + c2 < W) {  // W is a multiple of 4: both columns or neither
                    st_shared_v2(box + off_a + 32u * b, v[4 * b], v[4 * b + 1]);
                    st_shared_v2(box + off_b + 32u * b, v[4 * b + 2], v[4 * b + 3]);
                }
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) tma_store_4d(&p.out_map, box, 0, a0 + r, ci0, n);
        }
        return;
    }
    for (int gi = 0; gi < groups; ++gi) {
        const int ci0 = ti.mt * p.m_tile + q * 16 * groups + 16 * gi;
        if (ci0 >= p.Ci) break;
        // Rows of this 16-lane group: lanes 16*gi .. 16*gi+15 of the quadrant;
        // lanes 8h .. 8h+7 of the group hold the channels of box pass h.
        const int lg = lane - 16 * gi;
        const bool mine = lg >= 0 && lg < 16;
        const int half_of_lane = (lg >> 3) & 1;
        const uint32_t row_off = 4u * (uint32_t)(W * (lg & 7));
        for (int r = part; r < p.rows_per_tile && a0 + r < d.Hr; r += 2) {
            const uint32_t cbase = taddr + (uint32_t)(r * d.X);
            uint32_t v[64];
#pragma unroll
            for (int c = 0; c < 64; c += 16) {
                if (c >= W) break;
                uint32_t *vc = v + c;
                if (W - c >= 16) {
                    tmem_ld16(cbase + (uint32_t)c, *reinterpret_cast<uint32_t(*)[16]>(vc));
                } else if (W - c >= 8) {
                    tmem_ld8(cbase + (uint32_t)c, vc);
                    if (W - c > 8) tmem_ld4(cbase + (uint32_t)c + 8u, vc + 8);
                } else {
                    tmem_ld4(cbase + (uint32_t)c, vc);
                }
            }
            tmem_wait_ld64(v);
            for (int h = 0; h < 2; ++h) {
                if (ci0 + 8 * h >= p.Ci) break;
                // The store that last used this box must be done reading it
                // (with two boxes, the one before the latest).
                if (lane == 0) {
                    if (p.epi_boxes == 2)
                        bulk_wait_read_1();
                    else
                        bulk_wait_read_all();
                }
                __syncwarp();
                const uint32_t bx = box + (uint32_t)(bsel * p.epi_box_ci * W * 4);
                if (mine && half_of_lane == h) {
#pragma unroll
                    for (int e = 0; e < 64; e += 4)
                        if (e < W)
                            st_shared_v4(bx + row_off + 4u * e, v[e], v[e + 1], v[e + 2], v[e + 3]);
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) tma_store_4d(&p.out_map, bx, 0, a0 + r, ci0 + 8 * h, n);
                if (p.epi_boxes == 2) bsel ^= 1;
            }
        }
    }
}

// Stacked-phase epilogue: TMEM lane = tile position (frame row r, column b of
// the phase grid) within an M-block, column n = (rh * s + rw) * Ci + ci of that
// M-block's accumulator.  Lane quadrant q holds positions 128 mb + 32q .. +31;
// the warps of a quadrant (`parts` of them) split the phases.  Each value goes to grad_in[n][ci][s (a0 + r) + rh][s b + rw];
// consecutive lanes write consecutive columns of a phase, the other phases of
// the row fill the columns in between.
__device__ void epilogue_stacked(const TcParams &p, const PhaseDesc &d, const Tile &ti,
                                 uint32_t taddr, int q, int part, int parts, int lane) {
    const int tpi = (d.Hr + p.rows_per_tile - 1) / p.rows_per_tile;
    const int n = ti.pt / tpi, a0 = (ti.pt - n * tpi) * p.rows_per_tile;
    const int s = p.stride, phases = s * s;
    const int64_t HW = (int64_t)p.H * p.W;
    float *img = p.grad_in + (int64_t)n * p.Ci * HW;
    if (p.st_qhalo) {
        // Column taps on N: M-block mb is frame row a = a0 + mb; lane l of
        // quadrant q is frame element 32q + l, output column b = (32 - halo) q
        // + l for l < 32 - halo.  Column block i (window tap dx = st_dx0 + i)
        // of lane l + i holds that tap's term for b, so the output is the sum
        // over i of block i shifted down by i lanes -- within the warp.
        const int halo = p.st_qhalo, ncols = st_cols(p);
        const int b = (32 - halo) * q + lane;
        for (int mb = 0; mb < p.st_mblocks; ++mb) {
            const int a = a0 + mb;
            const bool row_ok = a < d.Hr;
            for (int g0 = 0; g0 < p.st_n; g0 += 16) {  // 16 columns (phase, ci) at a time
                uint32_t v[kStMaxTw][16];
#pragma unroll
                for (int i = 0; i < kStMaxTw; ++i)
                    if (i < p.st_tw) tmem_ld16(taddr + (uint32_t)(mb * ncols + i * p.st_n + g0), v[i]);
                tmem_wait_ld16x4(v);
                float out[16];
#pragma unroll
                for (int c = 0; c < 16; ++c) out[c] = __uint_as_float(v[0][c]);
#pragma unroll
                for (int i = 1; i < kStMaxTw; ++i) {
                    if (i < p.st_tw) {
#pragma unroll
                        for (int c = 0; c < 16; ++c)
                            out[c] += __shfl_down_sync(0xffffffffu, __uint_as_float(v[i][c]), i);
                    }
                }
                if (row_ok && lane < 32 - halo && b < d.Wr) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const int col = g0 + c, k = col / p.Ci, ci = col - k * p.Ci;
                        if (k >= phases) break;
                        if (k % parts != part) continue;
                        const int ih = s * a + k / s, iw = s * b + k % s;
                        if (ih < p.H && iw < p.W) img[(int64_t)ci * HW + (int64_t)ih * p.W + iw] = out[c];
                    }
                }
                __syncwarp();  // converge before the next (warp-collective) TMEM loads
            }
        }
        return;
    }
    for (int mb = 0; mb < p.st_mblocks; ++mb) {  // M-block mb: tile positions 128 mb ..
        uint32_t v[32];
        const uint32_t ta = taddr + (uint32_t)(mb * p.st_n);
        tmem_ld16(ta, *reinterpret_cast<uint32_t(*)[16]>(v));
        if (p.st_n > 16) tmem_ld16(ta + 16u, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
        tmem_wait_ld32(v);
        const int h = 128 * mb + 32 * q + lane;
        const int r = h / d.X, b = h - r * d.X;
        if (r >= p.rows_per_tile || a0 + r >= d.Hr || b >= d.Wr) continue;
        // Column c = k * Ci + ci, walked with (k, ci) kept alongside so that v
        // is indexed by constants only.
        int k = 0, ci = 0, rh = 0, rw = 0;
#pragma unroll
        for (int c = 0; c < 32; ++c) {
            if (k >= phases) break;
            if (k % parts == part) {
                const int ih = s * (a0 + r) + rh, iw = s * b + rw;
                if (ih < p.H && iw < p.W) img[(int64_t)ci * HW + (int64_t)ih * p.W + iw] = __uint_as_float(v[c]);
            }
            if (++ci == p.Ci) {
                ci = 0;
                ++k;
                if (++rw == s) {
                    rw = 0;
                    ++rh;
                }
            }
        }
    }
}

// Paired epilogue (stride 2; the column phases rw = 0 and 1 of the same
// output rows in TMEM buffers t0 and t1): per output row of the tile, the
// warp reads both phases' row once for all 32 lanes of its quadrant (one
// grad_in channel per lane), then in two halves of 16 lanes interleaves each
// lane's columns of the two phases into a whole grad_in row of a [16][W] box
// (p.epi_box_ci = 16) and stores the box with one TMA tensor store -- half the
// TMEM reads and half the stores of 8-channel boxes, whose per-store issue
// cost dominates this epilogue.
__device__ void epilogue_pair_tma(const TcParams &p, const PhaseDesc &d0, const PhaseDesc &d1,
                                  const Tile &ti, uint32_t t0, uint32_t t1, uint32_t box, int q,
                                  int part, int lane) {
    const int tpi = (d0.Hr + p.rows_per_tile - 1) / p.rows_per_tile;
    const int n = ti.pt / tpi, a0 = (ti.pt - n * tpi) * p.rows_per_tile;
    const int W = p.W, half = W / 2;  // frame columns of a member row (a multiple of 4, <= 32)
    const int ci_q = ti.mt * p.m_tile + q * 32;
    if (ci_q >= p.Ci) return;
    const uint32_t my_row = box + 4u * (uint32_t)(W * (lane & 15));
    for (int r = part; r < p.rows_per_tile && a0 + r < d0.Hr; r += 2) {
        const uint32_t a0c = t0 + (uint32_t)(r * d0.X), a1c = t1 + (uint32_t)(r * d1.X);
        uint32_t v[64];  // [0, 32): phase rw = 0, [32, 64): rw = 1, frame column c at c
#pragma unroll
        for (int c = 0; c < 32; c += 16) {
            const int rem = half - c;  // a multiple of 4
            if (rem >= 16) {
                tmem_ld16(a0c + c, *reinterpret_cast<uint32_t(*)[16]>(v + c));
                tmem_ld16(a1c + c, *reinterpret_cast<uint32_t(*)[16]>(v + 32 + c));
            } else if (rem > 0) {
                if (rem >= 8) {
                    tmem_ld8(a0c + c, v + c);
                    tmem_ld8(a1c + c, v + 32 + c);
                }
                if (rem == 12) {
                    tmem_ld4(a0c + c + 8, v + c + 8);
                    tmem_ld4(a1c + c + 8, v + 32 + c + 8);
                } else if (rem == 4) {
                    tmem_ld4(a0c + c, v + c);
                    tmem_ld4(a1c + c, v + 32 + c);
                }
            }
        }
        tmem_wait_ld64(v);
        const int ih = 2 * (a0 + r) + d0.rh;
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // lanes 16h .. 16h + 15: channels ci_q + 16h ..
            const int ci0 = ci_q + 16 * h;
            if (ci0 >= p.Ci) break;
            if (lane == 0) bulk_wait_read_all();  // the previous store has read the box
            __syncwarp();
            if ((lane >> 4) == h) {
#pragma unroll
                for (int e = 0; e < 16; ++e)  // grad_in columns 4e .. 4e + 3
                    if (2 * e < half)
                        st_shared_v4(my_row + 16u * (uint32_t)e, v[2 * e], v[32 + 2 * e], v[2 * e + 1],
                                     v[32 + 2 * e + 1]);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) tma_store_4d(&p.out_map, box, 0, ih, ci0, n);
        }
    }
}

template <int V>
__device__ void role_epilogue(const TcParams &p, Shared &sh, uint32_t stage, uint32_t tmem,
                              int warp, int lane) {
    const int64_t HW = (int64_t)p.H * p.W;
    const int q = warp & 3, part = warp >> 2;
    const int rows = p.m_tile == 64 ? 16 : 32;  // channels this warp's quadrant owns
    const uint32_t st_base = stage + (uint32_t)(p.epi_stage_bytes / kEpiWarps) * warp;
    int bsel = 0;  // TMA store box in use (double-buffered epilogue)
    int acc = 0;
    uint32_t accph = 0;
    for (int64_t t = first_tile<V>(p); t < p.total_tiles; t = next_tile<V>(p, t)) {
        if (V == kVarPair && (t & 1)) continue;  // a pair is stored at its first tile
        const Tile ti = decode_tile<V>(p, t);
        const PhaseDesc &d = p.ph[ti.phase];
        if (is_general(V) && d.Jh == 0) {  // no tap reaches this phase: grad_in is zero there
            const int ci_base = ti.mt * p.m_tile + q * rows;
            int ci_here = p.Ci - ci_base;
            ci_here = ci_here < 0 ? 0 : (ci_here > rows ? rows : ci_here);
            const int L0 = tile_start(p, d, ti.pt), own = tile_own(p, d, ti.pt);
            FramePos f = frame_pos(d, L0 + part * kEpiChunk + lane);
            for (int c0 = part * kEpiChunk; c0 < own; c0 += 2 * kEpiChunk) {
                const int64_t o = c0 + lane < own ? out_offset(p, d, f) : -1;
                if (o >= 0)
                    for (int r = 0; r < ci_here; ++r) p.grad_in[o + (int64_t)(ci_base + r) * HW] = 0.f;
                frame_advance(d, f, 2 * kEpiChunk);
            }
            continue;
        }
        if (!wait_bar_warp(smem_u32(&sh.acc_full[acc]), accph, p, sh, lane)) break;
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.tile_p);
        if constexpr (V == kVarPair) {
            // The pair's column phases rw = 0, 1 sit in accumulators 2 acc
            // and 2 acc + 1 of the pair buffer; both are stored together.
            const PhaseDesc &d1 = p.ph[ti.phase + 1];
            const uint32_t tq = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(2 * acc * p.tile_p);
            if (p.epi_tma) {
                epilogue_pair_tma(p, d, d1, ti, tq, tq + (uint32_t)p.tile_p, st_base, q, part, lane);
            } else {
                Tile t1 = ti;
                t1.phase = ti.phase + 1;
                epilogue_staged<32>(p, d, ti, tq, st_base, q, part, lane);
                epilogue_staged<32>(p, d1, t1, tq + (uint32_t)p.tile_p, st_base, q, part, lane);
            }
        } else
        if constexpr (V == kVarStacked)
            epilogue_stacked(p, d, ti, tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.st_mblocks * st_cols(p)),
                             q, part, Roles<V>::epi_warps / 4, lane);
        else if (V == kVarFrame64 || p.epi_tma)  // the 64-wide frame always stores through TMA
            epilogue_tma<V>(p, d, ti, taddr, st_base, q, part, lane, bsel);
        else if (rows == 16)
            epilogue_staged<16>(p, d, ti, taddr, st_base, q, part, lane);
        else
            epilogue_staged<32>(p, d, ti, taddr, st_base, q, part, lane);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.acc_empty[acc]));
        if (++acc == ((V == kVarPair && p.acc_single) ? 1 : 2)) {
            acc = 0;
            accph ^= 1u;
        }
    }
    // Every TMA store of this warp must be complete before the CTA exits.
    if (p.epi_tma && lane == 0) bulk_wait_all();
    __syncwarp();
}

// ------------------------------------------------- positions-on-M mode
// (plan_pm in plan.cu).  A tile is 4 output rows of one image; its window in
// a G stage is hbp rows of 128 bytes (64 grad_out channels), row h = 64u + b
// holding grad_out[n, :, ih0 + ph - (kH-1) + u, b - kPmLeft].

// MMA warp (converged; lane 0 issues): two M = 128 halves per tile, each into its own
// accumulator buffer (kW x 64 columns): for kernel row kh, A = window rows
// from 64 (kH-1-kh) + pw + 128 half, B = the kW packed taps (kh, 0..kW-1).
__device__ void role_mma_pm(const TcParams &p, Shared &sh, uint32_t g_base, uint32_t w_base,
                            uint32_t tmem) {
    const PhaseDesc &d = p.ph[0];
    const uint32_t acc_cols = (uint32_t)(d.Jw * 64);
    const uint32_t w_row = (uint32_t)(d.Jw * p.w_unit_bytes);  // one kernel row of taps
    int gs = 0, acc = 0;
    uint32_t gph = 0, accph = 0;
    bool aborted = !wait_bar(smem_u32(&sh.w_full), 0, p, sh);
    for (int64_t t = blockIdx.x; t < p.total_tiles && !aborted; t += gridDim.x) {
        if (!wait_bar(smem_u32(&sh.full_g[gs]), gph, p, sh)) break;
        tc_fence_after();
        const uint32_t g_stage = g_base + (uint32_t)gs * p.g_stage_bytes;
        for (int half = 0; half < 2; ++half) {
            if (!wait_bar(smem_u32(&sh.acc_empty[acc]), accph ^ 1u, p, sh)) {
                aborted = true;
                break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem + (uint32_t)acc * acc_cols;
            uint32_t accumulate = 0;
            for (int kh = 0; kh < d.Jh; ++kh) {
                const uint32_t a_row =
                    (uint32_t)(kPmPitch * (d.Jh - 1 - kh) + p.pad_w + 128 * half);
                const uint32_t a0 = g_stage + a_row * 128u, b0 = w_base + (uint32_t)kh * w_row;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    tc_mma<false>(d_tmem, sw128_desc(a0 + 32u * k), sw128_desc(b0 + 32u * k),
                                  p.idesc, accumulate);
                    accumulate = 1;
                }
            }
            tc_commit(smem_u32(&sh.acc_full[acc]));
            if (++acc == 2) {
                acc = 0;
                accph ^= 1u;
            }
        }
        if (aborted) break;
        tc_commit(smem_u32(&sh.empty_g[gs]));
        if (++gs == p.ng) {
            gs = 0;
            gph ^= 1u;
        }
    }
    tc_commit(smem_u32(&sh.mma_done));
    wait_drain(smem_u32(&sh.mma_done), 0, p, sh);
}

// Gather warps of the 64-wide frame (positions-on-M mode and the general
// mode's frame64 plans): the frame columns b < kPmLeft of every window row are
// zero in every tile, so they are cleared once per G stage (before its first
// use); each raw slice (16
// or 32 channels x raw_br rows x 56 columns) then lands in the window by 8x8
// block transposes: ldmatrix.trans reads 8 channels x 8 columns, stmatrix
// writes 8 window rows x 16 bytes (the slice's 16-byte channel chunks,
// swizzled).
template <int GW, int NG>  // gather warps, ldmatrix.x4 groups per warp and slice
__device__ void gather_pm(const TcParams &p, Shared &sh, uint32_t g_base, uint32_t raw_base,
                          uint32_t early_base, int gw, int lane) {
    const int slices = p.kc / p.raw_cs;
    const int cgs = p.raw_cs / 8;                      // 8-channel groups per slice (2 or 4)
    const uint32_t row_bytes = (uint32_t)(p.raw_bw * 2);
    const uint32_t ch_bytes = row_bytes * (uint32_t)p.raw_br;
    const int nb_col = p.raw_bw / 8;                   // 8-column blocks per grad_out row
    const int blocks = cgs * p.pm_rows * nb_col;       // 8x8 blocks per slice
    const int groups = (blocks + 3) / 4;               // ldmatrix.x4 per slice
    const int zrows = (p.hbp + kPmPitch - 1) / kPmPitch * kPmLeft;
    int stage = 0;
    uint32_t phase = 0, zeroed = 0;  // bit s: this warp has cleared its share of stage s
    RawCursor rc;
    bool early_done = false;
    bool withhold = (p.debug_flags & DGRAD_DEBUG_SKIP_ARRIVE) && gw == 0;
    // This lane's rows of the warp's (at most NG) ldmatrix.x4 groups,
    // the same for every slice: source offset in a raw slot, destination
    // window row and channel group.
    uint32_t src_off[NG], dst_row[NG];
    int cgk[NG];
    int ng_mine = 0;
    {
        const int m = lane >> 3, kr = lane & 7;
#pragma unroll
        for (int j = 0; j < NG; ++j) {
            const int gi = gw + j * GW;
            if (gi < groups) ng_mine = j + 1;
            int b = gi * 4 + m;
            b = b < blocks ? b : blocks - 1;  // a ragged last group repeats a block
            const int pb = b % nb_col, rest = b / nb_col;
            const int u = rest % p.pm_rows, cg = rest / p.pm_rows;
            const int h = kPmPitch * u + kPmLeft + 8 * pb + kr;
            src_off[j] = (uint32_t)(8 * cg + kr) * ch_bytes + (uint32_t)u * row_bytes + (uint32_t)pb * 16u;
            dst_row[j] = (uint32_t)h * 128u;
            cgk[j] = cg ^ (h & 7);  // XOR with the slice's chunk pair gives the swizzled chunk
        }
    }
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x)
    for (int cc = 0; cc < p.n_cchunks; ++cc) {
        if (!wait_bar_warp(smem_u32(&sh.empty_g[stage]), phase ^ 1u, p, sh, lane)) return;
        if (!stage_writable(p, sh, stage, early_done, lane)) return;
        const uint32_t s_base = g_base + (uint32_t)stage * p.g_stage_bytes;
        if (!(zeroed >> stage & 1u)) {  // frame columns b < kPmLeft: zero in every tile
            zeroed |= 1u << stage;
            for (int k = gw * 32 + lane; k < zrows * 8; k += GW * 32) {
                const int zr = k >> 3, h = (zr / kPmLeft) * kPmPitch + zr % kPmLeft;
                if (h < p.hbp)
                    st_shared_v4(s_base + (uint32_t)h * 128u + (uint32_t)(k & 7) * 16u, 0u, 0u, 0u, 0u);
            }
        }
        for (int sl = 0; sl < slices; ++sl) {
            uint32_t raw;
            if (!raw_acquire(p, sh, rc, raw_base, early_base, lane, raw)) return;
            uint32_t r[NG][4];
#pragma unroll
            for (int j = 0; j < NG; ++j)
                if (j < ng_mine) ldmatrix_x4_trans(raw + src_off[j], r[j]);
#pragma unroll
            for (int j = 0; j < NG; ++j)
                if (j < ng_mine)
                    stmatrix_x4(s_base + dst_row[j] + (uint32_t)(((cgs * sl) ^ cgk[j]) << 4), r[j]);
            raw_release(p, sh, rc, lane);
        }
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
            if (withhold)
                withhold = false;  // failure injection: this stage is never signalled
            else
                mbar_arrive(smem_u32(&sh.full_g[stage]));
        }
        if (++stage == p.ng) {
            stage = 0;
            phase ^= 1u;
        }
    }
}

// Entry of the exchange slot holding block kw (1 or 2) of even-quadrant lane
// l (32 - kw <= l <= 31): 0 for (1, 31), 1 and 2 for (2, 30) and (2, 31).
__device__ __forceinline__ int x_entry(int kw, int l) { return kw * (kw - 1) / 2 + l - (32 - kw); }

// Warps 0..15 in two groups of 8: group g = w / 8 drains half g of every
// tile (accumulator buffer g), so one group's stores overlap the other's TMEM
// reads and shuffles.  Warp w reads TMEM lane quadrant q = w mod 4 (positions
// 32q..32q+31 of the half: output row 2g + q / 2, columns 32 (q mod 2) + lane
// - kPmLeft) for the 16-channel chunks {2 part, 2 part + 1}, part = (w / 4)
// mod 2.  out(lane l) = sum over kw of block kw at lane l - kw: a shuffle
// within the warp, except for the first kw lanes of an odd quadrant, whose
// values come from the last lanes of the even quadrant below through a small
// shared buffer (the "pair" of warps q-1, q with the same group and part; one
// slot per chunk, each with a full / empty mbarrier).  Even quadrants' first
// lanes are frame padding (b < 8), so no value crosses a 64-position frame
// row.  Each store instruction writes 32 consecutive grad_in floats of one
// channel.
__device__ void epilogue_pm(const TcParams &p, Shared &sh, uint32_t xbase, uint32_t tmem,
                            int warp, int lane) {
    const PhaseDesc &d = p.ph[0];
    const int half = warp >> 3, q = warp & 3, part = (warp >> 2) & 1, odd = q & 1;
    const int pair = half * 4 + part * 2 + (q >> 1);
    const int Jw = d.Jw, nchunks = (p.Ci + 15) / 16;
    const int my_chunks = nchunks - 2 * part < 0 ? 0 : (nchunks - 2 * part > 2 ? 2 : nchunks - 2 * part);
    const uint32_t taddr =
        tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(half * Jw * 64);  // accumulator `half`
    const uint32_t acc_full = smem_u32(&sh.acc_full[half]), acc_empty = smem_u32(&sh.acc_empty[half]);
    const int tpi = (p.H + p.rows_per_tile - 1) / p.rows_per_tile;
    const int64_t HW = (int64_t)p.H * p.W;
    const int iw = 32 * odd + lane - kPmLeft;
    uint32_t accph = 0;
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x, accph ^= 1u) {
        const int n = (int)(t / tpi), ih0 = (int)(t - (int64_t)n * tpi) * p.rows_per_tile;
        const int ih = ih0 + 2 * half + (q >> 1);
        const bool valid = ih < p.H && iw >= 0 && iw < p.W;
        if (!wait_bar_warp(acc_full, accph, p, sh, lane)) return;
        tc_fence_after();
        if (my_chunks == 0) {
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty);
        }
        for (int lc = 0; lc < my_chunks; ++lc) {
            const int ci0 = (2 * part + lc) * 16;
            uint32_t v[kPmMaxKw][16] = {};
#pragma unroll
            for (int kw = 0; kw < kPmMaxKw; ++kw)
                if (kw < Jw) tmem_ld16(taddr + (uint32_t)(kw * 64 + ci0), v[kw]);
            tmem_wait_ld3(v);
            if (lc == my_chunks - 1) {
                // The accumulator is in registers: the MMA may reuse it.
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acc_empty);
            }
            const uint32_t xslot = xbase + (uint32_t)((pair * 2 + lc) * kPmXSlotBytes);
            const uint32_t xf = smem_u32(&sh.x_full[pair * 2 + lc]);
            const uint32_t xe = smem_u32(&sh.x_empty[pair * 2 + lc]);
            if (!odd && Jw > 1) {
                // Publish lanes 32-kw.. of block kw for the odd quadrant.
                if (!wait_bar_warp(xe, accph ^ 1u, p, sh, lane)) return;
#pragma unroll
                for (int kw = 1; kw < kPmMaxKw; ++kw) {
                    if (kw < Jw && lane >= 32 - kw) {
                        const uint32_t a = xslot + (uint32_t)(x_entry(kw, lane) * 64);
#pragma unroll
                        for (int k = 0; k < 16; k += 4)
                            st_shared_v4(a + 4u * k, v[kw][k], v[kw][k + 1], v[kw][k + 2], v[kw][k + 3]);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(xf);
            }
            // Sum of block kw at lane l - kw; an odd quadrant's first kw lanes
            // take that term from the exchange buffer instead.
            float out[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) out[k] = __uint_as_float(v[0][k]);
#pragma unroll
            for (int kw = 1; kw < kPmMaxKw; ++kw) {
                if (kw < Jw) {
                    const bool mine = !(odd && lane < kw);
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const float sv = __shfl_up_sync(0xffffffffu, __uint_as_float(v[kw][k]), kw);
                        out[k] += mine ? sv : 0.f;
                    }
                }
            }
            if (odd && Jw > 1) {
                if (!wait_bar_warp(xf, accph, p, sh, lane)) return;
                if (lane < Jw - 1) {
                    for (int kw = lane + 1; kw < Jw; ++kw) {
                        const uint32_t a = xslot + (uint32_t)(x_entry(kw, lane + 32 - kw) * 64);
#pragma unroll
                        for (int k = 0; k < 16; k += 4) {
                            const float4 x = ld_shared_f32x4(a + 4u * k);
                            out[k] += x.x;
                            out[k + 1] += x.y;
                            out[k + 2] += x.z;
                            out[k + 3] += x.w;
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(xe);
            }
            if (valid) {
                float *o = p.grad_in + ((int64_t)n * p.Ci + ci0) * HW + (int64_t)ih * p.W + iw;
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (ci0 + k < p.Ci) o[(int64_t)k * HW] = out[k];
            }
        }
    }
}

// Warp roles of the kernel variants: the general mode and the 64-wide frame
// share a layout, positions-on-M has its own.
// V (kVar*): which plan the kernel runs -- the general mode (any phase count,
// raw-slice or register gather, resident or streamed weights, TMA-store or
// staged epilogue), the 64-wide frame, or positions-on-M.  Each variant
// compiles only its own roles.
template <int ESIZE, int V>
__global__ void __launch_bounds__(Roles<V>::threads, 1)
    dgrad_tc_kernel(const __grid_constant__ TcParams p) {
    using R = Roles<V>;
    constexpr bool PM = V == kVarPosM;
    extern __shared__ __align__(1024) uint8_t smem[];
    // Layout (smem_layout_bytes): the base rounded up to 1 KB, the barrier
    // block, then epilogue staging, raw ring, G stages and weights, each ring
    // on a 1 KB boundary (the 128-byte swizzle pattern is tied to it).
    const uint32_t base = (smem_u32(smem) + 1023u) & ~1023u;
    Shared &sh = *reinterpret_cast<Shared *>(smem + (base - smem_u32(smem)));
    const uint32_t epi_stage = base + kBarrierBytes;
    const uint32_t raw_base = epi_stage + (((uint32_t)p.epi_stage_bytes + 1023u) & ~1023u);
    const uint32_t g_base =
        raw_base + (((uint32_t)(p.raw_nr * p.raw_slice_bytes) + 1023u) & ~1023u);
    const uint32_t w_base = g_base + (uint32_t)(p.ng * p.g_stage_bytes);
    const uint32_t early_base = g_base + (uint32_t)p.g_stage_bytes;  // G stage 1
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.ng; ++s) {
            mbar_init(smem_u32(&sh.full_g[s]), R::g_warps);
            mbar_init(smem_u32(&sh.empty_g[s]), 1);
        }
        for (int s = 0; s < p.nw; ++s) {
            mbar_init(smem_u32(&sh.full_w[s]), 1);
            mbar_init(smem_u32(&sh.empty_w[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&sh.acc_full[s]), 1);
            mbar_init(smem_u32(&sh.acc_empty[s]), PM ? R::epi_warps / 2 : R::epi_warps);
        }
        for (int s = 0; s < 16; ++s) {
            mbar_init(smem_u32(&sh.x_full[s]), 1);
            mbar_init(smem_u32(&sh.x_empty[s]), 1);
        }
        for (int s = 0; s < p.raw_nr; ++s) {
            mbar_init(smem_u32(&sh.full_raw[s]), 1);
            mbar_init(smem_u32(&sh.empty_raw[s]), R::g_warps);
        }
        for (int s = 0; s < kMaxEarly; ++s) mbar_init(smem_u32(&sh.full_early[s]), 1);
        mbar_init(smem_u32(&sh.early_free), R::g_warps);
        mbar_init(smem_u32(&sh.w_full), p.w_raw ? R::epi_warps : 1);
        mbar_init(smem_u32(&sh.mma_done), 1);
        sh.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == R::mma_warp) {
        tmem_alloc(smem_u32(&sh.tmem_base), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    if (warp == R::w_warp && lane == 0 && p.gather_tma)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.in_map)) : "memory");
    // Everything above touched only this CTA's shared memory, TMEM and its own
    // parameters, so it may overlap the previous kernel; global memory is used
    // only from here.
    if (threadIdx.x == 0) grid_launch_dependents();
    // The TMA producer (lane 0 of its warp) waits inside raw_producer, right
    // before its first global-memory access; the other lanes of that warp
    // never touch global memory.  Every other thread waits here.
    const bool lazy_wait = warp == R::w_warp && p.nw == 0 && p.gather_tma;
    if (!lazy_wait) grid_dependency_wait();

    if (warp == R::w_warp) {
        if (lane == 0) {
            if (R::w2_warp >= 0 && p.nw != 0 && p.gather_tma)  // raw slices here, weights on w2_warp
                raw_stream_producer(p, sh, raw_base);
            else
                role_weights<V>(p, sh, w_base, raw_base, early_base);
        }
        __syncwarp();
    } else if (R::w2_warp >= 0 && warp == R::w2_warp) {
        if (lane == 0 && p.nw != 0 && p.gather_tma) weight_stream_producer(p, sh, w_base);
        __syncwarp();
    } else if (warp == R::mma_warp) {
        {  // the whole warp: tc_mma / tc_commit issue from lane 0
            if constexpr (PM)
                role_mma_pm(p, sh, g_base, w_base, tmem);
            else
            {
                if constexpr (V == kVarStacked)
                    role_mma_stacked<ESIZE == 4>(p, sh, g_base, w_base, tmem);
                else
                    role_mma<ESIZE == 4, V>(p, sh, g_base, w_base, tmem);
            }
        }
        __syncwarp();
    } else if (warp >= R::g_warp0) {
        if constexpr (PM)
            gather_pm<kPmGWarps, kPmGroups>(p, sh, g_base, raw_base, early_base, warp - R::g_warp0, lane);
        else if constexpr (V == kVarFrame64)
            gather_pm<kGWarps, kF64Groups>(p, sh, g_base, raw_base, early_base, warp - R::g_warp0, lane);
        else if (ESIZE == 2 && p.mn_b)
            gather_mn<R::g_warps>(p, sh, g_base, raw_base, early_base, warp - R::g_warp0, lane);
        else if (p.gather_tma)
            gather_from_raw<ESIZE, R::g_warps>(p, sh, g_base, raw_base, early_base, warp - R::g_warp0, lane);
        else
            role_gather<ESIZE, R::g_warps>(p, sh, g_base, warp - R::g_warp0, lane);
    } else {
        if constexpr (ESIZE == 2 && (V == kVarGeneral || V == kVarFrame64)) {
            if (p.w_raw) pack_resident_weights(p, sh, w_base, (int)threadIdx.x, R::epi_warps * 32);
        }
        if constexpr (PM)
            epilogue_pm(p, sh, epi_stage, tmem, warp, lane);
        else
            role_epilogue<V>(p, sh, epi_stage, tmem, warp, lane);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == R::mma_warp) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
}

// Dynamic shared memory is raised once per device and variant to the full
// limit, so no attribute call happens on later launches (e.g. during stream
// capture).
template <int ESIZE, int V>
int launch_variant(const TcParams &p, int grid, cudaStream_t st, int dev) {
    static std::atomic<uint64_t> configured{0};  // bit per device
    auto kern = dgrad_tc_kernel<ESIZE, V>;
    const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
    if (!bit || !(configured.load() & bit)) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return (int)e;
        configured.fetch_or(bit);
    }
    // Launched with programmatic stream serialization: the prologue of this
    // kernel may overlap the tail of the previous one (see grid_dependency_wait).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(Roles<V>::threads);
    cfg.dynamicSmemBytes = (size_t)p.smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) return (int)e;
    return (int)cudaGetLastError();
}

int sm_count(int dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against the driver library).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            ptr = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }();
    return fn;
}

// grad_out as a 4-D tensor [N][Co][OH/g][g*OW] (g = raw_rowg grad_out rows
// per map row) with a [1][raw_cs][raw_br/g][raw_bw or g*OW] load box, for the
// tiled-mode raw gather; the bulk-copy modes need no map, only a 16-byte
// aligned grad_out.
bool encode_in_map(TcParams &p) {
    if (p.raw_nr <= 0 || p.rows_per_tile <= 0 || p.raw_mode == kRawNone) return false;
    if ((reinterpret_cast<uintptr_t>(p.grad_out) & 15u) != 0) return false;
    if (p.raw_mode != kRawTiled) return true;  // 1-D bulk copies: no tensor map
    if (((int64_t)p.OW * p.raw_rowg * p.esize) % 16 != 0) return false;  // map rows: raw_rowg grad_out rows
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const int64_t e = p.esize, g = p.raw_rowg;  // g grad_out rows per map row
    const cuuint64_t dims[4] = {(cuuint64_t)(p.OW * g), (cuuint64_t)(p.OH / g), (cuuint64_t)p.Co,
                                (cuuint64_t)p.N};
    const cuuint64_t strides[3] = {(cuuint64_t)(p.OW * g * e), (cuuint64_t)(p.OH * p.OW * e),
                                   (cuuint64_t)((int64_t)p.Co * p.OH * p.OW * e)};
    const cuuint32_t box[4] = {(cuuint32_t)(g > 1 ? p.OW * g : p.raw_bw), (cuuint32_t)(p.raw_br / g),
                               (cuuint32_t)p.raw_cs, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    const CUtensorMapDataType dt =
        e == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT16;
    CUresult r = fn(&p.in_map, dt, 4, const_cast<void *>(p.grad_out), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// grad_in as a 4-D float32 tensor [N][Ci][H][W] with a [1][epi_box_ci][1][W] store box;
// for the MN-major mode a 3-D tensor [N][Ci][H*W] with a 128-byte swizzled
// [1][channels][32] box (one box per warp and 32 positions).
bool encode_out_map(TcParams &p) {
    if (p.mn_b) {
        const int64_t HW = (int64_t)p.H * p.W;
        const int rows = p.m_tile == 64 ? 16 : 32;
        if ((reinterpret_cast<uintptr_t>(p.grad_in) & 15u) != 0 || (HW * 4) % 16 != 0) return false;
        if (p.epi_stage_bytes / kEpiWarps < rows * 128 || (p.epi_stage_bytes / kEpiWarps) % 1024 != 0)
            return false;
        PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
        if (!fn) return false;
        const cuuint64_t dims[3] = {(cuuint64_t)HW, (cuuint64_t)p.Ci, (cuuint64_t)p.N};
        const cuuint64_t strides[2] = {(cuuint64_t)HW * 4, (cuuint64_t)p.Ci * HW * 4};
        const cuuint32_t box[3] = {32u, (cuuint32_t)rows, 1u};
        const cuuint32_t estr[3] = {1u, 1u, 1u};
        CUresult r = fn(&p.out_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, p.grad_in, dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        return r == CUDA_SUCCESS;
    }
    if (p.rows_per_tile <= 0 || (p.stride != 1 && !p.pair_rw) || p.W % 4 != 0 || p.W > 64) return false;
    if ((reinterpret_cast<uintptr_t>(p.grad_in) & 15u) != 0) return false;
    if (p.epi_stage_bytes < kEpiWarps * p.epi_boxes * p.epi_box_ci * p.W * 4) return false;
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[4] = {(cuuint64_t)p.W, (cuuint64_t)p.H, (cuuint64_t)p.Ci,
                                (cuuint64_t)p.N};
    const cuuint64_t strides[3] = {(cuuint64_t)p.W * 4, (cuuint64_t)p.H * p.W * 4,
                                   (cuuint64_t)p.Ci * p.H * p.W * 4};
    const cuuint32_t box[4] = {(cuuint32_t)p.W, 1u, (cuuint32_t)p.epi_box_ci, 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = fn(&p.out_map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, p.grad_in, dims, strides, box,
                    estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

int launch_tc(const Plan &plan, const void *grad_out, const void *packed, float *grad_in,
              void *stream) {
    NvtxRange range("conv2d_grad_input: dgrad (tcgen05)");
    TcParams p = plan.tc;
    p.grad_out = grad_out;
    p.packed = packed;
    p.grad_in = grad_in;
    p.epi_tma = 0;
    p.gather_tma = encode_in_map(p) ? 1 : 0;
    if (!p.pos_m) p.epi_tma = encode_out_map(p) ? 1 : 0;
    if ((p.pos_m && !p.gather_tma) || (p.frame64 && !(p.gather_tma && p.epi_tma)) ||
        (p.mn_b && !p.gather_tma)) {
        // The positions-on-M mode and the MN-major operand need the TMA /
        // bulk-copy gather (grad_out 16-byte aligned), the 64-wide frame also
        // the TMA store epilogue (grad_in 16-byte aligned); the general plan
        // on the Wr + Jw - 1 frame shares their packed weights.
        p = plan.tc_alt;
        p.grad_out = grad_out;
        p.packed = packed;
        p.grad_in = grad_in;
        p.gather_tma = encode_in_map(p) ? 1 : 0;
        p.epi_tma = encode_out_map(p) ? 1 : 0;
    }
    if (!p.gather_tma) p.raw_early = 0;
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return (int)de;
    const int sms = sm_count(dev);
    if (sms <= 0) return (int)cudaErrorInvalidDevice;
    // At least half the shared memory of an SM, so a second CTA can never be
    // co-resident and contend for tensor memory.
    if (p.smem_bytes < kSmemLimit / 2 + 1024) p.smem_bytes = kSmemLimit / 2 + 1024;
    if (p.tile_group < 1) p.tile_group = 1;
    const int64_t groups = (p.total_tiles + p.tile_group - 1) / p.tile_group;
    const int grid = (int)(groups < sms ? groups : sms);
    if (grid <= 0) return (int)cudaSuccess;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (plan.esize == 2) {
        if (p.pos_m) return launch_variant<2, kVarPosM>(p, grid, st, dev);
        if (p.frame64) return launch_variant<2, kVarFrame64>(p, grid, st, dev);
        if (p.stacked) return launch_variant<2, kVarStacked>(p, grid, st, dev);
        if (p.pair_rw) return launch_variant<2, kVarPair>(p, grid, st, dev);
        if (p.mn_b) return launch_variant<2, kVarMN>(p, grid, st, dev);
        return launch_variant<2, kVarGeneral>(p, grid, st, dev);
    }
    if (p.stacked) return launch_variant<4, kVarStacked>(p, grid, st, dev);
    if (p.pair_rw) return launch_variant<4, kVarPair>(p, grid, st, dev);
    return launch_variant<4, kVarGeneral>(p, grid, st, dev);
}

int tc_read_and_clear_error(unsigned int *out) {
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_dgrad_error_word, sizeof(v));
    if (e != cudaSuccess) return (int)e;
    if (v != 0) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_dgrad_error_word, &zero, sizeof(zero));
        if (e != cudaSuccess) return (int)e;
    }
    *out = v;
    return (int)cudaSuccess;
}

}  // namespace dgrad
