// dgrad_tc.cu -- the sm_103a tensor-core dgrad kernel (tcgen05 + TMEM + mbarrier).
//
// What it computes is the page's implicit GEMM (conv2d_grad_input_gemm_coop.wgsl,
// header comment): per batch item C[Ci, H*W] = A[Ci, K] x B[K, H*W], K =
// Co*kH*kW, with the exact-adjoint index map of its strided staging branch.
// How it computes it is GB300-first rather than the shader's 2x2 grid of
// cooperative-matrix tiles with two workgroup barriers per K step:
//
//  * M = 128 grad_in pixels of one sub-pixel phase (the frame of
//    dgrad_internal.h), N = up to 256 input channels, K = grad_out channels x
//    the phase's own taps.  Strided problems never multiply structural zeros.
//  * A (the im2col operand) is never materialised per tap: for each block of
//    grad_out channels, gather warps write one frame window of
//    128 + (Jh-1)*X + Jw-1 pixels into shared memory as K-major,
//    no-swizzle core matrices, and every tap is the same window read through
//    a shared-memory descriptor whose start is shifted by that tap's offset.
//  * B (weights) comes pre-packed (pack.cu) in exactly its shared-memory image
//    and moves with cp.async.bulk: resident for the whole kernel when it fits,
//    otherwise through a ring of per-channel-block stages.
//  * One thread issues tcgen05.mma (kind::f16 for bf16/fp16, kind::tf32 for
//    fp32) into a double-buffered TMEM accumulator; four epilogue warps drain
//    the other buffer with tcgen05.ld and write float32 NCHW grad_in with
//    per-element predication, so a tile's epilogue overlaps the next tile's
//    MMAs.  Persistent grid: one CTA per SM walking the tile list.
//
// Every mbarrier wait is bounded by a wall-clock limit (globaltimer).  On
// expiry the CTA raises an abort flag in shared memory, sets bit 0 of the
// device error word, drains copies and MMAs it has in flight, releases TMEM
// and returns; no wait is unbounded and nothing traps.
#include <cuda_runtime.h>

#include <atomic>

#include "conv2d_grad_input.h"
#include "dgrad_internal.h"

namespace dgrad {

__device__ unsigned int g_dgrad_error_word = 0;

namespace {

struct Shared {
    uint64_t full_a[4], empty_a[4], full_b[4], empty_b[4];
    uint64_t acc_full[2], acc_empty[2];
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

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
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

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
                 "r"(d)
                 : "memory");
}

__device__ __forceinline__ uint32_t ldg_u16(const unsigned short *p) {
    unsigned short v;
    asm volatile("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint32_t ldg_tf32(const float *p) {
    float v;
    asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(v) : "l"(p));
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return r;
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

__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

template <bool TF32>
__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    if constexpr (TF32) {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    }
}

// 32 lanes x 16 consecutive float32 columns of TMEM, waited for before return.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor (tcgen05 format): K-major, no swizzle.
// Core matrices are 8 rows x 16 bytes stored contiguously; `lbo` is the byte
// step between core matrices adjacent in K, `sbo` the step between core
// matrices adjacent in M/N.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version
    return d;                // base offset 0, relative LBO, layout SWIZZLE_NONE
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

// Whole warp: lane 0 waits, the verdict is broadcast.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const TcParams &p,
                                              Shared &sh, int lane) {
    int ok = 0;
    if (lane == 0) ok = wait_bar(bar, parity, p, sh) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// Waits that must end even while aborting (copies / MMAs already in flight).
__device__ __forceinline__ void wait_drain(uint32_t bar, uint32_t parity, const TcParams &p,
                                           Shared &sh) {
    if (mbar_try_wait(bar, parity)) return;
    wait_slow(bar, parity, p.wait_limit_ns, sh, false);
}

// ------------------------------------------------------------ tile decode
struct Tile {
    int phase, mt, nt;
};

__device__ __forceinline__ Tile decode_tile(const TcParams &p, int64_t t) {
    int ph = 0;
    while (ph + 1 < p.n_phases && t >= p.ph[ph + 1].tile_begin) ++ph;
    const int64_t local = t - p.ph[ph].tile_begin;
    Tile r;
    r.phase = ph;
    r.mt = (int)(local / p.n_ntiles);
    r.nt = (int)(local - (int64_t)r.mt * p.n_ntiles);
    return r;
}

// ------------------------------------------------------------------ roles
// Warp 5, lane 0: packed weights into shared memory with bulk copies.
__device__ void role_weights(const TcParams &p, Shared &sh, uint32_t b_base) {
    const uint8_t *src = static_cast<const uint8_t *>(p.packed);
    if (p.nb == 0) {
        const uint32_t bar = smem_u32(&sh.w_full);
        mbar_arrive_expect_tx(bar, (uint32_t)p.packed_bytes);
        for (int64_t off = 0; off < p.packed_bytes; off += 32768) {
            const int64_t left = p.packed_bytes - off;
            bulk_g2s(b_base + (uint32_t)off, src + off, (uint32_t)(left < 32768 ? left : 32768), bar);
        }
        wait_drain(bar, 0, p, sh);  // never leave a copy in flight
        return;
    }
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    bool aborted = false;
    for (int64_t t = blockIdx.x; t < p.total_tiles && !aborted; t += gridDim.x) {
        const Tile ti = decode_tile(p, t);
        const PhaseDesc &d = p.ph[ti.phase];
        if (d.Jh == 0) continue;
        const int taps = d.Jh * d.Jw;
        const uint32_t bytes = (uint32_t)(taps * p.b_unit_bytes);
        for (int cc = 0; cc < p.n_cchunks; ++cc) {
            if (!wait_bar(smem_u32(&sh.empty_b[stage]), phase ^ 1u, p, sh)) {
                aborted = true;
                break;
            }
            const uint8_t *s =
                src + d.pack_off + ((int64_t)ti.nt * p.n_cchunks + cc) * taps * p.b_unit_bytes;
            const uint32_t full = smem_u32(&sh.full_b[stage]);
            mbar_arrive_expect_tx(full, bytes);
            bulk_g2s(b_base + (uint32_t)stage * p.b_stage_bytes, s, bytes, full);
            ++issued;
            if (++stage == p.nb) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
    if (aborted) {
        // Let every copy that may still be landing finish before the CTA exits.
        const int64_t k_end = issued < p.nb ? issued : p.nb;
        for (int64_t k = 0; k < k_end; ++k) {
            const int64_t q = issued - 1 - k;
            wait_drain(smem_u32(&sh.full_b[q % p.nb]), (uint32_t)((q / p.nb) & 1), p, sh);
        }
    }
}

// Warp 4, lane 0: tcgen05.mma issue.
template <bool TF32>
__device__ void role_mma(const TcParams &p, Shared &sh, uint32_t a_base, uint32_t b_base,
                         uint32_t tmem) {
    constexpr int E = TF32 ? 4 : 8;  // elements per 16 bytes
    const int ksteps = p.kc / (2 * E);  // MMA K-steps (32 bytes each) per tap and stage
    int as = 0, bs = 0, acc = 0;
    uint32_t aph = 0, bph = 0, accph = 0;
    bool aborted = false;
    if (p.nb == 0 && !wait_bar(smem_u32(&sh.w_full), 0, p, sh)) aborted = true;
    const uint32_t a_lbo = (uint32_t)p.hbp * 16u;
    const uint32_t b_lbo = (uint32_t)p.n_tile * 16u;
    for (int64_t t = blockIdx.x; t < p.total_tiles && !aborted; t += gridDim.x) {
        const Tile ti = decode_tile(p, t);
        const PhaseDesc &d = p.ph[ti.phase];
        if (d.Jh == 0) continue;
        if (!wait_bar(smem_u32(&sh.acc_empty[acc]), accph ^ 1u, p, sh)) {
            aborted = true;
            break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + (uint32_t)(acc * p.n_tile);
        const int taps = d.Jh * d.Jw;
        uint32_t accumulate = 0;
        for (int cc = 0; cc < p.n_cchunks; ++cc) {
            if (!wait_bar(smem_u32(&sh.full_a[as]), aph, p, sh)) {
                aborted = true;
                break;
            }
            uint32_t b_stage;
            if (p.nb == 0) {
                b_stage = b_base + (uint32_t)(d.pack_off + ((int64_t)ti.nt * p.n_cchunks + cc) *
                                                               taps * p.b_unit_bytes);
            } else {
                if (!wait_bar(smem_u32(&sh.full_b[bs]), bph, p, sh)) {
                    aborted = true;
                    break;
                }
                b_stage = b_base + (uint32_t)bs * p.b_stage_bytes;
            }
            tc_fence_after();
            const uint32_t a_stage = a_base + (uint32_t)as * p.a_stage_bytes;
            for (int j = 0; j < d.Jh; ++j) {
                for (int i = 0; i < d.Jw; ++i) {
                    const uint32_t a_tap =
                        a_stage + (uint32_t)(((d.Jh - 1 - j) * d.X + (d.Jw - 1 - i)) * 16);
                    const uint32_t b_tap = b_stage + (uint32_t)((j * d.Jw + i) * p.b_unit_bytes);
                    for (int k = 0; k < ksteps; ++k) {
                        const uint64_t ad = smem_desc(a_tap + 2u * k * a_lbo, a_lbo, 128);
                        const uint64_t bd = smem_desc(b_tap + 2u * k * b_lbo, b_lbo, 128);
                        tc_mma<TF32>(d_tmem, ad, bd, p.idesc, accumulate);
                        accumulate = 1;
                    }
                }
            }
            tc_commit(smem_u32(&sh.empty_a[as]));
            if (++as == p.na) {
                as = 0;
                aph ^= 1u;
            }
            if (p.nb != 0) {
                tc_commit(smem_u32(&sh.empty_b[bs]));
                if (++bs == p.nb) {
                    bs = 0;
                    bph ^= 1u;
                }
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

// Warps 6..9: grad_out frame windows into K-major core matrices.
template <int ESIZE, int CHUNKS>
__device__ void role_gather(const TcParams &p, Shared &sh, uint32_t a_base, int gw, int lane) {
    const int64_t plane = (int64_t)p.OH * p.OW;
    int stage = 0;
    uint32_t phase = 0;
    bool withhold = (p.debug_flags & DGRAD_DEBUG_SKIP_ARRIVE) && gw == 0;
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        const Tile ti = decode_tile(p, t);
        const PhaseDesc &d = p.ph[ti.phase];
        if (d.Jh == 0) continue;
        const int L0 = ti.mt * kTileM;
        const int img = d.R * d.X;
        for (int cc = 0; cc < p.n_cchunks; ++cc) {
            if (!wait_bar_warp(smem_u32(&sh.empty_a[stage]), phase ^ 1u, p, sh, lane)) return;
            const uint32_t s_base = a_base + (uint32_t)stage * p.a_stage_bytes;
            const int co0 = cc * p.kc;
            const int cleft = p.Co - co0;
            for (int h = gw * 32 + lane; h < p.hbp; h += kAWarps * 32) {
                const int lam = L0 + h;
                const int n = lam / img;
                const int rem = lam - n * img;
                const int rho = rem / d.X;
                const int kap = rem - rho * d.X;
                const int u = rho - (d.Jh - 1) + d.qh;
                const int v = kap - (d.Jw - 1) + d.qw;
                const bool ok = n < p.N && u >= 0 && u < p.OH && v >= 0 && v < p.OW;
                const int cvalid = ok ? (cleft < p.kc ? cleft : p.kc) : 0;
                const int64_t off =
                    ok ? ((int64_t)n * p.Co + co0) * plane + (int64_t)u * p.OW + v : 0;
                uint32_t q[CHUNKS][4];
                if constexpr (ESIZE == 2) {
                    const unsigned short *g = static_cast<const unsigned short *>(p.grad_out) + off;
#pragma unroll
                    for (int kc = 0; kc < CHUNKS; ++kc) {
#pragma unroll
                        for (int e = 0; e < 8; e += 2) {
                            const int c = kc * 8 + e;
                            const uint32_t lo = c < cvalid ? ldg_u16(g + c * plane) : 0u;
                            const uint32_t hi = c + 1 < cvalid ? ldg_u16(g + (c + 1) * plane) : 0u;
                            q[kc][e / 2] = lo | (hi << 16);
                        }
                    }
                } else {
                    const float *g = static_cast<const float *>(p.grad_out) + off;
#pragma unroll
                    for (int kc = 0; kc < CHUNKS; ++kc) {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int c = kc * 4 + e;
                            q[kc][e] = c < cvalid ? ldg_tf32(g + c * plane) : 0u;
                        }
                    }
                }
#pragma unroll
                for (int kc = 0; kc < CHUNKS; ++kc)
                    st_shared_v4(s_base + (uint32_t)(kc * p.hbp + h) * 16u, q[kc][0], q[kc][1],
                                 q[kc][2], q[kc][3]);
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                if (withhold)
                    withhold = false;  // failure injection: this stage is never signalled
                else
                    mbar_arrive(smem_u32(&sh.full_a[stage]));
            }
            if (++stage == p.na) {
                stage = 0;
                phase ^= 1u;
            }
        }
    }
}

// Warps 0..3: TMEM accumulator -> float32 NCHW grad_in.
__device__ void role_epilogue(const TcParams &p, Shared &sh, uint32_t tmem, int q, int lane) {
    const int64_t HW = (int64_t)p.H * p.W;
    int acc = 0;
    uint32_t accph = 0;
    for (int64_t t = blockIdx.x; t < p.total_tiles; t += gridDim.x) {
        const Tile ti = decode_tile(p, t);
        const PhaseDesc &d = p.ph[ti.phase];
        const int lam = ti.mt * kTileM + q * 32 + lane;
        const int img = d.R * d.X;
        const int n = lam / img;
        const int rem = lam - n * img;
        const int a = rem / d.X;
        const int b = rem - a * d.X;
        const bool valid = n < p.N && a < d.Hr && b < d.Wr;
        const int ci0 = ti.nt * p.n_tile;
        const int ci_lim = p.Ci - ci0 < p.n_tile ? p.Ci - ci0 : p.n_tile;
        const int64_t out_off =
            valid ? (((int64_t)n * p.Ci + ci0) * p.H + (p.stride * a + d.rh)) * p.W +
                        (p.stride * b + d.rw)
                  : 0;
        float *out = p.grad_in + out_off;
        if (d.Jh == 0) {  // no tap reaches this phase: grad_in is zero there
            if (valid)
                for (int c = 0; c < ci_lim; ++c) out[c * HW] = 0.f;
            continue;
        }
        if (!wait_bar_warp(smem_u32(&sh.acc_full[acc]), accph, p, sh, lane)) return;
        tc_fence_after();
        const uint32_t taddr = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * p.n_tile);
        for (int c0 = 0; c0 < p.n_tile; c0 += 16) {
            float v[16];
            tmem_ld16(taddr + (uint32_t)c0, v);
            if (valid) {
#pragma unroll
                for (int jj = 0; jj < 16; ++jj)
                    if (c0 + jj < ci_lim) out[(int64_t)(c0 + jj) * HW] = v[jj];
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.acc_empty[acc]));
        if (++acc == 2) {
            acc = 0;
            accph ^= 1u;
        }
    }
}

template <int ESIZE, int CHUNKS>
__global__ void __launch_bounds__(kThreads, 1) dgrad_tc_kernel(const __grid_constant__ TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    Shared &sh = *reinterpret_cast<Shared *>(smem);
    const uint32_t a_base = smem_u32(smem + kBarrierBytes);
    const uint32_t b_base = a_base + (uint32_t)(p.na * p.a_stage_bytes);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.na; ++s) {
            mbar_init(smem_u32(&sh.full_a[s]), kAWarps);
            mbar_init(smem_u32(&sh.empty_a[s]), 1);
        }
        for (int s = 0; s < p.nb; ++s) {
            mbar_init(smem_u32(&sh.full_b[s]), 1);
            mbar_init(smem_u32(&sh.empty_b[s]), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(smem_u32(&sh.acc_full[s]), 1);
            mbar_init(smem_u32(&sh.acc_empty[s]), kEpiWarps);
        }
        mbar_init(smem_u32(&sh.w_full), 1);
        mbar_init(smem_u32(&sh.mma_done), 1);
        sh.abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(smem_u32(&sh.tmem_base), p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;

    if (warp == kBWarp) {
        if (lane == 0) role_weights(p, sh, b_base);
        __syncwarp();
    } else if (warp == kMmaWarp) {
        if (lane == 0) role_mma<ESIZE == 4>(p, sh, a_base, b_base, tmem);
        __syncwarp();
    } else if (warp >= kAWarp0) {
        role_gather<ESIZE, CHUNKS>(p, sh, a_base, warp - kAWarp0, lane);
    } else {
        role_epilogue(p, sh, tmem, warp, lane);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, p.tmem_cols);
    }
}

// Dynamic shared memory is raised once per device and variant to the full
// limit, so no attribute call happens on later launches (e.g. during stream
// capture).
template <int ESIZE, int CHUNKS>
int launch_variant(const TcParams &p, int grid, cudaStream_t st, int dev) {
    static std::atomic<uint64_t> configured{0};  // bit per device
    auto kern = dgrad_tc_kernel<ESIZE, CHUNKS>;
    const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
    if (!bit || !(configured.load() & bit)) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return (int)e;
        configured.fetch_or(bit);
    }
    kern<<<grid, kThreads, p.smem_bytes, st>>>(p);
    return (int)cudaGetLastError();
}

int sm_count(int dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace

int launch_tc(const Plan &plan, const void *grad_out, const void *packed, float *grad_in,
              void *stream) {
    TcParams p = plan.tc;
    p.grad_out = grad_out;
    p.packed = packed;
    p.grad_in = grad_in;
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return (int)de;
    const int sms = sm_count(dev);
    if (sms <= 0) return (int)cudaErrorInvalidDevice;
    // At least half the shared memory of an SM, so a second CTA can never be
    // co-resident and contend for tensor memory.
    if (p.smem_bytes < kSmemLimit / 2 + 1024) p.smem_bytes = kSmemLimit / 2 + 1024;
    const int grid = (int)(p.total_tiles < sms ? p.total_tiles : sms);
    if (grid <= 0) return (int)cudaSuccess;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int chunks = p.kc / (16 / plan.esize);
    if (plan.esize == 2) {
        if (chunks == 8) return launch_variant<2, 8>(p, grid, st, dev);
        if (chunks == 4) return launch_variant<2, 4>(p, grid, st, dev);
        return launch_variant<2, 2>(p, grid, st, dev);
    }
    if (chunks == 8) return launch_variant<4, 8>(p, grid, st, dev);
    if (chunks == 4) return launch_variant<4, 4>(p, grid, st, dev);
    return launch_variant<4, 2>(p, grid, st, dev);
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
