// mha_grad_v_tc.cuh -- tensor-core kernel of the attention dV (included by
// mha_grad_v.cu): bf16 / fp16 Q, K, dO with head_dim 64, sm_103a.
//
// Work unit: 128 key positions t of one KV head g (units ordered by key tile,
// so under a causal mask the units with the most query blocks start first),
// one persistent CTA per SM.  For every block of 128 query positions that can
// reach the unit and every head h of the group (a "step"):
//   GEMM1  S^T[t][pos] = K_tile (128 x 64) . Q_block^T        tcgen05 M128 N128 K16 x4
//   P^T[t][pos]        = exp(min(S^T / sqrt(64) - max[pos], 0) - log_sum[pos]), masked
//   GEMM2  dV[t][:]   += P^T (128 x 128) . dO_block (128 x 64)  tcgen05 M128 N64 K16 x8
// with dV accumulating in TMEM over all the unit's steps.
//   * warp 17 (one thread): TMA loads -- the unit's K tile, then per step the
//     Q and dO blocks of head h through 3-D views [q_seq][H][64] (box
//     [128][1][64], 128-byte swizzle): Q lands as GEMM1's K-major B operand,
//     dO as GEMM2's MN-major B operand (atoms of 8 positions x 64 elements);
//   * warp 16 (one thread): GEMM1 of step i into one of two TMEM score buffers,
//     then GEMM2 of step i - 1 (so the softmax of step i overlaps it);
//   * warps 0-15 (warp w: TMEM lane quadrant w % 4, lane = key t, query
//     columns 32 (w / 4) .. + 31 of the step): each loads the 32 (max,
//     log_sum) pairs of its columns one per lane (the next step's while this
//     one computes) and shares them by shuffles, reads its 32 scores from
//     TMEM, forms P with the page's clamp and the causal / window mask
//     (hardware ex2), rounds it to the input type and writes it into GEMM2's
//     K-major A operand (two 128-byte swizzled chunks of 64 positions); after
//     the unit's last step each warp stores its 16 columns of dV.
// Every wait is bounded; on timeout the kernel raises its error flag, drains
// its copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include "tc_helpers.cuh"

namespace mhadv {
namespace {

using namespace tch;

constexpr int kTcT = 128, kTcP = 128, kTcD = 64;  // keys per unit, queries per step, head_dim
constexpr int kTcStages = 4;
constexpr int kTcSoftWarps = 16, kTcMmaWarp = 16, kTcLoadWarp = 17;
constexpr int kTcThreads = 32 * 18;
constexpr uint32_t kTile = 128 * 128;  // bytes of a [128][64] 16-bit tile
constexpr uint32_t kOffK = 4096, kOffStage = kOffK + kTile;
constexpr uint32_t kOffP = kOffStage + kTcStages * 2 * kTile;
constexpr uint32_t kTcSmem = 1024 + kOffP + 2 * 2 * kTile;  // + 1 KB alignment slack
static_assert(kTcSmem <= 232448, "shared memory over the per-block limit");

struct TcArgs {
    CUtensorMap q_map, k_map, o_map;  // [len][heads][64] views, box [128][1][64], 128-byte swizzle
    const float *lse;
    float *dv;
    int q_seq, kv, nh, nkv, hpk, window, causal, t_tiles;
    int64_t units;
    float scale;
    uint32_t idesc1, idesc2;
    int f16;
    uint64_t wait_limit_ns;
};

struct TcCtl {
    uint64_t full[kTcStages], empty[kTcStages];
    uint64_t k_full, k_empty;
    uint64_t s_full[2], s_empty[2], p_ready[2], p_empty[2];
    uint64_t dv_full, dv_empty, mma_done;
    uint32_t tmem_base;
    int abort_flag;
};
static_assert(sizeof(TcCtl) <= 1024, "control block too large");

__device__ __noinline__ bool tc_wait_long(uint32_t bar, uint32_t parity, const TcArgs &a, TcCtl &c, bool honour) {
    const uint64_t t0 = now_ns();
    const uint64_t max_spins = a.wait_limit_ns / 16 + (1u << 20);
    for (uint64_t spin = 1;; ++spin) {
        if (bar_try(bar, parity)) return true;
        if (honour && *reinterpret_cast<volatile int *>(&c.abort_flag)) return false;
        if (((spin & 31u) == 0 && now_ns() - t0 > a.wait_limit_ns) || spin > max_spins) {
            *reinterpret_cast<volatile int *>(&c.abort_flag) = 1;
            atomicOr(&g_mha_error_word, 1u);
            return false;
        }
    }
}
__device__ __forceinline__ bool tc_wait(uint32_t bar, uint32_t parity, const TcArgs &a, TcCtl &c) {
    return bar_try(bar, parity) || tc_wait_long(bar, parity, a, c, true);
}
__device__ __forceinline__ void tc_drain(uint32_t bar, uint32_t parity, const TcArgs &a, TcCtl &c) {
    if (!bar_try(bar, parity)) tc_wait_long(bar, parity, a, c, false);
}
__device__ __forceinline__ bool tc_wait_warp(uint32_t bar, uint32_t parity, const TcArgs &a, TcCtl &c, int lane) {
    int ok = 0;
    if (lane == 0) ok = tc_wait(bar, parity, a, c) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// This CTA's k-th unit, or -1: units are dealt to the CTAs in rounds, every
// other round in reverse order, so that under a causal mask (units sorted by
// decreasing work) a CTA with a heavy unit in one round gets a light one in
// the next.
__device__ __forceinline__ int64_t unit_of(const TcArgs &a, int k) {
    const int64_t G = gridDim.x;
    const int64_t u = (int64_t)k * G + ((k & 1) ? G - 1 - blockIdx.x : blockIdx.x);
    return u < a.units ? u : -1;
}

// The query blocks of a unit: [lo, hi) in steps of 128 (then the heads of the group).
__device__ __forceinline__ void unit_range(const TcArgs &a, int64_t u, int &t0, int &g, int &lo, int &nblk) {
    t0 = (int)(u / a.nkv) * kTcT;
    g = (int)(u % a.nkv);
    const int t_last = t0 + kTcT - 1 < a.kv ? t0 + kTcT - 1 : a.kv - 1;
    lo = a.causal ? t0 : 0;
    int hi = a.q_seq;
    if (a.window > 0 && t_last + a.window < hi) hi = t_last + a.window;
    nblk = hi > lo ? (hi - lo + kTcP - 1) / kTcP : 0;
}

__device__ void tc_role_load(const TcArgs &a, TcCtl &c, uint32_t smem) {
    int s = 0;
    uint32_t ph = 0, kph = 0;
    int64_t issued = 0, k_issued = 0;
    bool aborted = false;
    for (int k = 0; !aborted; ++k) {
        const int64_t u = unit_of(a, k);
        if (u < 0) break;
        int t0, g, lo, nblk;
        unit_range(a, u, t0, g, lo, nblk);
        if (nblk == 0) continue;  // no query reaches these keys: nothing to load
        if (!tc_wait(su32(&c.k_empty), kph ^ 1u, a, c)) break;
        bar_expect_tx(su32(&c.k_full), kTile);
        tma_load_3d(smem + kOffK, &a.k_map, 0, g, t0, su32(&c.k_full));
        ++k_issued;
        kph ^= 1u;
        for (int b = 0; b < nblk && !aborted; ++b)
            for (int r = 0; r < a.hpk; ++r) {
                if (!tc_wait(su32(&c.empty[s]), ph ^ 1u, a, c)) {
                    aborted = true;
                    break;
                }
                const int h = g * a.hpk + r, p0 = lo + b * kTcP;
                const uint32_t st = smem + kOffStage + (uint32_t)s * 2u * kTile;
                bar_expect_tx(su32(&c.full[s]), 2 * kTile);
                tma_load_3d(st, &a.q_map, 0, h, p0, su32(&c.full[s]));
                tma_load_3d(st + kTile, &a.o_map, 0, h, p0, su32(&c.full[s]));
                ++issued;
                if (++s == kTcStages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
    }
    // Copies still landing must finish before the CTA exits.
    const int64_t k_end = issued < kTcStages ? issued : kTcStages;
    for (int64_t q = issued - k_end; q < issued; ++q)
        tc_drain(su32(&c.full[q % kTcStages]), (uint32_t)((q / kTcStages) & 1), a, c);
    if (k_issued) tc_drain(su32(&c.k_full), (uint32_t)((k_issued - 1) & 1), a, c);
}

__device__ void tc_role_mma(const TcArgs &a, TcCtl &c, uint32_t smem, uint32_t tmem) {
    int s = 0, sb = 0;
    uint32_t ph = 0, sph = 0, kph = 0, dph = 0;
    int64_t gstep = 0;  // this CTA's steps so far: score / P buffer gstep % 2, its use gstep / 2
    bool aborted = false;
    for (int k = 0; !aborted; ++k) {
        const int64_t u = unit_of(a, k);
        if (u < 0) break;
        int t0, g, lo, nblk;
        unit_range(a, u, t0, g, lo, nblk);
        const int n = nblk * a.hpk;
        if (n == 0) continue;
        if (!tc_wait(su32(&c.k_full), kph, a, c)) break;
        kph ^= 1u;
        tc_after();
        const uint64_t kd = desc_k(smem + kOffK);
        int s_prev = 0, sb_prev = 0;
        int64_t g_prev = 0;
        for (int i = 0; i <= n && !aborted; ++i) {
            if (i < n) {  // GEMM1 of step i
                if (!tc_wait(su32(&c.full[s]), ph, a, c) || !tc_wait(su32(&c.s_empty[sb]), sph ^ 1u, a, c)) {
                    aborted = true;
                    break;
                }
                tc_after();
                const uint64_t qd = desc_k(smem + kOffStage + (uint32_t)s * 2u * kTile);
#pragma unroll
                for (int k16 = 0; k16 < 4; ++k16)
                    tc_mma_f16(tmem + (uint32_t)(sb * kTcP), kd + 2u * k16, qd + 2u * k16, a.idesc1, k16 != 0);
                tc_commit_to(su32(&c.s_full[sb]));
                if (i == n - 1) tc_commit_to(su32(&c.k_empty));  // the unit's last read of its K tile
            }
            if (i >= 1) {  // GEMM2 of step i - 1
                const int j = i - 1;
                if (!tc_wait(su32(&c.p_ready[sb_prev]), (uint32_t)((g_prev >> 1) & 1), a, c) ||
                    (j == 0 && !tc_wait(su32(&c.dv_empty), dph ^ 1u, a, c))) {
                    aborted = true;
                    break;
                }
                tc_after();
                const uint32_t pbuf = smem + kOffP + (uint32_t)sb_prev * 2u * kTile;
                const uint64_t od = desc_mn(smem + kOffStage + (uint32_t)s_prev * 2u * kTile + kTile, 1024u, 1024u);
#pragma unroll
                for (int k16 = 0; k16 < 8; ++k16)
                    tc_mma_f16(tmem + 2u * kTcP, desc_k(pbuf + (uint32_t)(k16 >> 2) * kTile) + 2u * (k16 & 3),
                               od + 128u * k16, a.idesc2, (j | k16) != 0);
                tc_commit_to(su32(&c.p_empty[sb_prev]));
                tc_commit_to(su32(&c.empty[s_prev]));
            }
            if (i < n) {
                s_prev = s;
                sb_prev = sb;
                g_prev = gstep++;
                if (++s == kTcStages) {
                    s = 0;
                    ph ^= 1u;
                }
                if (++sb == 2) {
                    sb = 0;
                    sph ^= 1u;
                }
            }
        }
        if (aborted) break;
        tc_commit_to(su32(&c.dv_full));
        dph ^= 1u;
    }
    tc_commit_to(su32(&c.mma_done));
    tc_drain(su32(&c.mma_done), 0, a, c);
}

__device__ __forceinline__ float fast_exp2(float x) {  // the SFU's 2^x (x <= 0 here)
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Softmax and dV store warps: warp w holds key rows t0 + 32 (w % 4) + lane and
// query columns 32 (w / 4) .. + 31 of every step.
__device__ void tc_role_soft(const TcArgs &a, TcCtl &c, uint32_t smem, uint32_t tmem, int w, int lane) {
    const int qd = w & 3, cq = w >> 2;
    const int u = 32 * qd + lane;  // key row within the unit
    const bool f16 = a.f16 != 0;
    const float l2e = 1.4426950408889634f;  // log2(e): exp(x) = 2^(x log2(e))
    int sb = 0;
    uint32_t sph = 0, dph = 0;
    int64_t steps = 0;  // this CTA's steps so far (P buffer parity)
    // (max, log_sum) of query column 32 cq + lane of a step, times log2(e).
    auto load_stats = [&](int p0, int h) {
        const int pos = p0 + 32 * cq + lane;
        float2 st = make_float2(0.f, 0.f);
        if (pos < a.q_seq) st = __ldg(reinterpret_cast<const float2 *>(a.lse + ((int64_t)pos * a.nh + h) * 2));
        return make_float2(st.x * l2e, st.y * l2e);
    };
    for (int k = 0;; ++k) {
        const int64_t un = unit_of(a, k);
        if (un < 0) break;
        int t0, g, lo, nblk;
        unit_range(a, un, t0, g, lo, nblk);
        const int t = t0 + u;
        const int start = a.causal ? t : 0;
        int end = a.q_seq;
        if (a.window > 0 && t + a.window < end) end = t + a.window;
        const bool t_live = t < a.kv;
        const int n = nblk * a.hpk;
        float2 st_next = n > 0 ? load_stats(lo, g * a.hpk) : make_float2(0.f, 0.f);
        for (int i = 0; i < n; ++i, ++steps) {
            const int b = i / a.hpk, r = i - b * a.hpk;
            const int h = g * a.hpk + r, p0 = lo + b * kTcP;
            const float2 st_mine = st_next;
            if (i + 1 < n) {
                const int b1 = (i + 1) / a.hpk;
                st_next = load_stats(lo + b1 * kTcP, g * a.hpk + (i + 1 - b1 * a.hpk));
            }
            if (!tc_wait_warp(su32(&c.s_full[sb]), sph, a, c, lane)) return;
            tc_after();
            uint32_t v[32];
            tc_ld_32x32(tmem + ((uint32_t)(32 * qd) << 16) + (uint32_t)(sb * kTcP + 32 * cq), v);
            tc_wait_ld(v);
            uint32_t pk[16];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
                float pr[2];
#pragma unroll
                for (int z = 0; z < 2; ++z) {
                    const int pos = p0 + 32 * cq + e + z;
                    const float mx = __shfl_sync(0xffffffffu, st_mine.x, e + z);
                    const float ls = __shfl_sync(0xffffffffu, st_mine.y, e + z);
                    const float x = fminf(__uint_as_float(v[e + z]) * (a.scale * l2e) - mx, 0.f) - ls;
                    pr[z] = (t_live && pos >= start && pos < end) ? fast_exp2(x) : 0.f;
                }
                if (f16) {
                    const __half2 hh = __floats2half2_rn(pr[0], pr[1]);
                    pk[e >> 1] = *reinterpret_cast<const uint32_t *>(&hh);
                } else {
                    const __nv_bfloat162 hh = __floats2bfloat162_rn(pr[0], pr[1]);
                    pk[e >> 1] = *reinterpret_cast<const uint32_t *>(&hh);
                }
            }
            tc_before();
            __syncwarp();
            if (lane == 0) bar_arrive(su32(&c.s_empty[sb]));  // scores read: the buffer may be refilled
            if (!tc_wait_warp(su32(&c.p_empty[sb]), (uint32_t)(((steps >> 1) & 1) ^ 1), a, c, lane)) return;
            // Columns 32 cq .. + 31: chunk cq / 2 of the row, 16-byte pieces
            // 4 (cq % 2) .. + 3 at their swizzled slots.
            const uint32_t row = smem + kOffP + (uint32_t)sb * 2u * kTile + (uint32_t)(cq >> 1) * kTile + (uint32_t)u * 128u;
#pragma unroll
            for (int pc = 0; pc < 4; ++pc) {
                const int piece = 4 * (cq & 1) + pc;
                sts128(row + (uint32_t)((piece ^ (u & 7)) << 4), pk[4 * pc], pk[4 * pc + 1], pk[4 * pc + 2],
                       pk[4 * pc + 3]);
            }
            fence_async_proxy();  // GEMM2 (async proxy) reads the P these threads wrote
            __syncwarp();
            if (lane == 0) bar_arrive(su32(&c.p_ready[sb]));
            if (++sb == 2) {
                sb = 0;
                sph ^= 1u;
            }
        }
        if (n == 0) {  // no query reaches these keys: dV is zero
            if (t_live)
                for (int d = 16 * cq; d < 16 * cq + 16; d += 4)
                    *reinterpret_cast<float4 *>(a.dv + ((int64_t)t * a.nkv + g) * kTcD + d) = make_float4(0.f, 0.f, 0.f, 0.f);
            continue;
        }
        // dV of the unit: this warp's 16 columns (TMEM 256 + 16 cq ..) of lane u.
        if (!tc_wait_warp(su32(&c.dv_full), dph, a, c, lane)) return;
        dph ^= 1u;
        tc_after();
        uint32_t v[32];
        tc_ld_32x32(tmem + ((uint32_t)(32 * qd) << 16) + 2u * kTcP + (uint32_t)(16 * cq), v);  // 32 columns read,
        tc_wait_ld(v);                                                                            // 16 used
        if (t_live) {
            float4 *out = reinterpret_cast<float4 *>(a.dv + ((int64_t)t * a.nkv + g) * kTcD + 16 * cq);
#pragma unroll
            for (int e = 0; e < 4; ++e)
                out[e] = make_float4(__uint_as_float(v[4 * e]), __uint_as_float(v[4 * e + 1]),
                                     __uint_as_float(v[4 * e + 2]), __uint_as_float(v[4 * e + 3]));
        }
        tc_before();
        __syncwarp();
        if (lane == 0) bar_arrive(su32(&c.dv_empty));
    }
}

__global__ void __launch_bounds__(kTcThreads, 1) mha_grad_v_tc_kernel(const __grid_constant__ TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t smem = (su32(smem_raw) + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (smem - su32(smem_raw));
    TcCtl &c = *reinterpret_cast<TcCtl *>(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            bar_init(su32(&c.full[s]), 1);
            bar_init(su32(&c.empty[s]), 1);
        }
        bar_init(su32(&c.k_full), 1);
        bar_init(su32(&c.k_empty), 1);
        for (int b = 0; b < 2; ++b) {
            bar_init(su32(&c.s_full[b]), 1);
            bar_init(su32(&c.s_empty[b]), kTcSoftWarps);
            bar_init(su32(&c.p_ready[b]), kTcSoftWarps);
            bar_init(su32(&c.p_empty[b]), 1);
        }
        bar_init(su32(&c.dv_full), 1);
        bar_init(su32(&c.dv_empty), kTcSoftWarps);
        bar_init(su32(&c.mma_done), 1);
        c.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kTcMmaWarp) tc_alloc(su32(&c.tmem_base), 512);
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = c.tmem_base;
    if (warp == kTcLoadWarp && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.q_map)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.k_map)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.o_map)) : "memory");
    }
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (warp == kTcLoadWarp) {
        if (lane == 0) tc_role_load(a, c, smem);
        __syncwarp();
    } else if (warp == kTcMmaWarp) {
        if (lane == 0) tc_role_mma(a, c, smem, tmem);
        __syncwarp();
    } else {
        tc_role_soft(a, c, smem, tmem, warp, lane);
    }
    tc_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_after();
        tc_dealloc(tmem, 512);
    }
}

bool tc_applies(const void *q, const void *k, const void *go, const float *lse, const float *dv,
                const mha_grad_v_params *p, int dtype) {
    return dtype != DGRAD_F32 && p->head_dim == (uint32_t)kTcD && aligned(q, 16) && aligned(k, 16) &&
           aligned(go, 16) && aligned(lse, 8) && aligned(dv, 16);
}

PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            ptr = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }();
    return fn;
}

// [len][heads][64] 16-bit tensor, box [128][1][64], 128-byte swizzle.
bool encode_heads_map(CUtensorMap *m, const void *ptr, int len, int heads) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = tc_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)kTcD, (cuuint64_t)heads, (cuuint64_t)len};
    const cuuint64_t strides[2] = {(cuuint64_t)kTcD * 2, (cuuint64_t)heads * kTcD * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kTcD, 1, 128};
    const cuuint32_t es[3] = {1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int launch_tc(const void *q, const void *k, const void *go, const float *lse, float *dv, const mha_grad_v_params *p,
              int dtype, cudaStream_t st) {
    TcArgs a{};
    a.q_seq = (int)p->q_seq;
    a.causal = p->kv_seq == 0;
    a.kv = a.causal ? a.q_seq : (int)p->kv_seq;
    a.nh = (int)p->num_heads;
    a.nkv = (int)p->num_kv_heads;
    a.hpk = a.nh / a.nkv;
    a.window = (int)p->window_size;
    a.t_tiles = (a.kv + kTcT - 1) / kTcT;
    a.units = (int64_t)a.t_tiles * a.nkv;
    a.scale = 1.0f / sqrtf((float)kTcD);
    a.lse = lse;
    a.dv = dv;
    a.f16 = dtype == DGRAD_F16 ? 1 : 0;
    const uint32_t fmt = dtype == DGRAD_BF16 ? 1u : 0u;
    // D float32, A and B of the input type; GEMM1: both K-major, N = 128;
    // GEMM2: B (dO) MN-major, N = 64; M = 128.
    a.idesc1 = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(kTcP >> 3) << 17) | ((uint32_t)(kTcT >> 4) << 24);
    a.idesc2 = (1u << 4) | (fmt << 7) | (fmt << 10) | (1u << 16) | ((uint32_t)(kTcD >> 3) << 17) |
               ((uint32_t)(kTcT >> 4) << 24);
    a.wait_limit_ns = 2000000000ull;
    if (!encode_heads_map(&a.q_map, q, a.q_seq, a.nh) || !encode_heads_map(&a.k_map, k, a.kv, a.nkv) ||
        !encode_heads_map(&a.o_map, go, a.q_seq, a.nh))
        return DGRAD_ERR_UNSUPPORTED;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGRAD_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return DGRAD_ERR_CUDA;
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
    if (!bit || !(configured.load() & bit)) {
        if (cudaFuncSetAttribute(mha_grad_v_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem) !=
            cudaSuccess)
            return DGRAD_ERR_CUDA;
        configured.fetch_or(bit);
    }
    const int grid = (int)(a.units < sms ? a.units : sms);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = kTcSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, mha_grad_v_tc_kernel, a) == cudaSuccess ? DGRAD_OK : DGRAD_ERR_CUDA;
}

}  // namespace
}  // namespace mhadv
