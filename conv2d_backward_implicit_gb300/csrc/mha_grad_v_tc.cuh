// mha_grad_v_tc.cuh -- tensor-core kernel of the attention dV (included by
// mha_grad_v.cu): bf16 / fp16 Q, K, dO with head_dim 64, sm_103a.
//
// Work unit: 128 key positions t of one KV head g (units ordered by key tile,
// so under a causal mask the units with the most query blocks come first,
// dealt to the persistent CTAs, one per SM, in rounds of alternating
// direction).  For every block of 128 query positions that can reach the unit
// and every head h of the group (a "step"):
//   GEMM1  S^T[t][pos] = K_tile (128 x 64) . Q_block^T        tcgen05 M128 N128 K16 x4
//   P^T[t][pos]        = exp(min(S^T / sqrt(64) - max[pos], 0) - log_sum[pos]), masked
//   GEMM2  dV[t][:]   += P^T (128 x 128) . dO_block (128 x 64)  tcgen05 M128 N64 K16 x8
// with dV accumulating in TMEM over all the unit's steps, one partial sum per
// step parity.
//   * warps 18-19 (one thread each): TMA loads of the Q and dO blocks of head
//     h through 3-D views [q_seq][H][64] (box [128][1][64], 128-byte swizzle):
//     Q lands as GEMM1's K-major B operand, dO as GEMM2's MN-major B operand
//     (atoms of 8 positions x 64 elements).  One thread's copies complete one
//     after another (about 1.1K cycles each) while different warps' overlap, so
//     warp 18 loads the Q blocks and the unit's K tile, warp 19 the dO blocks
//     and with each the forward statistics of its positions (for the head pair
//     of h, through a [q_seq][2 H] float32 view);
//   * warps 16 and 17 (converged, lane 0 issuing), one per step parity: GEMM1
//     of the parity's next step (into its TMEM scores) ahead of GEMM2 of its
//     current one (P^T from TMEM as the A operand, into its dV partial sum),
//     each warp with its own waits and commits;
//   * warps 0-15, two groups of 8 taking alternate steps (warp w: TMEM lane
//     quadrant w % 4, lane = key t, query columns 64 ((w / 4) % 2) .. + 63):
//     fold the forward statistics of their columns, read their scores from
//     TMEM, form P with the page's clamp and the causal / window mask
//     (hardware ex2), round it to the input type and store it, two values per
//     column, into the parity's TMEM P buffer; after the unit's last step each
//     warp adds the two parities' partial sums for 16 columns of dV and stores
//     them.
// Every wait is bounded; on timeout the kernel raises its error flag, drains
// its copies and MMAs, frees TMEM and returns.
#include <cudaTypedefs.h>

#include "tc_helpers.cuh"

namespace mhadv {
namespace {

using namespace tch;

constexpr int kTcT = 128, kTcP = 128, kTcD = 64;  // keys per unit, queries per step, head_dim
constexpr int kTcStages = 4;
constexpr int kTcSoftWarps = 16, kTcMmaWarp = 16, kTcMma2Warp = 17, kTcLoadWarp = 18, kTcLoadWarps = 2;
constexpr int kTcThreads = 32 * (kTcLoadWarp + kTcLoadWarps);
constexpr int kTcLoadPar = kTcLoadWarps / 2;  // step parities (one Q and one dO warp each)
static_assert(kTcLoadWarps % 2 == 0 && kTcStages % kTcLoadPar == 0, "load warps own whole stages");
constexpr uint32_t kTile = 128 * 128;  // bytes of a [128][64] 16-bit tile
// Control block [0, 1 KB); per softmax warp 512 bytes: its 64 folded
// (b, -l) pairs; then the K tile, the Q and dO rings (1 KB aligned for the
// 128-byte swizzle) and the statistics ring: beside each dO slot, (max,
// log_sum) of its 128 positions for an even / odd head pair.
constexpr uint32_t kOffStats = 1024, kStatsBytes = 512;
constexpr uint32_t kOffK = 9216;
static_assert(kOffStats + kTcSoftWarps * kStatsBytes <= kOffK, "statistics overlap the K tile");
constexpr uint32_t kOffQ = kOffK + kTile, kOffO = kOffQ + kTcStages * kTile;
constexpr uint32_t kOffL = kOffO + kTcStages * kTile, kLseBox = 128 * 16;  // [128][4] float32 per slot
// Tensor memory columns, one set per step parity p: scores S^T (128
// float32) at 128 p, a dV partial sum (64 float32) at 256 + 64 p, P^T (64
// columns, each two 16-bit values) at 384 + 64 p.
constexpr uint32_t kColS = 0, kColDv = 256, kColP = 384;
constexpr uint32_t kTcSmem = 1024 + kOffL + kTcStages * kLseBox;  // + 1 KB alignment slack
static_assert(kOffK % 1024 == 0, "operand tiles must be 1 KB aligned");
static_assert(kTcSmem <= 232448, "shared memory over the per-block limit");

struct TcArgs {
    CUtensorMap q_map, k_map, o_map;  // [len][heads][64] views, box [128][1][64], 128-byte swizzle
    CUtensorMap l_map;                // LSE as [q_seq][2 H] float32, box [128][4] (two heads' pairs)
    const float *lse;
    float *dv;
    int q_seq, kv, nh, nkv, hpk, window, causal, t_tiles;
    int64_t units;
    float scale;
    uint32_t idesc1, idesc2;
    uint64_t wait_limit_ns;
};

struct TcCtl {
    uint64_t full_q[kTcStages], full_o[kTcStages], empty_q[kTcStages], empty_o[kTcStages];
    uint64_t k_full, k_empty;
    uint64_t s_full[2], s_empty[2], p_ready[2], p_empty[2];
    uint64_t dv_full[2], dv_empty, mma_done[2];
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

// Load warp lw: tensor lw % 2 (0: Q, 1: dO) of the steps whose index in this
// CTA is lw / 2 modulo kTcLoadPar; warp 0 also loads K.
__device__ void tc_role_load(const TcArgs &a, TcCtl &c, uint32_t smem, int lw) {
    const int tensor = lw & 1, par = lw >> 1;
    const CUtensorMap *map = tensor ? &a.o_map : &a.q_map;
    uint64_t *full = tensor ? c.full_o : c.full_q;
    uint64_t *empty = tensor ? c.empty_o : c.empty_q;
    const uint32_t ring = smem + (tensor ? kOffO : kOffQ);
    int64_t gi = 0;  // this CTA's steps so far
    int64_t k_issued = 0, last = -1;
    uint32_t kph = 0;
    bool aborted = false;
    for (int k = 0; !aborted; ++k) {
        const int64_t u = unit_of(a, k);
        if (u < 0) break;
        int t0, g, lo, nblk;
        unit_range(a, u, t0, g, lo, nblk);
        if (nblk == 0) continue;  // no query reaches these keys: nothing to load
        if (lw == 0) {
            if (!tc_wait(su32(&c.k_empty), kph ^ 1u, a, c)) break;
            bar_expect_tx(su32(&c.k_full), kTile);
            tma_load_3d(smem + kOffK, &a.k_map, 0, g, t0, su32(&c.k_full));
            ++k_issued;
            kph ^= 1u;
        }
        for (int b = 0; b < nblk && !aborted; ++b)
            for (int r = 0; r < a.hpk; ++r, ++gi) {
                if (gi % kTcLoadPar != par) continue;
                const int s = (int)(gi % kTcStages);
                if (!tc_wait(su32(&empty[s]), (uint32_t)(((gi / kTcStages) & 1) ^ 1), a, c)) {
                    aborted = true;
                    break;
                }
                const int h = g * a.hpk + r, p0 = lo + b * kTcP;
                bar_expect_tx(su32(&full[s]), tensor ? kTile + kLseBox : kTile);
                tma_load_3d(ring + (uint32_t)s * kTile, map, 0, h, p0, su32(&full[s]));
                if (tensor) tma_load_2d(smem + kOffL + (uint32_t)s * kLseBox, &a.l_map, 4 * (h >> 1), p0, su32(&full[s]));
                last = gi;
            }
    }
    // Copies still landing must finish before the CTA exits: this warp owns
    // kTcStages / kTcLoadPar stages, so only its last that many can be in flight.
    for (int j = 0; j < kTcStages / kTcLoadPar; ++j) {
        const int64_t q = last - (int64_t)j * kTcLoadPar;
        if (q >= 0) tc_drain(su32(&full[q % kTcStages]), (uint32_t)((q / kTcStages) & 1), a, c);
    }
    if (k_issued) tc_drain(su32(&c.k_full), (uint32_t)((k_issued - 1) & 1), a, c);
}

// The MMA issue, split by step parity: warp 16 + p issues GEMM1 and GEMM2 of
// this CTA's steps gs with gs % 2 = p (a thread's tcgen05 commit tracks only
// its own MMAs, and the two parities share no accumulator; issuing the small
// MMAs is what bounds one thread).  The whole warp runs the loop (waits and
// descriptors warp-uniform); lane 0 alone issues the MMAs and commits.  GEMM1
// of a parity's next step is issued as soon as the softmax has read the
// current step's scores, before GEMM2 of the current step.  Ring slots and
// barrier phases follow gs: Q / dO slot gs % kTcStages; the parity's scores,
// P and dV columns and barriers once per own step.
__device__ void tc_role_mma(const TcArgs &a, TcCtl &c, uint32_t smem, uint32_t tmem, int par, uint32_t leader) {
    uint32_t kph = 0, dph = 0, ph = 0;  // K tile, dV (per unit), own-step phases
    uint32_t base = 0;                  // this CTA's steps before the current unit
    const uint32_t s_col = tmem + kColS + 128u * (uint32_t)par, dv_col = tmem + kColDv + 64u * (uint32_t)par;
    const uint32_t p_col = tmem + kColP + 64u * (uint32_t)par;
    bool ok = true;
    auto gemm1 = [&](uint32_t gs, uint64_t kd, uint32_t phase) {
        const uint32_t s = gs % kTcStages;
        if (!tc_wait(su32(&c.full_q[s]), (gs / kTcStages) & 1u, a, c) ||
            !tc_wait(su32(&c.s_empty[par]), phase ^ 1u, a, c))  // scores of the previous own step read
            return false;
        tc_after();
        const uint64_t qd = desc_k(smem + kOffQ + s * kTile);
#pragma unroll
        for (int k16 = 0; k16 < 4; ++k16)
            tc_mma_f16_if(s_col, kd + 2u * k16, qd + 2u * k16, a.idesc1, k16 != 0, leader);
        tc_commit_to_if(su32(&c.s_full[par]), leader);
        tc_commit_to_if(su32(&c.empty_q[s]), leader);
        return true;
    };
    auto gemm2 = [&](uint32_t gs, uint32_t phase, bool first) {
        const uint32_t s = gs % kTcStages;
        if (!tc_wait(su32(&c.full_o[s]), (gs / kTcStages) & 1u, a, c) ||
            !tc_wait(su32(&c.p_ready[par]), phase, a, c) ||
            (first && !tc_wait(su32(&c.dv_empty), dph ^ 1u, a, c)))
            return false;
        tc_after();
        const uint64_t od = desc_mn(smem + kOffO + s * kTile, 1024u, 1024u);
#pragma unroll
        for (int k16 = 0; k16 < 8; ++k16)  // A = P^T from tensor memory, 8 columns (16 positions) per K step
            tc_mma_f16_ts_if(dv_col, p_col + 8u * k16, od + 128u * k16, a.idesc2, !first || k16 != 0, leader);
        tc_commit_to_if(su32(&c.p_empty[par]), leader);
        tc_commit_to_if(su32(&c.empty_o[s]), leader);
        return true;
    };
    for (int k = 0; ok; ++k) {
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
        const int i0 = (int)((base ^ (uint32_t)par) & 1u);  // this parity's first step of the unit
        if (i0 < n) ok = gemm1(base + (uint32_t)i0, kd, ph);
        for (int i = i0; i < n && ok; i += 2) {
            if (i + 2 < n) ok = gemm1(base + (uint32_t)i + 2, kd, ph ^ 1u);
            ok = ok && gemm2(base + (uint32_t)i, ph, i == i0);
            ph ^= 1u;
        }
        if (!ok) break;
        // Both parities' last reads of the K tile are done once both commit
        // (with no GEMM1 in this unit, the commit covers earlier MMAs only).
        tc_commit_to_if(su32(&c.k_empty), leader);
        if (i0 < n) tc_commit_to_if(su32(&c.dv_full[par]), leader);
        dph ^= 1u;
        base += (uint32_t)n;
    }
    tc_commit_to_if(su32(&c.mma_done[par]), leader);
    tc_drain(su32(&c.mma_done[par]), 0, a, c);
}

__device__ __forceinline__ float fast_exp2(float x) {  // the SFU's 2^x (x <= 0 here)
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// P^T of one 32-column chunk of a warp's scores v (this lane's row): 2^x with
// x = min(S c - b, -l) from the folded pairs at `pairs`, masked per column
// when kMasked (row t, columns cc ..; kept where start <= pos < end and the
// row exists), rounded to T and packed two columns per 32-bit value.
template <bool kF16, bool kMasked>
__device__ __forceinline__ void softmax_chunk(const uint32_t (&v)[32], uint32_t pairs, float cs, int cc, int start,
                                              int end, bool t_live, uint32_t (&pk)[16]) {
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        const uint4 bl = lds128(pairs + (uint32_t)e * 8u);  // (b, -l) of columns e, e + 1
        float pr[2];
        pr[0] = fast_exp2(fminf(fmaf(__uint_as_float(v[e]), cs, -__uint_as_float(bl.x)), __uint_as_float(bl.y)));
        pr[1] = fast_exp2(fminf(fmaf(__uint_as_float(v[e + 1]), cs, -__uint_as_float(bl.z)), __uint_as_float(bl.w)));
        if (kMasked) {
#pragma unroll
            for (int z = 0; z < 2; ++z) {
                const int pos = cc + e + z;
                if (!(t_live && pos >= start && pos < end)) pr[z] = 0.f;
            }
        }
        if (kF16) {
            const __half2 hh = __floats2half2_rn(pr[0], pr[1]);
            pk[e >> 1] = *reinterpret_cast<const uint32_t *>(&hh);
        } else {
            const __nv_bfloat162 hh = __floats2bfloat162_rn(pr[0], pr[1]);
            pk[e >> 1] = *reinterpret_cast<const uint32_t *>(&hh);
        }
    }
}

// Softmax and dV store warps, two groups of 8 taking alternate steps (group
// gs % 2 takes this CTA's step gs, with scores buffer gs % 2), so that one
// group's waits and stores overlap the other's exponentials.  Warp w of group
// w / 8 holds key rows t0 + 32 (w % 4) + lane and query columns 64 ((w / 4) % 2)
// .. + 63 of its steps, in two chunks of 32.  Lane l takes the forward
// statistics of columns l and 32 + l of its 64 from the step's slot of the
// statistics ring (landed with dO, so valid until GEMM2 has run), folds them
// and shares them through the warp's 64 folded pairs.  With c = log2(e) /
// sqrt(64), m = max log2(e) and l = log_sum log2(e) of a column, the page's
// P = exp(min(s - max, 0) - log_sum) is 2^x with x = min(S c - (m + l), -l):
// one FMA, one min and the SFU's 2^x per score.
template <bool kF16>
__device__ void tc_role_soft(const TcArgs &a, TcCtl &c, uint32_t smem, uint32_t tmem, int w, int lane) {
    const int qd = w & 3, ch = (w >> 2) & 1, gp = w >> 3, cq = w >> 2;
    const int u = 32 * qd + lane;  // key row within the unit
    const float l2e = 1.4426950408889634f;  // log2(e): exp(x) = 2^(x log2(e))
    const float cs = a.scale * l2e;
    const uint32_t stats = smem + kOffStats + (uint32_t)w * kStatsBytes;  // this warp's 64 (b, -l) pairs
    const uint32_t lane_tm = (uint32_t)(32 * qd) << 16;
    uint32_t own = 0;             // phase of this group's scores / P barriers (once per own step)
    uint32_t dph0 = 0, dph1 = 0;  // phases of the two parities' dV barriers
    uint32_t base = 0;            // this CTA's steps before the current unit
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
        int i = (int)((base ^ (uint32_t)gp) & 1u);  // this group's first step of the unit
        int qb = i / a.hpk, r = i - qb * a.hpk;     // its query block and head of the group
        for (; i < n; i += 2) {
            const uint32_t gs = base + (uint32_t)i;
            const int c0 = lo + qb * kTcP + 64 * ch;  // this warp's first query column
            const uint32_t slot = gs % kTcStages;
            if (!tc_wait(su32(&c.full_o[slot]), (gs / kTcStages) & 1u, a, c)) return;
            {
                // (max, log_sum) of columns c0 + lane and c0 + 32 + lane, head h of the pair (h & 1)
                const uint32_t src = smem + kOffL + slot * kLseBox + (uint32_t)(64 * ch + lane) * 16u +
                                     (uint32_t)((g * a.hpk + r) & 1) * 8u;
                float2 s0, s1;
                asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(s0.x), "=f"(s0.y) : "r"(src) : "memory");
                asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(s1.x), "=f"(s1.y) : "r"(src + 512u) : "memory");
                __syncwarp();  // the previous step's readers of the folded pairs are done
                const float l0 = s0.y * l2e, l1 = s1.y * l2e;
                asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(stats + (uint32_t)lane * 8u), "f"(fmaf(s0.x, l2e, l0)),
                             "f"(-l0)
                             : "memory");
                asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(stats + 256u + (uint32_t)lane * 8u),
                             "f"(fmaf(s1.x, l2e, l1)), "f"(-l1)
                             : "memory");
                __syncwarp();
            }
            if (!tc_wait(su32(&c.s_full[gp]), own, a, c)) return;
            tc_after();
#pragma unroll
            for (int kc = 0; kc < 2; ++kc) {
                uint32_t v[32];
                tc_ld_32x32(tmem + lane_tm + kColS + (uint32_t)(gp * kTcP + 64 * ch + 32 * kc), v);
                tc_wait_ld(v);
                if (kc == 1) {  // both chunks read: the scores buffer may be refilled
                    tc_before();
                    __syncwarp();
                    if (lane == 0) bar_arrive(su32(&c.s_empty[gp]));
                }
                const int cc = c0 + 32 * kc;
                // Every column of this chunk inside the mask: no per-score test.
                const bool whole = t_live && start <= cc && cc + 31 < end;
                uint32_t pk[16];
                if (whole)
                    softmax_chunk<kF16, false>(v, stats + 256u * (uint32_t)kc, cs, cc, start, end, t_live, pk);
                else
                    softmax_chunk<kF16, true>(v, stats + 256u * (uint32_t)kc, cs, cc, start, end, t_live, pk);
                if (kc == 0) {  // the parity's P buffer free (GEMM2 of its previous step has run)
                    if (!tc_wait(su32(&c.p_empty[gp]), own ^ 1u, a, c)) return;
                    tc_after();
                }
                // P^T of this warp's rows, query columns 64 ch + 32 kc .. + 31:
                // tensor memory columns 32 ch + 16 kc .. + 15 of the parity's P buffer.
                tc_st_32x16(tmem + lane_tm + kColP + 64u * (uint32_t)gp + (uint32_t)(32 * ch + 16 * kc), pk);
            }
            tc_wait_st();
            tc_before();
            __syncwarp();
            if (lane == 0) bar_arrive(su32(&c.p_ready[gp]));
            own ^= 1u;
            r += 2;
            while (r >= a.hpk) {
                r -= a.hpk;
                ++qb;
            }
        }
        base += (uint32_t)n;
        if (n == 0) {  // no query reaches these keys: dV is zero
            if (t_live)
                for (int d = 16 * cq; d < 16 * cq + 16; d += 4)
                    *reinterpret_cast<float4 *>(a.dv + ((int64_t)t * a.nkv + g) * kTcD + d) = make_float4(0.f, 0.f, 0.f, 0.f);
            continue;
        }
        // dV of the unit: the sum of the two parities' partial sums (a parity
        // without steps in the unit has none), this warp's 16 columns of lane u.
        float acc[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[e] = 0.f;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            if ((int)(((base - (uint32_t)n) ^ (uint32_t)p) & 1u) >= n) continue;
            if (!tc_wait(su32(&c.dv_full[p]), p ? dph1 : dph0, a, c)) return;
            if (p) dph1 ^= 1u; else dph0 ^= 1u;
            tc_after();
            uint32_t v[32];
            tc_ld_32x32(tmem + lane_tm + kColDv + 64u * (uint32_t)p + (uint32_t)(16 * cq), v);  // 16 of 32 used
            tc_wait_ld(v);
#pragma unroll
            for (int e = 0; e < 16; ++e) acc[e] += __uint_as_float(v[e]);
        }
        if (t_live) {
            float4 *out = reinterpret_cast<float4 *>(a.dv + ((int64_t)t * a.nkv + g) * kTcD + 16 * cq);
#pragma unroll
            for (int e = 0; e < 4; ++e) out[e] = make_float4(acc[4 * e], acc[4 * e + 1], acc[4 * e + 2], acc[4 * e + 3]);
        }
        tc_before();
        __syncwarp();
        if (lane == 0) bar_arrive(su32(&c.dv_empty));
    }
}

template <bool kF16>
__global__ void __launch_bounds__(kTcThreads, 1) mha_grad_v_tc_kernel(const __grid_constant__ TcArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t smem = (su32(smem_raw) + 1023u) & ~1023u;
    uint8_t *base = smem_raw + (smem - su32(smem_raw));
    TcCtl &c = *reinterpret_cast<TcCtl *>(base);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            bar_init(su32(&c.full_q[s]), 1);
            bar_init(su32(&c.full_o[s]), 1);
            bar_init(su32(&c.empty_q[s]), 1);
            bar_init(su32(&c.empty_o[s]), 1);
        }
        bar_init(su32(&c.k_full), 1);
        bar_init(su32(&c.k_empty), 2);  // both MMA warps
        for (int b = 0; b < 2; ++b) {
            bar_init(su32(&c.s_full[b]), 1);
            bar_init(su32(&c.s_empty[b]), kTcSoftWarps / 2);  // one group
        }
        for (int b = 0; b < 2; ++b) {
            bar_init(su32(&c.p_ready[b]), kTcSoftWarps / 2);
            bar_init(su32(&c.p_empty[b]), 1);
            bar_init(su32(&c.dv_full[b]), 1);
        }
        bar_init(su32(&c.dv_empty), kTcSoftWarps);
        bar_init(su32(&c.mma_done[0]), 1);
        bar_init(su32(&c.mma_done[1]), 1);
        c.abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kTcMmaWarp) tc_alloc(su32(&c.tmem_base), 512);
    tc_before();
    __syncthreads();
    tc_after();
    const uint32_t tmem = c.tmem_base;
    if (warp >= kTcLoadWarp && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.q_map)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.k_map)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.o_map)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&a.l_map)) : "memory");
    }
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (warp >= kTcLoadWarp) {
        if (lane == 0) tc_role_load(a, c, smem, warp - kTcLoadWarp);
        __syncwarp();
    } else if (warp == kTcMmaWarp || warp == kTcMma2Warp) {
        tc_role_mma(a, c, smem, tmem, warp - kTcMmaWarp, lane == 0 ? 1u : 0u);
        __syncwarp();
    } else {
        tc_role_soft<kF16>(a, c, smem, tmem, warp, lane);
    }
    tc_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_after();
        tc_dealloc(tmem, 512);
    }
}

// The statistics view needs rows of a multiple of 16 bytes: an even head count.
bool tc_applies(const void *q, const void *k, const void *go, const float *lse, const float *dv,
                const mha_grad_v_params *p, int dtype) {
    return dtype != DGRAD_F32 && p->head_dim == (uint32_t)kTcD && p->num_heads % 2 == 0 && aligned(q, 16) &&
           aligned(k, 16) && aligned(go, 16) && aligned(lse, 16) && aligned(dv, 16);
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

// LSE [q_seq][heads][2] float32 as [q_seq][2 heads], box [128][4], no swizzle.
bool encode_lse_map(CUtensorMap *m, const float *ptr, int len, int heads) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = tc_encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)heads * 2, (cuuint64_t)len};
    const cuuint64_t strides[1] = {(cuuint64_t)heads * 2 * sizeof(float)};
    const cuuint32_t box[2] = {4, 128};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
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
    const uint32_t fmt = dtype == DGRAD_BF16 ? 1u : 0u;
    // D float32, A and B of the input type; GEMM1: both K-major, N = 128;
    // GEMM2: B (dO) MN-major, N = 64; M = 128.
    a.idesc1 = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(kTcP >> 3) << 17) | ((uint32_t)(kTcT >> 4) << 24);
    a.idesc2 = (1u << 4) | (fmt << 7) | (fmt << 10) | (1u << 16) | ((uint32_t)(kTcD >> 3) << 17) |
               ((uint32_t)(kTcT >> 4) << 24);
    a.wait_limit_ns = 2000000000ull;
    if (!encode_heads_map(&a.q_map, q, a.q_seq, a.nh) || !encode_heads_map(&a.k_map, k, a.kv, a.nkv) ||
        !encode_heads_map(&a.o_map, go, a.q_seq, a.nh) || !encode_lse_map(&a.l_map, lse, a.q_seq, a.nh))
        return DGRAD_ERR_UNSUPPORTED;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DGRAD_ERR_CUDA;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return DGRAD_ERR_CUDA;
    static std::atomic<uint64_t> configured{0};
    const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
    if (!bit || !(configured.load() & bit)) {
        if (cudaFuncSetAttribute(mha_grad_v_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kTcSmem) != cudaSuccess ||
            cudaFuncSetAttribute(mha_grad_v_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kTcSmem) != cudaSuccess)
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
    const cudaError_t e = dtype == DGRAD_F16 ? cudaLaunchKernelEx(&cfg, mha_grad_v_tc_kernel<true>, a)
                                             : cudaLaunchKernelEx(&cfg, mha_grad_v_tc_kernel<false>, a);
    return e == cudaSuccess ? DGRAD_OK : DGRAD_ERR_CUDA;
}

}  // namespace
}  // namespace mhadv
