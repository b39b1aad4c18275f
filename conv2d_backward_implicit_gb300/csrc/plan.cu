// plan.cu -- host-side validation and planning (no device work).
//
// Validation follows the Params struct of conv2d_grad_input_gemm_coop.wgsl
// (twelve u32 fields, one stride, separate paddings); out_h and out_w are
// inputs there, so they are checked against floor((in + 2p - k)/s) + 1.
// Planning splits the problem into the stride's sub-pixel phases (see
// dgrad_internal.h) and sizes the tensor-core kernel's tiles, stages and
// shared memory, or selects the CUDA-core kernel.
#include <algorithm>
#include <cstring>

#include "conv2d_grad_input.h"
#include "dgrad_internal.h"

namespace dgrad {
namespace {

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// Try to build a tensor-core plan.  Returns false when the shape is outside
// what the tcgen05 kernel supports; the caller then uses the CUDA-core kernel.
bool plan_tc(const conv2d_grad_input_params &p, int esize, int dtype, Plan *plan) {
    TcParams &t = plan->tc;
    std::memset(&t, 0, sizeof(t));
    const int s = (int)p.stride;
    if (s > 4) return false;
    const int64_t H = p.in_h, W = p.in_w, kH = p.kernel_h, kW = p.kernel_w;
    const int64_t N = p.batch, Ci = p.in_channels, Co = p.out_channels;
    const int E = 16 / esize;

    t.N = (int)N; t.Ci = (int)Ci; t.H = (int)H; t.W = (int)W; t.Co = (int)Co;
    t.OH = (int)p.out_h; t.OW = (int)p.out_w; t.stride = s;

    t.n_ntiles = (int)cdiv(Ci, 256);
    t.n_tile = (int)round_up(cdiv(Ci, t.n_ntiles), 16);

    // Phases.
    int max_hb = 0, max_taps = 0, np = 0;
    for (int rh = 0; rh < s; ++rh) {
        for (int rw = 0; rw < s; ++rw) {
            PhaseDesc d;
            std::memset(&d, 0, sizeof(d));
            d.rh = rh; d.rw = rw;
            d.Hr = rh < H ? (int)cdiv(H - rh, s) : 0;
            d.Wr = rw < W ? (int)cdiv(W - rw, s) : 0;
            if (d.Hr == 0 || d.Wr == 0) continue;  // no grad_in pixel in this phase
            d.th = (int)((rh + p.padding_h) % s);
            d.qh = (int)((rh + p.padding_h) / s);
            d.tw = (int)((rw + p.padding_w) % s);
            d.qw = (int)((rw + p.padding_w) / s);
            d.Jh = d.th < kH ? (int)cdiv(kH - d.th, s) : 0;
            d.Jw = d.tw < kW ? (int)cdiv(kW - d.tw, s) : 0;
            if (d.Jh == 0 || d.Jw == 0) {
                d.Jh = d.Jw = 0;          // zero-filled phase
                d.X = d.Wr;
                d.R = d.Hr;
                d.hb = 0;
            } else {
                d.X = d.Wr + d.Jw - 1;
                d.R = d.Hr + d.Jh - 1;
                d.hb = kTileM + (d.Jh - 1) * d.X + (d.Jw - 1);
            }
            const int64_t positions = N * d.R * d.X;
            if (positions + 4096 > INT32_MAX) return false;  // 32-bit frame arithmetic
            d.m_tiles = (int)cdiv(positions, kTileM);
            max_hb = std::max(max_hb, d.hb);
            max_taps = std::max(max_taps, d.Jh * d.Jw);
            t.ph[np++] = d;
        }
    }
    t.n_phases = np;
    if (np == 0) return false;

    const int budget = kSmemLimit - kBarrierBytes;
    // Grad_out channels per stage: 2, 4 or 8 sixteen-byte chunks (K = 32, 64, 128 bytes).
    int chunks_pref = Co > 4 * E ? 8 : (Co > 2 * E ? 4 : 2);
    bool ok = false;
    for (int chunks = chunks_pref; chunks >= 2 && !ok; chunks /= 2) {
        t.kc = chunks * E;
        t.n_cchunks = (int)cdiv(Co, t.kc);
        t.hbp = (int)round_up(std::max(max_hb, 8), 8);
        const int64_t a_stage = (int64_t)chunks * t.hbp * 16;
        const int64_t b_unit = (int64_t)chunks * t.n_tile * 16;  // one tap, one channel chunk
        int64_t packed = 0;
        for (int i = 0; i < np; ++i) {
            PhaseDesc &d = t.ph[i];
            d.pack_off = packed;
            packed += (int64_t)t.n_ntiles * t.n_cchunks * d.Jh * d.Jw * b_unit;
        }
        if (a_stage > budget) continue;
        t.a_stage_bytes = (int)a_stage;
        t.b_unit_bytes = (int)b_unit;
        t.packed_bytes = packed;
        // Resident weights when they fit beside three A stages.
        if (packed + 3 * a_stage <= budget && packed <= (int64_t)160 * 1024) {
            t.nb = 0;
            t.b_stage_bytes = (int)(max_taps * b_unit);
            t.na = (int)std::min<int64_t>(4, (budget - packed) / a_stage);
            ok = t.na >= 2;
            if (ok) t.smem_bytes = kBarrierBytes + (int)(packed + t.na * a_stage);
            continue;
        }
        const int64_t b_stage = std::max<int64_t>(1, max_taps) * b_unit;
        if (2 * b_stage + 2 * a_stage > budget) continue;
        t.b_stage_bytes = (int)b_stage;
        t.nb = (int)std::min<int64_t>(4, (budget - 2 * a_stage) / b_stage);
        t.na = (int)std::min<int64_t>(4, (budget - t.nb * b_stage) / a_stage);
        ok = t.na >= 2 && t.nb >= 2;
        if (ok) t.smem_bytes = kBarrierBytes + (int)(t.nb * b_stage + t.na * a_stage);
    }
    if (!ok) return false;

    int64_t tiles = 0;
    for (int i = 0; i < np; ++i) {
        t.ph[i].tile_begin = tiles;
        tiles += (int64_t)t.ph[i].m_tiles * t.n_ntiles;
    }
    t.total_tiles = tiles;

    // tcgen05 instruction descriptor: D f32, A/B K-major, M = 128, N = n_tile.
    uint32_t fmt = dtype == DGRAD_F32 ? 2u : (dtype == DGRAD_BF16 ? 1u : 0u);
    t.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(t.n_tile >> 3) << 17) |
              ((uint32_t)(kTileM >> 4) << 24);
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * t.n_tile)) cols *= 2;
    t.tmem_cols = cols;

    // Pack parameters mirror the layout above.
    PackParams &k = plan->pack;
    std::memset(&k, 0, sizeof(k));
    k.Ci = (int)Ci; k.Co = (int)Co; k.kH = (int)kH; k.kW = (int)kW; k.stride = s;
    k.n_tile = t.n_tile; k.n_ntiles = t.n_ntiles; k.kc = t.kc; k.n_cchunks = t.n_cchunks;
    k.elems16 = E;
    k.n_phases = np;
    for (int i = 0; i < np; ++i) {
        k.elem_begin[i] = t.ph[i].pack_off / esize;
        k.th[i] = t.ph[i].th; k.tw[i] = t.ph[i].tw;
        k.Jh[i] = t.ph[i].Jh; k.Jw[i] = t.ph[i].Jw;
    }
    k.elem_begin[np] = t.packed_bytes / esize;
    k.total_elems = t.packed_bytes / esize;
    plan->workspace = (size_t)t.packed_bytes;
    return true;
}

}  // namespace

int make_plan(const void *params_v, int dtype, int forced_kernel, Plan *plan) {
    if (!params_v || !plan) return DGRAD_ERR_INVALID_ARG;
    if (dtype != DGRAD_F32 && dtype != DGRAD_BF16 && dtype != DGRAD_F16) return DGRAD_ERR_INVALID_ARG;
    const conv2d_grad_input_params &p = *static_cast<const conv2d_grad_input_params *>(params_v);
    const uint32_t f[12] = {p.batch, p.in_channels, p.in_h, p.in_w, p.out_channels, p.kernel_h,
                            p.kernel_w, p.stride, p.padding_h, p.out_h, p.out_w, p.padding_w};
    for (int i = 0; i < 12; ++i)
        if (f[i] > (uint32_t)INT32_MAX / 4) return DGRAD_ERR_UNSUPPORTED;
    if (!p.batch || !p.in_channels || !p.in_h || !p.in_w || !p.out_channels || !p.kernel_h ||
        !p.kernel_w || !p.stride || !p.out_h || !p.out_w)
        return DGRAD_ERR_SHAPE;
    const int64_t span_h = (int64_t)p.in_h + 2 * (int64_t)p.padding_h - p.kernel_h;
    const int64_t span_w = (int64_t)p.in_w + 2 * (int64_t)p.padding_w - p.kernel_w;
    if (span_h < 0 || span_w < 0) return DGRAD_ERR_SHAPE;
    if ((int64_t)p.out_h != span_h / p.stride + 1 || (int64_t)p.out_w != span_w / p.stride + 1)
        return DGRAD_ERR_SHAPE;
    // Element counts of the three tensors (guard int64 and per-plane int32 use).
    const int64_t go = (int64_t)p.batch * p.out_channels * p.out_h * p.out_w;
    const int64_t wt = (int64_t)p.out_channels * p.in_channels * p.kernel_h * p.kernel_w;
    const int64_t gi = (int64_t)p.batch * p.in_channels * p.in_h * p.in_w;
    const int64_t lim = (int64_t)1 << 40;
    if (go > lim || wt > lim || gi > lim) return DGRAD_ERR_UNSUPPORTED;
    if ((int64_t)p.out_h * p.out_w > INT32_MAX || (int64_t)p.in_h * p.in_w > INT32_MAX)
        return DGRAD_ERR_UNSUPPORTED;

    std::memset(plan, 0, sizeof(*plan));
    plan->dtype = dtype;
    plan->esize = dtype == DGRAD_F32 ? 4 : 2;
    SimtParams &sp = plan->simt;
    sp.N = (int)p.batch; sp.Ci = (int)p.in_channels; sp.H = (int)p.in_h; sp.W = (int)p.in_w;
    sp.Co = (int)p.out_channels; sp.kH = (int)p.kernel_h; sp.kW = (int)p.kernel_w;
    sp.stride = (int)p.stride; sp.ph = (int)p.padding_h; sp.pw = (int)p.padding_w;
    sp.OH = (int)p.out_h; sp.OW = (int)p.out_w;

    if (forced_kernel == DGRAD_KERNEL_SIMT) {
        plan->kernel = DGRAD_KERNEL_SIMT;
        return DGRAD_OK;
    }
    if (plan_tc(p, plan->esize, dtype, plan)) {
        plan->kernel = DGRAD_KERNEL_TC;
        return DGRAD_OK;
    }
    if (forced_kernel == DGRAD_KERNEL_TC) return DGRAD_ERR_UNSUPPORTED;
    plan->kernel = DGRAD_KERNEL_SIMT;
    plan->workspace = 0;
    return DGRAD_OK;
}

}  // namespace dgrad
