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
#include <numeric>

#include "conv2d_grad_input.h"
#include "dgrad_internal.h"

namespace dgrad {
namespace {

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t Co_of(const conv2d_grad_input_params &p) { return p.out_channels; }
int64_t round_up(int64_t a, int64_t b) { return cdiv(a, b) * b; }

// Raw-slice geometry of the gather (tiles of whole frame rows only): each
// slice holds raw_cs grad_out channels x raw_br rows x raw_bw columns, and the
// gather warps turn it into the frame window.  Returns 1 and fills the raw_*
// fields when one of the load modes applies to the shape (none: clear them).
//  * tiled: grad_out rows a multiple of 16 bytes -- a 4-D TMA box over the
//    columns that hold data, rows outside the grid zero-filled by the TMA unit;
//  * planes: every tile covers whole images and raw_cs channel planes are a
//    multiple of 16 bytes -- one 1-D bulk copy of raw_cs whole planes;
//  * rows: channel planes a multiple of 16 bytes -- the window's rows from
//    a row whose byte offset is a multiple of 16 (a multiple of raw_rowg
//    rows, so a slice holds up to raw_rowg - 1 extra rows above the window):
//    one TMA box of a map whose rows are raw_rowg grad_out rows when the
//    planes split into whole such groups (tiled mode with raw_rowg > 1),
//    else one 1-D bulk copy per channel of the rows inside the grid.
int plan_raw_slices(const conv2d_grad_input_params &p, int esize, TcParams &t, bool none = false,
                    int cs = 0) {
    t.raw_nr = 0;
    t.raw_mode = kRawNone;
    t.raw_rowg = 1;
    t.raw_x0 = t.raw_bw = t.raw_br = t.raw_cs = t.raw_slice_bytes = 0;
    if (none || t.rows_per_tile <= 0) return 0;
    // Every window row a gather thread owns keeps its slice offset in a register.
    if (t.hbp > kGWarps * 32 * kMaxGatherRows) return 0;
    const int64_t OH = p.out_h, OW = p.out_w, Co = p.out_channels;
    const int64_t row_bytes = OW * esize, plane_bytes = OH * OW * esize;
    const int A = 16 / esize;  // elements per 16 bytes
    if (cs <= 0) cs = 32 / esize;  // default: two 16-byte channel chunks per slice
    // Frame columns that carry grad_out data, over all phases, and the rows
    // one window spans.
    int64_t vmin = INT32_MAX, vmax = INT32_MIN, rows = 1;
    bool whole = true;
    for (int i = 0; i < t.n_phases; ++i) {
        const PhaseDesc &d = t.ph[i];
        if (d.Jh == 0) continue;
        vmin = std::min<int64_t>(vmin, d.qw - (d.Jw - 1));
        vmax = std::max<int64_t>(vmax, d.Wr - 1 + d.qw);
        rows = std::max<int64_t>(rows, (t.hbp - 1) / d.X + 1);
        if (t.rows_per_tile < d.Hr) whole = false;
    }
    if (vmin > vmax) return 0;  // no phase reads grad_out
    int mode = kRawNone;
    if (row_bytes % 16 == 0) {
        const int64_t lo = std::max<int64_t>(vmin, 0), hi = std::min<int64_t>(vmax, OW - 1);
        const int64_t x0 = lo / A * A;
        const int64_t bw = round_up(std::max<int64_t>(hi - x0 + 1, 1), A);
        if (bw <= 256 && rows <= 256) {
            mode = kRawTiled;
            t.raw_x0 = (int)x0;
            t.raw_bw = (int)bw;
            t.raw_br = (int)rows;
        }
    }
    if (mode == kRawNone && whole && (Co * plane_bytes) % 16 == 0 && (cs * plane_bytes) % 16 == 0 &&
        cs * plane_bytes <= kRawPlaneMaxBytes) {
        mode = kRawPlanes;
        t.raw_bw = (int)OW;
        t.raw_br = (int)OH;
    }
    if (mode == kRawNone && plane_bytes % 16 == 0) {
        // Windows start on a multiple of g rows (g rows = a multiple of 16
        // bytes).  When the planes split into whole g-row groups, a TMA map
        // over [N][Co][OH/g][g*OW] loads each slice as one box; otherwise one
        // 1-D copy per channel.
        const int64_t g = 16 / std::gcd<int64_t>(16, row_bytes);
        const int64_t br = round_up(rows + g - 1, g);
        mode = (OH % g == 0 && OW * g <= 256 && br / g <= 256) ? kRawTiled : kRawRows;
        t.raw_rowg = (int)g;
        t.raw_x0 = 0;
        t.raw_bw = (int)OW;
        t.raw_br = (int)br;
    }
    if (mode == kRawNone) return 0;
    t.raw_mode = mode;
    t.raw_cs = cs;
    t.raw_slice_bytes = (int)round_up((int64_t)cs * t.raw_br * t.raw_bw * esize, 128);
    t.raw_nr = 3;
    return 1;
}

// Try to build a tensor-core plan.  Returns false when the shape is outside
// what the tcgen05 kernel supports; the caller then uses the CUDA-core kernel.
// pair: plan paired column phases (TcParams::pair_rw) or fail: stride 2,
// four phases with taps, one 128-row channel tile, W a multiple of 8 up to 64,
// the two column phases of each row phase reading the same frame (equal
// Jw - qw), tiles of at most 128 positions.  The four phases then share one
// frame pitch X (the larger one), so a pair's window is gathered once.
bool plan_tc(const conv2d_grad_input_params &p, int esize, int dtype, Plan *plan, bool pair = false) {
    TcParams &t = plan->tc;
    std::memset(&t, 0, sizeof(t));
    const int s = (int)p.stride;
    if (s > 4) return false;
    const int64_t H = p.in_h, W = p.in_w, kH = p.kernel_h, kW = p.kernel_w;
    const int64_t N = p.batch, Ci = p.in_channels, Co = p.out_channels;
    const int E = 16 / esize;

    t.N = (int)N; t.Ci = (int)Ci; t.H = (int)H; t.W = (int)W; t.Co = (int)Co;
    t.OH = (int)p.out_h; t.OW = (int)p.out_w; t.stride = s;
    t.esize = esize;

    // Input channels on the MMA M side: one 64-row tile, or 128-row tiles.
    t.m_tile = Ci <= 64 ? 64 : 128;
    t.n_mtiles = (int)cdiv(Ci, t.m_tile);

    // Widest frame row and tallest phase over the stride's phases.
    int64_t X1 = 1, Hr1 = 1;
    for (int r = 0; r < s; ++r) {
        const int64_t Wr = r < W ? cdiv(W - r, s) : 0, Hr = r < H ? cdiv(H - r, s) : 0;
        const int64_t tw = (r + p.padding_w) % s;
        const int64_t Jw = tw < kW ? cdiv(kW - tw, s) : 0;
        X1 = std::max(X1, Jw > 0 ? Wr + Jw - 1 : Wr);
        Hr1 = std::max(Hr1, Hr);
    }

    // Output positions per tile: 256 (full-rate N); 128 when a 256-wide
    // tile's frame window would not leave room for two stages.
    bool ok = false;
    int np = 0;
    for (int cap = kTileP; cap >= 128 && !ok; cap /= 2) {
        // Tiles of whole frame rows (k rows of the widest phase's X positions,
        // the accumulator rounded up to 16 columns), so each tile owns
        // complete output rows of its phase; when one row is wider than the
        // tile, tiles are `cap` consecutive frame positions.
        int tile_p = cap, rows_per_tile = 0;
        {
            int64_t k = cap / X1;
            while (k > 0 && round_up(k * X1, 16) > cap) --k;
            if (k > 0) {
                rows_per_tile = (int)std::min<int64_t>(k, Hr1);
                tile_p = (int)round_up(rows_per_tile * X1, 16);
            }
        }
        t.rows_per_tile = rows_per_tile;
        // Phases.
        int max_hb = 0, max_taps = 0;
        np = 0;
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
                    d.hb = tile_p + (d.Jh - 1) * d.X + (d.Jw - 1);
                }
                const int64_t positions = N * d.R * d.X;
                if (positions + 8192 > INT32_MAX) return false;  // 32-bit frame arithmetic
                d.p_tiles = rows_per_tile > 0 ? (int)(N * cdiv(d.Hr, rows_per_tile))
                                              : (int)cdiv(positions, tile_p);
                max_hb = std::max(max_hb, d.hb);
                max_taps = std::max(max_taps, d.Jh * d.Jw);
                t.ph[np++] = d;
            }
        }
        t.n_phases = np;
        if (np == 0) return false;
        if (pair) {
            if (s != 2 || np != 4 || rows_per_tile <= 0 || Ci > 128 || W % 8 != 0 || W > 64) return false;
            // (the pair variant runs kGWarps - 1 gather warps beside two producers)
            if (round_up(tile_p + 2 * X1 + 8, 8) > (int64_t)(kGWarps - 1) * 32 * kMaxGatherRows) return false;
            for (int i = 0; i < 4; ++i) {
                const PhaseDesc &d = t.ph[i];
                const PhaseDesc &o = t.ph[i ^ 1];  // the other column phase of the row phase
                if (d.Jh == 0 || d.Jw == 0 || d.rh != i / 2 || d.rw != i % 2 || 2 * d.Wr != W ||
                    d.Jw - d.qw != o.Jw - o.qw)
                    return false;
            }
            max_hb = 0;
            for (int i = 0; i < 4; ++i) {
                PhaseDesc &d = t.ph[i];
                d.X = (int)X1;
                d.hb = tile_p + (d.Jh - 1) * d.X + (d.Jw - 1);
                if ((int64_t)N * d.R * d.X + 8192 > INT32_MAX) return false;
                max_hb = std::max(max_hb, d.hb);
            }
        }
        t.tile_p = tile_p;

        // Shared memory: barriers, 1 KB to align the rings to 1024 B, then the
        // grad_out (G) ring and the weight (W) ring.
        // Epilogue staging: padded 33-float rows per channel of a warp, or (TMA
        // store epilogue, stride 1 with W a multiple of 4 up to 64) one box of
        // 8 channels x W floats per warp.
        int epi = kEpiWarps * (t.m_tile / 4) * kEpiRowFloats * 4;
        if (rows_per_tile > 0 && W % 4 == 0 && W <= 64)
            epi = std::max(epi, (int)(kEpiWarps * kTmaBoxCi * W * 4));
        epi = (int)round_up(epi, kEpiWarps * 128);  // each warp's area 128-byte aligned
        t.epi_stage_bytes = epi;
        t.epi_boxes = 1;
        t.epi_box_ci = kTmaBoxCi;
        // Each stage carries 128 bytes of grad_out channels per frame element or
        // weight row (64 bf16/fp16 or 32 fp32 channels): one 128-byte swizzle row.
        t.kc = 128 / esize;
        t.n_cchunks = (int)cdiv(Co, t.kc);
        t.hbp = (int)round_up(std::max(max_hb, 8), 8);
        const int64_t g_stage = (int64_t)t.hbp * 128;
        const int64_t w_unit = (int64_t)t.m_tile * 128;  // one tap, one channel chunk
        int64_t packed = 0;
        for (int i = 0; i < np; ++i) {
            PhaseDesc &d = t.ph[i];
            d.pack_off = packed;
            packed += (int64_t)t.n_mtiles * t.n_cchunks * d.Jh * d.Jw * w_unit;
        }
        t.g_stage_bytes = (int)g_stage;
        t.w_unit_bytes = (int)w_unit;
        t.packed_bytes = packed;
        // When the weights cannot stay resident beside the raw ring, they are
        // streamed, preferably with raw slices of a whole channel chunk (one
        // copy and one hand-over per stage instead of several), when at least
        // two such slices fit beside two G stages and two weight stages.
        const bool narrow_raw = rows_per_tile > 0 && plan_raw_slices(p, esize, t);
        if (narrow_raw && t.kc > 32 / esize &&
            packed + 2 * g_stage + 2 * (int64_t)t.raw_slice_bytes > kSmemLimit - smem_layout_bytes(epi, 0, 0) &&
            plan_raw_slices(p, esize, t, false, t.kc)) {
            const int64_t room = kSmemLimit - smem_layout_bytes(epi, 0, 0) - 2 * g_stage - 1024;
            const int64_t slice = t.raw_slice_bytes, w_stage = w_unit;
            for (int64_t nw = std::min<int64_t>(kMaxW, std::max<int64_t>(2, room / 2 / w_stage)); nw >= 2 && !ok; --nw) {
                const int64_t nr = std::min<int64_t>(kMaxRaw, (room - nw * w_stage) / slice);
                if (nr < 2) continue;
                t.raw_nr = (int)nr;
                t.nw = (int)nw;
                t.ng = 2;
                t.taps_per_w = 1;
                t.w_stage_bytes = (int)w_stage;
                t.smem_bytes = (int)(smem_layout_bytes(epi, nr * slice, 0) + nw * w_stage + 2 * g_stage);
                ok = t.smem_bytes <= kSmemLimit;
            }
        }
        // Raw grad_out slices for the TMA / bulk-copy gather, reserved when a
        // load mode applies (tried first; without them if G and W do not fit).
        const int plan_raw = ok ? 1 : (rows_per_tile > 0 ? plan_raw_slices(p, esize, t) : 0);
        // Raw slices with streamed weights: two G stages (the gather turns a
        // slice around in far less time than the MMAs of a stage take), and
        // the rest of shared memory split between the weight ring and the raw
        // ring -- the data in flight that covers L2 latency.
        if (!ok && plan_raw && packed + 2 * g_stage + 2 * (int64_t)t.raw_slice_bytes >
                            kSmemLimit - smem_layout_bytes(epi, 0, 0)) {
            const int64_t room = kSmemLimit - smem_layout_bytes(epi, 0, 0) - 2 * g_stage - 1024;
            const int64_t slice = t.raw_slice_bytes;
            const int64_t tpw = 1;
            const int64_t w_stage = tpw * w_unit;
            const int64_t nw = std::min<int64_t>(kMaxW, std::max<int64_t>(2, room / 2 / w_stage));
            const int64_t nr = std::min<int64_t>(kMaxRaw, (room - nw * w_stage) / slice);
            if (nr >= 2 && room >= nw * w_stage + nr * slice) {
                t.raw_nr = (int)nr;
                t.nw = (int)nw;
                t.ng = 2;
                t.taps_per_w = (int)tpw;
                t.w_stage_bytes = (int)w_stage;
                t.smem_bytes = (int)(smem_layout_bytes(epi, nr * slice, 0) + nw * w_stage + 2 * g_stage);
                ok = t.smem_bytes <= kSmemLimit;
            }
        }
        // Otherwise ring depths tried: 3 raw slots, 2, then none.
        for (int nr = plan_raw ? 3 : 0; nr >= 0 && !ok; nr = nr == 2 ? 0 : nr - 1) {
            if (nr == 0) plan_raw_slices(p, esize, t, /*none=*/true);
            t.raw_nr = nr;
            const int raw = t.raw_nr * t.raw_slice_bytes;
            const int budget = (int)(kSmemLimit - smem_layout_bytes(epi, raw, 0));
            if (2 * g_stage > budget) continue;
            const int fixed = (int)smem_layout_bytes(epi, raw, 0);
            if (packed + (raw ? 2 : 3) * g_stage <= budget) {
                // Resident weights: loaded once per CTA, beside at least three G
                // stages (two when the raw ring also needs room).
                t.nw = 0;
                t.taps_per_w = std::max(max_taps, 1);
                t.w_stage_bytes = (int)(t.taps_per_w * w_unit);
                t.ng = (int)std::min<int64_t>(4, (budget - packed) / g_stage);
                ok = true;
                t.smem_bytes = fixed + (int)(packed + t.ng * g_stage);
            } else {
                // Streamed weights: each W stage holds a group of up to taps_per_w
                // consecutive taps of one channel chunk; four stages when they fit.
                const int64_t room = budget - 2 * g_stage;
                int64_t tpw = std::min<int64_t>(std::max(max_taps, 1), room / (4 * w_unit));
                if (tpw < 1) tpw = std::min<int64_t>(std::max(max_taps, 1), room / (2 * w_unit));
                if (tpw >= 1) {
                    t.taps_per_w = (int)tpw;
                    const int64_t w_stage = tpw * w_unit;
                    t.w_stage_bytes = (int)w_stage;
                    t.nw = (int)std::min<int64_t>(4, room / w_stage);
                    t.ng = (int)std::min<int64_t>(4, (budget - t.nw * w_stage) / g_stage);
                    ok = t.ng >= 2 && t.nw >= 2;
                    t.smem_bytes = fixed + (int)(t.nw * w_stage + t.ng * g_stage);
                }
            }
        }
    }
    if (!ok) return false;
    t.raw_early = (t.raw_nr > 0 && t.ng >= 2 && t.nw == 0)
                      ? (int)std::min<int64_t>(kMaxEarly, t.g_stage_bytes / t.raw_slice_bytes)
                      : 0;

    t.tile_group = 1;
    int64_t tiles = 0;
    t.interleave = np > 1 ? 1 : 0;
    for (int i = 0; i < np; ++i) {
        t.ph[i].tile_begin = tiles;
        tiles += (int64_t)t.ph[i].p_tiles * t.n_mtiles;
        if (t.ph[i].p_tiles != t.ph[0].p_tiles) t.interleave = 0;
    }
    t.total_tiles = tiles;

    // tcgen05 instruction descriptor: D f32, A (weights) and B (grad_out
    // window) K-major, M = m_tile, N = tile_p.
    const uint32_t fmt = dtype == DGRAD_F32 ? 2u : (dtype == DGRAD_BF16 ? 1u : 0u);
    t.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(t.tile_p >> 3) << 17) |
              ((uint32_t)(t.m_tile >> 4) << 24);
    uint32_t cols = 32;  // double-buffered accumulator, allocated in a power of two
    while (cols < (uint32_t)((pair ? 4 : 2) * t.tile_p)) cols *= 2;
    if (pair && cols > 512) {
        // A pair of accumulators of the tile's columns: double-buffered when
        // two pairs fit in TMEM's 512 columns, else one buffer.
        t.acc_single = 1;
        for (cols = 32; cols < (uint32_t)(2 * t.tile_p);) cols *= 2;
    }
    t.tmem_cols = cols;
    if (pair) {
        if (cols > 512 || !t.interleave || t.n_mtiles != 1 || t.m_tile != 128 ||
            t.epi_stage_bytes < kEpiWarps * 2 * kTmaBoxCi * (int)W * 4)
            return false;
        t.pair_rw = 1;
        t.tile_group = 2;
        t.epi_box_ci = 2 * kTmaBoxCi;  // the paired epilogue stores 16-channel boxes
    }

    // Pack parameters mirror the layout above.
    PackParams &k = plan->pack;
    std::memset(&k, 0, sizeof(k));
    k.Ci = (int)Ci; k.Co = (int)Co; k.kH = (int)kH; k.kW = (int)kW; k.stride = s;
    k.m_tile = t.m_tile; k.n_mtiles = t.n_mtiles; k.kc = t.kc; k.n_cchunks = t.n_cchunks;
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

// Positions-on-M plan (stride 1, 16-bit, Ci <= 64, Co <= 64, kW <= 3,
// W <= 56, OW <= 56 with 16-byte grad_out rows), derived from the general
// plan `g` whose packed weights it shares: [kh][kw][ci 0..63][co 0..63],
// 128-byte swizzled rows.
//
// Frame: kPmPitch = 64 positions per grad_out row, kPmLeft = 8 zero columns
// first, so window row h = 64u + b of a tile whose first output row is ih0
// holds grad_out[oh = ih0 + ph - (kH-1) + u, ow = b - 8] (zero outside the
// grid).  A tile is 4 output rows = 256 positions, processed as two halves of
// 128 on the MMA M side.  For kernel row kh the MMA reads the window from row
// 64 (kH-1-kh) + pw + 128 half, with the kW taps' weights stacked on N, so
// column block kw of lane l holds the tap (kh, kw) sum for output column
// c = (l mod 64) + kw; the epilogue adds block kw of lane l - kw.  Output
// (ih0 + r, iw) is lane 64 r + iw + 8.
bool plan_pm(const conv2d_grad_input_params &p, int esize, const TcParams &g, TcParams *out) {
    if (p.stride != 1 || esize != 2) return false;
    const int64_t H = p.in_h, W = p.in_w, kH = p.kernel_h, kW = p.kernel_w;
    const int64_t Ci = p.in_channels, Co = p.out_channels;
    if (Ci > 64 || Co > 64 || kW > kPmMaxKw || W > kPmPitch - kPmLeft) return false;
    if (p.out_w > (uint32_t)(kPmPitch - kPmLeft) || (p.out_w * (int64_t)esize) % 16 != 0) return false;
    if (p.padding_w > (uint32_t)kPmLeft) return false;
    if (g.m_tile != 64 || g.n_mtiles != 1 || g.n_cchunks != 1 || g.n_phases != 1) return false;
    TcParams t = g;
    t.pos_m = 1;
    t.pad_w = (int)p.padding_w;
    t.rows_per_tile = 4;
    t.tile_p = 4 * kPmPitch;
    const int64_t view_end = kPmPitch * (kH - 1) + p.padding_w + t.tile_p;  // rows the MMA reads
    t.pm_rows = (int)cdiv(view_end - kPmLeft, kPmPitch);
    t.hbp = (int)round_up(std::max<int64_t>(view_end, (int64_t)kPmPitch * t.pm_rows), 8);
    // 8x8 transpose blocks of one 16-channel slice, four per gather ldmatrix.x4.
    if (2 * t.pm_rows * ((kPmPitch - kPmLeft) / 8) > 4 * kPmGWarps * kPmGroups) return false;
    t.g_stage_bytes = t.hbp * 128;
    PhaseDesc &d = t.ph[0];
    std::memset(&d, 0, sizeof(d));
    d.Hr = (int)H; d.Wr = (int)W;
    d.Jh = (int)kH; d.Jw = (int)kW;
    d.qh = (int)p.padding_h; d.qw = (int)p.padding_w;
    d.X = kPmPitch; d.R = (int)(H + kH - 1);
    d.p_tiles = (int)((int64_t)p.batch * cdiv(H, t.rows_per_tile));
    d.hb = t.hbp;
    t.n_phases = 1;
    t.total_tiles = d.p_tiles;
    // Raw slices: 16 channels x raw_br rows x 56 columns from column 0; an
    // odd row count keeps the transposing ldmatrix reads free of bank
    // conflicts (channel pitch an odd number of 16-byte units).
    t.raw_mode = kRawTiled;
    t.raw_rowg = 1;
    t.raw_cs = 16;
    t.raw_bw = kPmPitch - kPmLeft;
    t.raw_x0 = 0;
    t.raw_br = t.pm_rows | 1;
    t.raw_slice_bytes = (int)round_up((int64_t)t.raw_cs * t.raw_br * t.raw_bw * esize, 128);
    t.epi_stage_bytes = kPmXBytes;
    t.epi_boxes = 0;
    t.ng = 2;
    t.nw = 0;
    const int64_t gw = t.packed_bytes + 2 * (int64_t)t.g_stage_bytes;
    t.raw_nr = 0;
    for (int r = 4; r >= 2 && !t.raw_nr; --r)
        if (smem_layout_bytes(t.epi_stage_bytes, (int64_t)r * t.raw_slice_bytes, gw) <= kSmemLimit) t.raw_nr = r;
    if (!t.raw_nr) return false;
    t.raw_early = (int)std::min<int64_t>(kMaxEarly, t.g_stage_bytes / t.raw_slice_bytes);
    t.smem_bytes = (int)smem_layout_bytes(t.epi_stage_bytes, (int64_t)t.raw_nr * t.raw_slice_bytes, gw);
    // M = 128 positions, N = kW x 64 (taps of one kernel row), A and B K-major.
    const uint32_t fmt = (g.idesc >> 7) & 7u;  // operand format of the general plan
    const int n = (int)kW * 64;
    t.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * n)) cols *= 2;  // two accumulator buffers
    t.tmem_cols = cols;
    *out = t;
    return true;
}

// General mode on the 64-wide frame (stride 1, 16-bit, W <= 56, OW <= 56
// with 16-byte grad_out rows), derived from the general plan `g` (same packed
// weights, same tiles of output rows).  Window row h = 64u + b holds
// grad_out[oh = ih0 + ph - (kH-1) + u, ow = b - kPmLeft]; output position
// 64 r + iw reads tap (kh, kw) at row 64 (r + kH-1-kh) + iw + pw - kw + 8,
// i.e. the tap's view starts at (kH-1-kh) * 64 + (kW-1-kw) + view0 with
// view0 = pw + 8 - (kW-1).  Needs the TMA gather and the TMA store epilogue.
bool plan_frame64(const conv2d_grad_input_params &p, int esize, const TcParams &g, TcParams *out) {
    if (p.stride != 1 || esize != 2 || g.n_phases != 1 || g.rows_per_tile <= 0 || g.nw != 0)
        return false;
    const int64_t H = p.in_h, W = p.in_w, kH = p.kernel_h, kW = p.kernel_w;
    if (W > kPmPitch - kPmLeft || p.out_w > (uint32_t)(kPmPitch - kPmLeft)) return false;
    if ((p.out_w * (int64_t)esize) % 16 != 0 || W % 4 != 0) return false;
    if (kW - 1 > (int64_t)p.padding_w + kPmLeft || p.padding_w > (uint32_t)kPmLeft) return false;
    TcParams t = g;
    t.frame64 = 1;
    t.view0 = (int)(p.padding_w + kPmLeft - (kW - 1));
    t.rows_per_tile = 4;
    t.tile_p = 4 * kPmPitch;
    const int64_t view_end = kPmPitch * (kH - 1) + p.padding_w + kPmLeft + t.tile_p;
    t.pm_rows = (int)(t.rows_per_tile + kH - 1);
    t.hbp = (int)round_up(std::max<int64_t>(view_end, (int64_t)kPmPitch * t.pm_rows), 8);

    t.g_stage_bytes = t.hbp * 128;
    PhaseDesc &d = t.ph[0];
    d.X = kPmPitch;
    d.R = (int)(H + kH - 1);
    d.p_tiles = (int)((int64_t)p.batch * cdiv(H, t.rows_per_tile));
    d.hb = t.hbp;
    d.tile_begin = 0;
    t.total_tiles = (int64_t)d.p_tiles * t.n_mtiles;
    t.raw_mode = kRawTiled;
    t.raw_rowg = 1;
    t.raw_bw = kPmPitch - kPmLeft;
    t.raw_x0 = 0;
    t.raw_br = t.pm_rows | 1;
    // TMA store boxes only: 64-row tiles read a quadrant's 16 channels with
    // the 16x256b TMEM shape (all 32 threads busy) into one 16-channel box
    // per warp; 128-row tiles use 8-channel boxes, two per warp when that
    // still leaves two raw slots, else one.
    t.epi_box_ci = t.m_tile == 64 ? 16 : kTmaBoxCi;
    const int64_t box = (int64_t)t.epi_box_ci * W * 4;
    t.ng = 2;
    const int64_t gw = t.packed_bytes + 2 * (int64_t)t.g_stage_bytes;
    t.raw_nr = 0;
    // Raw slices of 32 channels (one TMA load per half chunk) when a ring of
    // at least one such slice fits, else 16: a TMA load costs about the same
    // time whatever its size up to tens of KB, so fewer, larger loads move
    // the window in far less time.  The ldmatrix groups per gather warp
    // (kF64Groups) bound the slice's 8x8 blocks.
    for (int cs = 16; cs >= 16 && !t.raw_nr; cs /= 2) {
        if ((cs / 8) * t.pm_rows * ((kPmPitch - kPmLeft) / 8) > 4 * kGWarps * kF64Groups) continue;
        if (Co_of(p) % cs != 0 && cs == 32) continue;  // whole slices of the chunk's channels
        t.raw_cs = cs;
        t.raw_slice_bytes = (int)round_up((int64_t)t.raw_cs * t.raw_br * t.raw_bw * esize, 128);
        for (int boxes = t.epi_box_ci == 16 ? 1 : 2; boxes >= 1 && !t.raw_nr; --boxes) {
            const int64_t epi = round_up(kEpiWarps * boxes * box, kEpiWarps * 128);
            for (int r = cs == 32 ? 2 : 3; r >= (cs == 32 ? 1 : 2) && !t.raw_nr; --r) {
                if (smem_layout_bytes(epi, (int64_t)r * t.raw_slice_bytes, gw) <= kSmemLimit) {
                    t.raw_nr = r;
                    t.epi_boxes = boxes;
                    t.epi_stage_bytes = (int)epi;
                }
            }
        }
    }
    if (!t.raw_nr) return false;
    t.raw_early = (int)std::min<int64_t>(kMaxEarly, t.g_stage_bytes / t.raw_slice_bytes);
    t.smem_bytes = (int)smem_layout_bytes(t.epi_stage_bytes, (int64_t)t.raw_nr * t.raw_slice_bytes, gw);
    t.idesc = (g.idesc & ~(0x3Fu << 17)) | ((uint32_t)(t.tile_p >> 3) << 17);  // N = 256

    t.tmem_cols = 2 * t.tile_p;
    *out = t;
    return true;
}

// MN-major plan for 1x1, stride-1, unpadded 16-bit problems whose tiles are
// whole images loaded as raw planes of a whole channel chunk (weights
// streamed): derived from the
// general plan `g` (same tiles, same packed weights).  A G stage holds kc / 8
// channel groups x mn_atoms atoms of 1 KB; the rings are re-fitted around it.
bool plan_mn(const conv2d_grad_input_params &p, int esize, const TcParams &g, TcParams *out) {
    if (p.stride != 1 || p.kernel_h != 1 || p.kernel_w != 1 || p.padding_h || p.padding_w || esize != 2)
        return false;
    // Channel planes start 8-byte aligned in the raw slice (the gather's 8-byte loads).
    if (((int64_t)p.out_h * p.out_w) % 4 != 0) return false;
    // Raw slices must be whole channel planes, [c][OH][OW] with no padding:
    // plane copies, or tensor-map boxes that span whole rows and planes.
    const bool planes = g.raw_mode == kRawPlanes ||
                        (g.raw_mode == kRawTiled && g.raw_rowg == 1 && g.raw_x0 == 0 &&
                         g.raw_bw == (int)p.out_w && g.raw_br == (int)p.out_h);
    if (g.n_phases != 1 || g.rows_per_tile < (int)p.in_h || !planes || g.raw_cs != g.kc || g.nw < 2 ||
        g.raw_nr < 2 || g.tile_p > 256)
        return false;
    TcParams t = g;
    t.mn_b = 1;
    t.mn_atoms = (int)cdiv(t.tile_p, 64);
    t.g_stage_bytes = (t.kc / 8) * t.mn_atoms * 1024;
    t.hbp = t.mn_atoms * 64;
    // (the MN-major variant runs kGWarps - 1 gather warps beside two producers)
    if ((int64_t)t.kc * t.mn_atoms * 8 > (int64_t)kMaxMnPieces * (kGWarps - 1) * 32) return false;
    t.ph[0].hb = t.hbp;
    // Epilogue staging per warp: a 1 KB-aligned swizzled [channels][32]
    // float box for the plane TMA store, with room for the staged epilogue's
    // padded block when that store cannot be used.
    t.epi_stage_bytes = kEpiWarps * (int)round_up((int64_t)32 * kEpiRowFloats * 4, 1024);
    const int64_t slice = t.raw_slice_bytes, w_stage = t.w_stage_bytes;
    auto bytes = [&](int64_t nr, int64_t nw) {
        return smem_layout_bytes(t.epi_stage_bytes, nr * slice, 0) + nw * w_stage + 2 * (int64_t)t.g_stage_bytes;
    };
    int64_t nr = t.raw_nr, nw = t.nw;
    while (bytes(nr, nw) > kSmemLimit && (nw > 2 || nr > 2)) {
        if (nw > 2 && (nw >= nr || nr <= 2)) --nw; else --nr;
    }
    if (bytes(nr, nw) > kSmemLimit) return false;
    t.raw_nr = (int)nr;
    t.nw = (int)nw;
    t.smem_bytes = (int)bytes(nr, nw);
    t.idesc |= 1u << 16;  // B (grad_out) MN-major
    *out = t;
    return true;
}

// Stacked-phase plan (stride 2..4, stride^2 x Ci <= 32; see
// TcParams::stacked).  Tap (j, i) of phase (rh, rw) reads grad_out
// (a + qh - j, b + qw - i) for output (a, b) of the phase grid; the window
// taps (dy, dx) are the union of those offsets over the phases, dy in
// [st_dy0, st_dy0 + st_th) and dx likewise.  The frame of ph[0] (pitch
// X = Wr + st_tw - 1) holds grad_out[a + dy][b + dx] at frame row
// a + dy - st_dy0, column b + dx - st_dx0: the frame convention of
// dgrad_internal.h with Jh = st_th and qh = st_th - 1 + st_dy0, so the
// general mode's raw-slice loads and gather serve it unchanged.  Tiles are
// whole frame rows, 128 positions at most (MMA M = 128); the weights stay
// resident.
bool plan_stacked(const conv2d_grad_input_params &p, int esize, int dtype, Plan *plan) {
    const int s = (int)p.stride;
    const int64_t H = p.in_h, W = p.in_w, kH = p.kernel_h, kW = p.kernel_w;
    const int64_t N = p.batch, Ci = p.in_channels, Co = p.out_channels;
    if (s < 2 || s > 4 || (int64_t)s * s * Ci > 32) return false;
    TcParams &t = plan->tc;
    std::memset(&t, 0, sizeof(t));
    PackParams &k = plan->pack;
    std::memset(&k, 0, sizeof(k));
    t.N = (int)N; t.Ci = (int)Ci; t.H = (int)H; t.W = (int)W; t.Co = (int)Co;
    t.OH = (int)p.out_h; t.OW = (int)p.out_w; t.stride = s;
    t.esize = esize;
    int64_t dy0 = INT32_MAX, dy1 = INT32_MIN, dx0 = INT32_MAX, dx1 = INT32_MIN;
    for (int rh = 0; rh < s; ++rh) {
        for (int rw = 0; rw < s; ++rw) {
            const int ph = rh * s + rw;
            k.th[ph] = (int)((rh + p.padding_h) % s);
            k.qh[ph] = (int)((rh + p.padding_h) / s);
            k.tw[ph] = (int)((rw + p.padding_w) % s);
            k.qw[ph] = (int)((rw + p.padding_w) / s);
            k.Jh[ph] = k.th[ph] < kH ? (int)cdiv(kH - k.th[ph], s) : 0;
            k.Jw[ph] = k.tw[ph] < kW ? (int)cdiv(kW - k.tw[ph], s) : 0;
            if (k.Jh[ph] == 0 || k.Jw[ph] == 0 || rh >= H || rw >= W) continue;
            dy0 = std::min<int64_t>(dy0, k.qh[ph] - k.Jh[ph] + 1);
            dy1 = std::max<int64_t>(dy1, k.qh[ph]);
            dx0 = std::min<int64_t>(dx0, k.qw[ph] - k.Jw[ph] + 1);
            dx1 = std::max<int64_t>(dx1, k.qw[ph]);
        }
    }
    if (dy0 > dy1 || dx0 > dx1) return false;  // no phase reads grad_out
    const int64_t Th = dy1 - dy0 + 1, Tw = dx1 - dx0 + 1;
    const int64_t Hr = cdiv(H, s), Wr = cdiv(W, s);
    const int64_t X = Wr + Tw - 1, R = Hr + Th - 1;
    if (X > 128 || N * R * 128 + 8192 > INT32_MAX) return false;
    PhaseDesc &d = t.ph[0];
    d.Hr = (int)Hr; d.Wr = (int)Wr;
    d.Jh = (int)Th; d.Jw = (int)Tw;
    d.qh = (int)(Th - 1 + dy0); d.qw = (int)(Tw - 1 + dx0);
    d.X = (int)X; d.R = (int)R;
    t.n_phases = 1;
    t.m_tile = 128;
    t.n_mtiles = 1;
    t.tile_p = 128;
    t.kc = 128 / esize;
    t.n_cchunks = (int)cdiv(Co, t.kc);
    t.stacked = 1;
    t.st_n = (int)round_up(std::max<int64_t>((int64_t)s * s * Ci, 16), 16);
    t.st_th = (int)Th; t.st_tw = (int)Tw;
    t.st_dy0 = (int)dy0; t.st_dx0 = (int)dx0;
    const int64_t w_unit = (int64_t)t.st_n * 128;
    const int64_t packed = (int64_t)t.n_cchunks * Th * Tw * w_unit;
    t.w_unit_bytes = (int)w_unit;
    t.packed_bytes = packed;
    t.epi_stage_bytes = 0;
    bool ok = false;
    // First choice: the column taps on N as well (TcParams::st_qhalo), so an
    // MMA covers st_tw taps at once (N = st_tw x st_n) and a tile issues
    // st_tw times fewer of them.  The quadrant-halo frame (X = 128, each
    // 32-element quadrant covering 32 - (st_tw - 1) output columns) keeps the
    // epilogue's column shifts inside one warp; it needs st_tw - 1 <= 3 and
    // Wr <= 4 (33 - st_tw).  Tiles of two frame rows (two M-blocks).  The
    // gather warps read grad_out straight from global memory (no raw slices:
    // a frame row is consecutive grad_out columns, so the loads coalesce, and
    // the two 80 KB-class G stages leave room for only two raw slots, too few
    // loads in flight); the weights stay resident when they fit, else stream
    // one row tap (st_tw taps) per stage.
    const int64_t nq = Tw * t.st_n;
    if (Tw >= 2 && Tw <= kStMaxTw && nq <= 256 && 4 * (33 - Tw) >= Wr) {
        const int rows = (int)std::min<int64_t>(2, Hr);
        t.st_qhalo = (int)(Tw - 1);
        t.st_mblocks = rows;
        t.rows_per_tile = rows;
        d.X = 128;
        d.p_tiles = (int)(N * cdiv(Hr, rows));
        d.hb = (int)((rows + Th - 1) * 128);
        t.hbp = d.hb;
        const int64_t g_stage = (int64_t)t.hbp * 128;
        t.g_stage_bytes = (int)g_stage;
        plan_raw_slices(p, esize, t, /*none=*/true);
        const int64_t w_stage = Tw * w_unit;  // one row tap: st_tw taps
        const int64_t fixed = smem_layout_bytes(0, 0, 2 * g_stage);
        const int64_t nw = std::min<int64_t>(std::min<int64_t>(kMaxW, Th * t.n_cchunks),
                                             (kSmemLimit - fixed) / w_stage);
        if (fixed + packed <= kSmemLimit) {  // resident weights
            ok = true;
            t.ng = 2;
            t.nw = 0;
            t.taps_per_w = (int)(Th * Tw);
            t.w_stage_bytes = (int)(Th * Tw * w_unit);
            t.smem_bytes = (int)(fixed + packed);
        } else if (nw >= 2) {
            ok = true;
            t.ng = 2;
            t.nw = (int)nw;
            t.taps_per_w = (int)Tw;
            t.w_stage_bytes = (int)w_stage;
            t.smem_bytes = (int)(fixed + nw * w_stage);
        } else {
            t.st_qhalo = 0;
            d.X = (int)X;
        }
    }
    // Otherwise, tile shapes tried in turn: two M-blocks of 128 positions
    // (whole frame rows up to 256 positions; the window's halo rows are then
    // shared by twice the outputs) with the weights streamed in tap groups,
    // then one M-block with the weights resident.  Each with raw slices when
    // a load mode applies (two or three slots), else the gather reads
    // grad_out directly.
    for (int mblocks = 2; mblocks >= 1 && !ok; --mblocks) {
        const int rows = (int)std::min<int64_t>(mblocks * 128 / X, Hr);
        if (mblocks == 2 && rows <= 128 / X) continue;  // no more rows than one M-block holds
        t.st_mblocks = mblocks;
        t.rows_per_tile = rows;
        d.p_tiles = (int)(N * cdiv(Hr, rows));
        d.hb = (int)(mblocks * 128 + (Th - 1) * X + (Tw - 1));
        t.hbp = (int)round_up(d.hb, 8);
        const int64_t g_stage = (int64_t)t.hbp * 128;
        t.g_stage_bytes = (int)g_stage;
        const int raw = plan_raw_slices(p, esize, t);
        // (two M-blocks: two raw slots, the rest of shared memory for weights)
        for (int nr = raw ? (mblocks == 2 ? 2 : 3) : 0; nr >= (raw ? 2 : 0) && !ok; --nr) {
            const int64_t fixed = smem_layout_bytes(0, (int64_t)nr * t.raw_slice_bytes, 2 * g_stage);
            if (mblocks == 1) {  // resident weights
                if (fixed + packed <= kSmemLimit) {
                    ok = true;
                    t.nw = 0;
                    t.taps_per_w = (int)(Th * Tw);
                    t.w_stage_bytes = (int)(Th * Tw * w_unit);
                    t.smem_bytes = (int)(fixed + packed);
                }
            } else {  // two weight stages of as many taps as fit
                const int64_t tpw = std::min<int64_t>(Th * Tw, (kSmemLimit - fixed) / (2 * w_unit));
                if (tpw >= 1) {
                    ok = true;
                    t.nw = 2;
                    t.taps_per_w = (int)tpw;
                    t.w_stage_bytes = (int)(tpw * w_unit);
                    t.smem_bytes = (int)(fixed + 2 * tpw * w_unit);
                }
            }
            if (ok) {
                t.raw_nr = nr;
                t.ng = 2;
            }
        }
        if (!ok && raw && mblocks == 1) {  // without raw slices: the gather reads grad_out directly
            plan_raw_slices(p, esize, t, /*none=*/true);
            const int64_t bytes = smem_layout_bytes(0, 0, packed + 2 * g_stage);
            if (bytes <= kSmemLimit) {
                ok = true;
                t.nw = 0;
                t.taps_per_w = (int)(Th * Tw);
                t.w_stage_bytes = (int)(Th * Tw * w_unit);
                t.ng = 2;
                t.smem_bytes = (int)bytes;
            }
        }
    }
    if (!ok) return false;
    t.raw_early = 0;
    t.total_tiles = d.p_tiles;
    t.tile_group = 1;
    const uint32_t fmt = dtype == DGRAD_F32 ? 2u : (dtype == DGRAD_BF16 ? 1u : 0u);
    const int ncols = t.st_qhalo ? (int)nq : t.st_n;  // MMA N = accumulator columns per M-block
    t.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(ncols >> 3) << 17) | ((uint32_t)(128 >> 4) << 24);
    uint32_t cols = 32;  // two buffers of st_mblocks accumulators of ncols columns
    while (cols < (uint32_t)(2 * t.st_mblocks * ncols)) cols *= 2;
    t.tmem_cols = cols;
    k.Ci = (int)Ci; k.Co = (int)Co; k.kH = (int)kH; k.kW = (int)kW; k.stride = s;
    k.m_tile = t.st_n; k.n_mtiles = 1; k.kc = t.kc; k.n_cchunks = t.n_cchunks;
    k.elems16 = 16 / esize;
    k.n_phases = s * s;
    k.stacked = 1;
    k.st_n = t.st_n; k.st_th = t.st_th; k.st_tw = t.st_tw; k.st_dy0 = t.st_dy0; k.st_dx0 = t.st_dx0;
    k.total_elems = packed / esize;
    plan->workspace = (size_t)packed;
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
    if (plan_stacked(p, plan->esize, dtype, plan)) {
        plan->kernel = DGRAD_KERNEL_TC;
        plan->tc_alt = plan->tc;
        return DGRAD_OK;
    }
    if (plan_tc(p, plan->esize, dtype, plan, /*pair=*/true)) {
        plan->kernel = DGRAD_KERNEL_TC;
        plan->tc_alt = plan->tc;  // pairing needs no TMA (staged epilogue without it)
        return DGRAD_OK;
    }
    if (plan_tc(p, plan->esize, dtype, plan)) {
        plan->kernel = DGRAD_KERNEL_TC;
        plan->tc_alt = plan->tc;
        TcParams v;
        if (forced_kernel == DGRAD_KERNEL_TC_POSM && plan_pm(p, plan->esize, plan->tc_alt, &v))
            plan->tc = v;
        else if (plan_frame64(p, plan->esize, plan->tc_alt, &v)) {
            plan->tc = v;
            // One stride-1 phase with resident weights (the general plan's
            // too): the kernel packs them from the weight tensor itself.
            plan->tc.w_raw = plan->tc_alt.w_raw = 1;
            plan->workspace = 0;
        }
        else if (plan_mn(p, plan->esize, plan->tc_alt, &v))
            plan->tc = v;
        else if (plan->esize == 2 && p.stride == 1 && plan->tc.nw == 0 && !plan->tc.pos_m) {
            // General mode, one stride-1 phase, resident weights: packed in
            // the kernel as on the 64-wide frame.
            plan->tc.w_raw = plan->tc_alt.w_raw = 1;
            plan->workspace = 0;
        }
        return DGRAD_OK;
    }
    if (forced_kernel == DGRAD_KERNEL_TC || forced_kernel == DGRAD_KERNEL_TC_POSM)
        return DGRAD_ERR_UNSUPPORTED;
    plan->kernel = DGRAD_KERNEL_SIMT;
    plan->workspace = 0;
    return DGRAD_OK;
}

}  // namespace dgrad
