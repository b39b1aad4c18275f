// dgrad_internal.h -- plan and kernel-parameter structures shared by the host
// planner (plan.cu / api.cu) and the kernels (pack.cu, dgrad_tc.cu,
// dgrad_simt.cu).  Not part of the public ABI.
//
// The sub-pixel phase split.  For stride s, grad_in pixel (ih, iw) belongs to
// phase (rh, rw) = (ih mod s, iw mod s) and sits at (a, b) = (ih div s, iw div
// s) of that phase's grid.  Following the divisibility test of the page's
// strided staging branch (conv2d_grad_input_gemm_coop.wgsl), tap kh reaches
// ih iff ih + ph - kh = s*oh.  Writing th = (rh + ph) mod s and qh = (rh + ph)
// div s, the taps of the phase are kh = s*j + th for j < Jh = ceil((kH - th) /
// s), and they read oh = a + qh - j.  So every phase is a dense stride-1
// correlation over the grad_out grid with its own (Jh x Jw) sub-kernel: no
// structural-zero products are ever issued.  Stride 1 is the single phase
// th = ph mod 1 = 0, qh = ph, Jh = kH.
//
// The frame.  Each phase's output positions are laid out in a linear space
// Lambda of pitch X = Wr + Jw - 1 and R = Hr + Jh - 1 rows per image; output
// (n, a, b) sits at Lambda = (n*R + a)*X + b.  The grad_out value that tap
// (j, i) needs for that output sits at Lambda + (Jh-1-j)*X + (Jw-1-i), where
// frame element (rho, kappa) of image n holds grad_out[n, rho-(Jh-1)+qh,
// kappa-(Jw-1)+qw] (zero outside the grad_out grid).  A tile of kTileP = 256
// consecutive outputs therefore needs one contiguous window of
// 256 + (Jh-1)*X + Jw-1 frame elements, and each tap is the same window seen
// from a different start: the tap loop runs backwards over the frame, which is
// the kernel flip of the forward-style correlation.
//
// The GEMM per tile is D[ci, position] += W[ci, co] * G[co, position] for
// each tap: input channels on the tcgen05 M side (64 or 128 rows), the 256
// positions on the N side (the tensor cores run at full rate only when N is
// wide), grad_out channels (128 bytes at a time) on K.
#pragma once

#include <cuda.h>

#include <cstddef>
#include <cstdint>

#include "nvtx_range.h"

namespace dgrad {

constexpr int kMaxPhases = 16;  // stride <= 4
constexpr int kTileP = 256;     // output positions per tile (tcgen05 N); 128 for very wide frames
constexpr int kEpiWarps = 8;    // warps 0..7: TMEM -> global epilogue (two per lane quadrant)
constexpr int kMmaWarp = 8;     // warp 8: TMEM alloc + MMA issue
constexpr int kWWarp = 9;       // warp 9: packed-weight bulk copies / raw grad_out TMA loads
constexpr int kGWarp0 = 10;     // warps 10..: grad_out gather
constexpr int kGWarps = 6;
constexpr int kThreads = 32 * (kGWarp0 + kGWarps);
constexpr int kSmemLimit = 232448;  // 227 KB dynamic shared memory per block
constexpr int kBarrierBytes = 1024;
// Shared memory of a plan: 1 KB to align the base, the barrier block, then the
// epilogue staging and the raw ring each rounded up to 1 KB, the G stages and
// the weights (multiples of 1 KB): the rings start on 1 KB boundaries, which
// the 128-byte swizzle pattern is tied to.
constexpr int64_t smem_layout_bytes(int64_t epi, int64_t raw, int64_t g_and_w) {
    return 1024 + kBarrierBytes + (epi + 1023) / 1024 * 1024 + (raw + 1023) / 1024 * 1024 + g_and_w;
}
constexpr int kEpiChunk = 32;                 // positions per step of the staged epilogue
constexpr int kEpiRowFloats = kEpiChunk + 1;  // padded staging row (conflict-free)
constexpr int kTmaBoxCi = 8;                  // channels per TMA store box (one box per warp)
constexpr int kMaxEarly = 4;                  // raw slices parked in G stage 1 at the start
constexpr int kRawNone = 0, kRawTiled = 1, kRawRows = 2, kRawPlanes = 3;  // TcParams::raw_mode
constexpr int kRawPlaneMaxBytes = 49152;      // largest whole-plane raw slice
constexpr int kMaxRaw = 8;                    // raw-slice ring slots
constexpr int kMaxW = 8;                      // streamed weight stages
constexpr int kMaxGatherRows = 6;             // window rows per gather thread (raw-slice gather)
constexpr int kMaxMnPieces = 13;              // 16-byte pieces per gather thread and stage (MN-major)
constexpr int kStMaxTw = 4;                   // stacked mode: column taps stacked on N (at most)
constexpr int kPmPitch = 64;  // positions-on-M mode: frame positions per grad_out row
constexpr int kPmLeft = 8;    // zero columns before grad_out column 0 in each frame row
constexpr int kPmMaxKw = 3;   // column taps stacked on N (kW x 64 columns)
constexpr int kPmEpiWarps = 16;  // positions-on-M roles: warps 0..15 epilogue (4 per quadrant),
constexpr int kPmMmaWarp = 16;   // 16 MMA, 17 raw loads + weights, 18..21 gather
constexpr int kPmWWarp = 17;
constexpr int kPmGWarp0 = 18;
constexpr int kPmGWarps = 4;
constexpr int kPmThreads = 32 * (kPmGWarp0 + kPmGWarps);
constexpr int kPmGroups = 6;  // ldmatrix.x4 groups per gather warp and raw slice (at most)
constexpr int kF64Groups = 7; // the same with the general mode's kGWarps gather warps
// Boundary-exchange buffer of the positions-on-M epilogue: 8 warp pairs x 2
// slots x 3 (tap, lane) values x 16 floats: block 1 of lane 31, block 2 of
// lanes 30 and 31.
constexpr int kPmXSlotBytes = 3 * 16 * 4;
constexpr int kPmXBytes = 8 * 2 * kPmXSlotBytes;

struct PhaseDesc {
    int rh, rw;         // residues of (ih, iw) modulo the stride
    int Hr, Wr;         // grad_in pixels of this phase per image (rows, columns)
    int Jh, Jw;         // taps per axis (0: no tap reaches this phase)
    int th, tw;         // kh = s*j + th, kw = s*i + tw
    int qh, qw;         // oh = a + qh - j, ow = b + qw - i
    int X, R;           // frame pitch and frame rows per image
    int p_tiles;        // position tiles of this phase
    int hb;             // frame elements one tile needs
    int64_t tile_begin; // first global tile of this phase (p-tiles x m-tiles)
    int64_t pack_off;   // byte offset of this phase's packed weights
};

struct TcParams {
    CUtensorMap out_map;    // grad_in as [N][Ci][H][W] float32 (TMA store epilogue only)
    CUtensorMap in_map;     // grad_out as [N][Co][OH][OW] (TMA gather only)
    const void *grad_out;
    const void *packed;
    float *grad_in;
    int N, Ci, H, W, Co, OH, OW, stride;
    int esize;              // bytes per grad_out / weight element
    int n_phases;
    int m_tile, n_mtiles;   // input channels per tile (MMA M: 64 or 128) and tiles over Ci
    int tile_p;             // accumulator columns per tile (MMA N)
    int rows_per_tile;      // > 0: tiles are whole frame rows of one phase, this many per tile
    int epi_tma;            // 1: epilogue stores through TMA (set at launch)
    int epi_stage_bytes;    // shared-memory staging of the epilogue
    int epi_boxes;          // TMA store boxes per epilogue warp (1, or 2: double-buffered)
    int epi_box_ci;         // channels per TMA store box: 8, or 16 (64-row tiles, 16x256b reads)
    // Raw-slice gather (whole-row tiles): grad_out rows arrive as [raw_cs
    // channels][raw_br rows][raw_bw columns] slices starting at column raw_x0,
    // through a ring of raw_nr slots, and are transposed in shared memory into
    // the frame window.
    int gather_tma;         // 1: use it (set at launch)
    int raw_nr, raw_cs, raw_br, raw_bw, raw_x0, raw_slice_bytes;
    // How raw slices are loaded (kRaw*): a 4-D TMA tensor map whose rows are
    // raw_rowg grad_out rows (a multiple of 16 bytes), one 1-D bulk copy per
    // channel of a row range (channel planes a multiple of 16 bytes), or one
    // 1-D bulk copy of whole planes of raw_cs consecutive channels (tiles that
    // cover whole images).  With raw_rowg > 1 a slice starts on a row that is
    // a multiple of raw_rowg.
    int raw_mode, raw_rowg;
    // 1: tiles are ordered (position tile, phase, channel tile), so the phases
    // of the same output rows run side by side (all phases have p_tiles).
    int interleave;
    // The first raw_early slices (at most kMaxEarly) land in G stage 1, idle
    // until the second tile, so more of the first tile's grad_out is in flight.
    int raw_early;
    int kc, n_cchunks;      // grad_out channels per stage (128 bytes), stages per tile
    int hbp;                // frame elements per G stage (multiple of 8)
    int g_stage_bytes;      // grad_out frame window stage
    int w_unit_bytes;       // one tap x one channel chunk of packed weights
    int w_stage_bytes;      // one streamed weight stage (taps_per_w taps)
    int taps_per_w;         // taps per streamed weight stage
    int ng, nw;             // ring depths; nw == 0: all packed weights resident
    int64_t packed_bytes;
    int64_t total_tiles;
    uint32_t idesc;         // tcgen05 instruction descriptor
    uint32_t tmem_cols;
    int smem_bytes;
    int debug_flags;
    uint64_t wait_limit_ns;
    // Positions-on-M mode (stride 1, Ci <= 64, Co <= 64, kW <= 3, 16-bit,
    // W <= 56): the MMA takes 128 frame positions on M and the kW column taps
    // of one kernel row stacked on N (kW x 64 columns); the frame pitch is 64
    // with kPmLeft zero columns in front of each grad_out row.  See dgrad_tc.cu.
    int pos_m;
    // 64-wide frame in the general mode (stride 1, 16-bit, W <= 56): the
    // window layout of positions-on-M mode (kPmLeft zero columns, then the
    // grad_out row), filled by the same ldmatrix transpose; tap (j, i)
    // reads it from row (Jh-1-j) * 64 + (Jw-1-i) + view0.
    int frame64;
    int view0;
    int pad_w;              // padding_w: start of the row-tap views in the window
    int pm_rows;            // window rows holding grad_out data (raw_br >= pm_rows)
    // 1x1 stride-1 convolutions whose tiles are whole images (a plain GEMM per
    // image): the grad_out operand is read MN-major -- [channel][position], as
    // NCHW memory holds it -- from 128-byte swizzled atoms of 8 channels x 64
    // positions, so the gather regroups 16-byte pieces instead of transposing.
    // Atom (channel group g, position block m) sits at g * 1024 * mn_atoms +
    // m * 1024 in a G stage.
    int mn_b;
    int mn_atoms;           // 64-position atoms per channel group (tile_p <= 64 * mn_atoms)
    // Stacked-phase mode (few input channels, stride > 1): 128 positions of
    // the phase grid on the MMA M side, every phase's input channels stacked
    // on N (column n = (rh * stride + rw) * Ci + ci, st_n columns), K = grad_out
    // channels x the st_th x st_tw window taps (dy, dx) = (st_dy0 + t / st_tw,
    // st_dx0 + t mod st_tw) that any phase uses.  The single frame of ph[0]
    // holds grad_out[a + dy][b + dx] for output (a, b); A = that frame seen
    // from the tap's shift, B = the packed weights of (channel chunk, tap),
    // st_n rows, zero where a phase does not use the tap.
    int stacked;
    int st_n, st_th, st_tw, st_dy0, st_dx0;
    int st_mblocks;         // 128-position MMA M-blocks per tile (1 or 2), one accumulator each
    // > 0: the stacked mode with the column taps on N as well (N = st_tw x
    // st_n: column block i of lane e holds the window tap dx = st_dx0 + i of
    // frame element e), on a quadrant-halo frame: X = 128 elements per frame
    // row, element e = 32q + l holding frame column (32 - st_qhalo) q + l, so
    // each 32-lane TMEM quadrant covers 32 - st_qhalo outputs plus st_qhalo =
    // st_tw - 1 halo columns, and the epilogue adds block i of lane l + i
    // within the warp.  An M-block is one frame row (one output row of the
    // phase grid); K = grad_out channels x the st_th row taps.
    int st_qhalo;
    // A CTA takes tiles in groups of tile_group consecutive tiles (groups
    // dealt round-robin over the grid).  pair_rw (stride 2, four phases
    // interleaved, one channel tile): tiles 2u and 2u + 1 are the column
    // phases rw = 0 and 1 of the same output rows, gathered once (one frame
    // pitch for all phases) into a pair of TMEM accumulators, and one epilogue
    // interleaves them into whole grad_in rows.
    int tile_group;
    int pair_rw;
    int acc_single;         // 1: one TMEM accumulator buffer (the epilogue does not overlap the MMA)
    // 1: `packed` is the weight tensor itself ([Co][Ci][kH][kW], 16-bit, one
    // stride-1 phase, resident weights): the epilogue warps build the packed
    // image in shared memory while the first grad_out tile loads, so no pack
    // kernel runs before the launch.
    int w_raw;
    PhaseDesc ph[kMaxPhases];
};

// Frame column held by frame element x of a row: x itself, or on the
// quadrant-halo frame (TcParams::st_qhalo) (32 - halo) * (x / 32) + x mod 32.
__host__ __device__ __forceinline__ int frame_column(int x, int qhalo) {
    return qhalo > 0 ? (32 - qhalo) * (x >> 5) + (x & 31) : x;
}

struct PackParams {
    int Ci, Co, kH, kW, stride;
    // Stacked-phase layout (TcParams::stacked): per channel chunk and window
    // tap, st_n rows; phase k = rh * stride + rw uses tap (dy, dx) when
    // j = qh[k] - dy and i = qw[k] - dx are taps of it.
    int stacked, st_n, st_th, st_tw, st_dy0, st_dx0;
    int qh[kMaxPhases], qw[kMaxPhases];
    int m_tile, n_mtiles, kc, n_cchunks, elems16;  // elems16: elements per 16 bytes
    int n_phases;
    int64_t total_elems;
    int64_t elem_begin[kMaxPhases + 1];
    int th[kMaxPhases], tw[kMaxPhases], Jh[kMaxPhases], Jw[kMaxPhases];
};

// The strided forward convolution as a stride-1 valid correlation (api.cu,
// pack.cu): residues r of kh - ph (c of kw - pw) modulo the stride that some
// tap reaches, X''[n][(pr, pc, ci)][a][b] = x[n][ci][s (a + jmin) + R[pr]]
// [s (b + imin) + C[pc]] (zero outside the image), W''[co][(pr, pc, ci)][j][i]
// = w[co][ci][s (j + jmin) + R[pr] + ph][s (i + imin) + C[pc] + pw] (zero
// outside the kernel).
constexpr int kMaxFwdStride = 8;
struct FwdSplit {
    int N, Ci, H, W, Co, kH, kW, s, ph, pw;
    int nr, nc, R[kMaxFwdStride], C[kMaxFwdStride];
    int jmin, imin, KH, KW, Hx, Wx, OH, OW;
};

struct SimtParams {
    int N, Ci, H, W, Co, kH, kW, stride, ph, pw, OH, OW;
};

// A complete host-side plan for one (params, dtype) pair.
struct Plan {
    int dtype;
    int esize;
    int kernel;          // DGRAD_KERNEL_TC or DGRAD_KERNEL_SIMT
    TcParams tc;         // valid when kernel == TC
    TcParams tc_alt;     // general-mode plan with the Wr + Jw - 1 frame (same packed weights),
                         // used when tc needs TMA (gather or store) that the pointers rule out
    PackParams pack;     // valid when kernel == TC
    SimtParams simt;
    size_t workspace;    // packed-weight bytes (TC without w_raw), 0 otherwise
};

// plan.cu: validation + planning.  Returns a dgrad_status.
int make_plan(const void *params, int dtype, int forced_kernel, Plan *out);
// api.cu: make_plan with the process-wide kernel choice, debug flags and wait limit.
int plan_with_settings(const void *params, int dtype, Plan *out);

// Launchers (return cudaError_t as int).
int launch_pack(const Plan &plan, const void *weight, void *packed, void *stream);
// wt[ci][co][kh][kw] = w[co][ci][kH-1-kh][kW-1-kw] (pack.cu).
int launch_flip_transpose(const void *w, void *wt, int Co, int Ci, int kH, int kW, int esize,
                          void *stream);
// X'' and W'' of a FwdSplit (esize 2 or 4), in `stream` order.
int launch_space_to_depth(const FwdSplit &f, const void *x, void *xs, int esize, void *stream);
int launch_split_weights(const FwdSplit &f, const void *w, void *ws, int esize, void *stream);
int launch_tc(const Plan &plan, const void *grad_out, const void *packed, float *grad_in,
              void *stream);
int launch_simt(const Plan &plan, const void *grad_out, const void *weight, float *grad_in,
                void *stream);
int tc_read_and_clear_error(unsigned int *out);  // cudaError_t

}  // namespace dgrad
