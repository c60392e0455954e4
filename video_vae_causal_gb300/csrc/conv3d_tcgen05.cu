// conv3d_tcgen05.cu -- host side of CausalConv3d as an implicit GEMM on the
// sm_103a tensor cores: argument checks, the tiling plan, TMA descriptors and
// the launch.  The kernel itself is in conv3d_tcgen05.cuh; its instantiations
// are spread over conv3d_kernels_*.cu so that they compile in parallel.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "conv3d_tcgen05.cuh"
#include "kernels.h"
#include "norm_act.cuh"

namespace wanvae {
namespace {

using namespace conv;

// Kernel-variant overrides (set_kernel_variant): -1 = chosen per call.
enum { kVarPair = 0, kVarHalo = 1, kVarWide = 2, kVarNarrow = 3, kVarFuse = 4, kNumVar = 5 };
std::atomic<int> g_variant[kNumVar] = {{-1}, {-1}, {-1}, {-1}, {-1}};

// ------------------------------------------------------------------ host
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
typedef CUresult (*EncodeIm2colFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const int *,
                                   const int *, cuuint32_t, cuuint32_t, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn g_encode_tiled = nullptr;
EncodeIm2colFn g_encode_im2col = nullptr;
std::once_flag g_encode_once;

bool load_encoders() {
    std::call_once(g_encode_once, [] {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_tiled = reinterpret_cast<EncodeTiledFn>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &fn, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_im2col = reinterpret_cast<EncodeIm2colFn>(fn);
    });
    return g_encode_tiled && g_encode_im2col;
}

CUtensorMapSwizzle swizzle_for(int sw) {
    return sw == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                    : (sw == 32 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

// 2-D bf16 matrix [rows][cols] (cols contiguous), box (box_cols x box_rows).
bool encode_2d(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_cols,
               uint32_t box_rows, int sw) {
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t es[2] = {1, 1};
    return g_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(sw),
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// NHWC im2col view of `frames` frames of H x W x C, bounding box shrunk by 1
// on every side of H and W (the 3x3 window's one-element pad), 128 pixels of
// `sw` channels per load.
bool encode_im2col(CUtensorMap *m, const void *base, int C, int W, int H, int frames, int sw) {
    cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)frames};
    cuuint64_t strides[3] = {(cuuint64_t)C * 2, (cuuint64_t)W * C * 2, (cuuint64_t)H * W * C * 2};
    int lower[2] = {-1, -1};
    int upper[2] = {-1, -1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return g_encode_im2col(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                           strides, lower, upper, (cuuint32_t)sw, (cuuint32_t)kBlockM, es,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(sw),
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [frames][HW][C] bf16 view with a (64 channels x 128 rows x 1 frame) box,
// 128-byte swizzle: rows of a tile past the frame's end are out of bounds
// (stores skip them, loads read zeros).
bool encode_frames(CUtensorMap *m, const void *base, int C, int HW, int frames) {
    cuuint64_t dims[3] = {(cuuint64_t)C, (cuuint64_t)HW, (cuuint64_t)frames};
    cuuint64_t strides[2] = {(cuuint64_t)C * 2, (cuuint64_t)HW * C * 2};
    cuuint32_t box[3] = {64, (cuuint32_t)kBlockM, 1};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Weights [c_out][K] (K contiguous) viewed as [n_pieces][pair][half_n][K] with
// a box of (sw, half_n, 1, n_pieces): one load brings a CTA's rows of every
// N-piece, landing as [piece][half_n rows][sw] -- the B layout the MMAs read.
// With nsub > 0 a fifth dimension of nsub sub-tiles (sw channels apart in K)
// lands as [sub-tile][piece][half_n rows][sw]: one load for a whole chunk.
//
// Narrow layers (c_out < 16, n_pieces = 1, the piece padded to 16 rows per
// CTA): the row dimension is the true c_out and the pair dimension has extent
// 1; a CTA's box starts at row rank * half_n, and rows past c_out read as zeros.
bool encode_weights(CUtensorMap *m, const void *base, uint64_t K, int c_out, int pair,
                    int n_pieces, int sw, int nsub, int npad = 0, int nphase = 1) {
    const bool narrow = npad > c_out;
    const int piece_n = (narrow ? npad : c_out) / n_pieces, half_n = piece_n / pair;
    // (an upsampler's nphase weight sets follow each other: nphase x n_pieces pieces)
    cuuint64_t dims[5] = {K, (cuuint64_t)(narrow ? c_out : half_n),
                          (cuuint64_t)(narrow ? 1 : pair), (cuuint64_t)(n_pieces * nphase),
                          (cuuint64_t)(nsub > 0 ? nsub : 1)};
    cuuint64_t strides[4] = {K * 2, (cuuint64_t)half_n * K * 2, (cuuint64_t)piece_n * K * 2,
                             (cuuint64_t)sw * 2};
    cuuint32_t box[5] = {(cuuint32_t)sw, (cuuint32_t)half_n, 1, (cuuint32_t)n_pieces,
                         (cuuint32_t)(nsub > 0 ? nsub : 1)};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return g_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, nsub > 0 ? 5 : 4,
                          const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(sw),
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Weights [c_out][27 * c_in] of one N piece (n_pieces == 1) viewed as
// (K, half_n rows, pair rank, nsub sub-tiles sw apart, tb taps c_in apart): one
// box holds this CTA's rows of tb consecutive taps of one channel chunk, laid
// out [tap][sub-tile][row][sw], the order the halo-mode MMAs step through.
bool encode_weight_taps(CUtensorMap *m, const void *base, uint64_t K, int c_in, int c_out,
                        int pair, int sw, int nsub, int tb, int npad = 0, int nphase = 1) {
    const bool narrow = npad > c_out;  // as in encode_weights
    const int half_n = (narrow ? npad : c_out) / pair;
    // (an upsampler's nphase weight sets follow each other along the rank dimension)
    cuuint64_t dims[5] = {K, (cuuint64_t)(narrow ? c_out : half_n),
                          (cuuint64_t)(narrow ? 1 : pair * nphase), (cuuint64_t)nsub,
                          (cuuint64_t)tb};
    cuuint64_t strides[4] = {K * 2, (cuuint64_t)half_n * K * 2, (cuuint64_t)sw * 2,
                             (cuuint64_t)c_in * 2};
    cuuint32_t box[5] = {(cuuint32_t)sw, (cuuint32_t)half_n, 1, (cuuint32_t)nsub,
                         (cuuint32_t)tb};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return g_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(sw),
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// NHWC input as (C, W, H, frames) with a (sw, halo_w, 18, 1) box: the 18 x
// halo_w pixels around a patch, sw channels each, land as one swizzled row
// per pixel (row-major over the halo) -- the layout the halo-mode windows
// read.  Pixels outside the frame read as zeros (the conv's spatial pad).
bool encode_halo(CUtensorMap *m, const void *base, int C, int W, int H, int frames, int sw,
                 int halo_w) {
    cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)frames};
    cuuint64_t strides[3] = {(cuuint64_t)C * 2, (cuuint64_t)W * C * 2, (cuuint64_t)H * W * C * 2};
    cuuint32_t box[4] = {(cuuint32_t)sw, (cuuint32_t)halo_w, kHaloH, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return g_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(sw),
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// NHWC input viewed as (8 channels, W, H, C/8 planes, frames): one 18 x
// halo_w pixel box of `chunk` channels lands as planes [chunk/8][18][halo_w][8]
// with 16 bytes per pixel, the no-swizzle layout of halo planes.
bool encode_halo_planes(CUtensorMap *m, const void *base, int C, int W, int H, int frames,
                        int chunk, int halo_w) {
    cuuint64_t dims[5] = {8, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)(C / 8),
                          (cuuint64_t)frames};
    cuuint64_t strides[4] = {(cuuint64_t)C * 2, (cuuint64_t)W * C * 2, 16,
                             (cuuint64_t)H * W * C * 2};
    cuuint32_t box[5] = {8, (cuuint32_t)halo_w, kHaloH, (cuuint32_t)(chunk / 8), 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return g_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// NHWC tensor as (C, W, H, frames) with a (box_c, 8, 16, 1) box: one 16 x 8
// patch, swizzled by box_c (its smem rows are the patch's pixels in order).
bool encode_patch(CUtensorMap *m, const void *base, int C, int W, int H, int frames, int box_c,
                  int sw) {
    cuuint64_t dims[4] = {(cuuint64_t)C, (cuuint64_t)W, (cuuint64_t)H, (cuuint64_t)frames};
    cuuint64_t strides[3] = {(cuuint64_t)C * 2, (cuuint64_t)W * C * 2, (cuuint64_t)H * W * C * 2};
    cuuint32_t box[4] = {(cuuint32_t)box_c, 8, 16, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return g_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle_for(sw),
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The upsampler's output y [frames][2H][2W][C] seen per sub-pixel phase
// (a, b): as (b C + c, j, a, i, frame), the element at phase coordinates
// b C + c (dimension 0 spans both column phases' channels), column j, row
// phase a, row i is y[frame][2i + a][2j + b][c].  A (box_c, 8, 1, 4, 1) box is
// one epilogue warp's 4 x 8 low-res pixels of one phase, box_c channels each.
bool encode_phase_view(CUtensorMap *m, const void *base, int C, int W, int H, int frames,
                       int box_c) {
    cuuint64_t dims[5] = {(cuuint64_t)2 * C, (cuuint64_t)W, 2, (cuuint64_t)H,
                          (cuuint64_t)frames};
    cuuint64_t strides[4] = {(cuuint64_t)2 * C * 2, (cuuint64_t)2 * W * C * 2,
                             (cuuint64_t)4 * W * C * 2, (cuuint64_t)4 * H * W * C * 2};
    cuuint32_t box[5] = {(cuuint32_t)box_c, 8, 1, 4, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return g_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void *>(base), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int pick_sw(int c) { return c % 64 == 0 ? 64 : (c % 32 == 0 ? 32 : 16); }

// Channels per phase-view store box of the upsampler's epilogue: 48 where
// both column halves of the eight-warp split are multiples of 48 (one box per
// warp and sub-tile at c_out = 96), else 16.
int up_box_channels(int c_out) {
    const int c_split = (c_out / 2 + 15) / 16 * 16;
    return (c_split % 48 == 0 && (c_out - c_split) % 48 == 0) ? 48 : 16;
}

struct Plan {
    int pair;  // 1: one CTA per 128-row tile; 2: CTA pair per 256 rows (cta_group::2)
    int sw, nsub, kc_main, kc_short, n_pieces, piece_n, stages;
    uint32_t a_sub, b_sub, a_bytes, stage_bytes;
    uint32_t off_bars, off_misc, off_vec, smem_bytes;
    int acc_cols, nacc, tmem_cols;
    int staged;
    uint32_t off_stage;
    int halo;  // 16 x 8 patch tiles with halo loads
    int itb;   // im2col: taps per stage
    int tb;  // spatial taps per weight stage (halo mode)
    int nq, halo_w;  // sub-tiles per CTA tile, halo width in pixels (halo mode)
    uint32_t stg_warp;  // epilogue staging bytes per warp
    int narrow, npad;  // c_out < 16: N padded to npad
    uint32_t sub_stride;  // halo rows: bytes between sw-channel regions
    int halo_rows;        // halo layout: swizzled pixel rows (sw = 64, 32) or 8-channel planes
    int acc_stride;
    uint32_t off_a, a_stride, a_tx;
    int na;  // halo mode: A ring buffers
    int fuse;  // the input norm fused into the halo loads (conv3d_transform warps)
};

// Halo tiles (16 x 8 patches, one halo load per temporal tap and channel
// chunk feeding all nine spatial taps) move ~6x fewer A bytes and 9x fewer A
// loads than per-tap im2col, but cover H x W in whole patches: chosen when the
// patches tile the frame exactly.  The choice depends on the frame, never on
// T, so that a clip run frame by frame and run whole use the same tiles (and
// give the same bits); pick_ragged_halo adds halo tiles for one-frame calls
// where both tilings give the same bits.  The kernel-variant setting
// (set_kernel_variant) can force either.
int halo_choice(const ConvSpec &s) {
    if (s.k != 3) return 0;
    const int v = g_variant[kVarHalo].load(std::memory_order_relaxed);
    if (v == 0 || v == 1) return v;
    return s.H % 16 == 0 && s.W % 8 == 0;
}

// CTA pairs halve each CTA's share of the B (weight) operand -- half the
// shared-memory bytes per stage, so a deeper pipeline, and half the L2->SM
// traffic for B.  The kernel-variant setting can select the single-CTA kernel.
int pair_choice() {
    return g_variant[kVarPair].load(std::memory_order_relaxed) == 1 ? 1 : 2;
}

// Wide halo tiles (16 x 16 patches, two accumulators per CTA) where the
// patches tile the frame, the layer is narrow enough (make_plan checks c_out
// and the shortcut) and a frame holds at least 16 of them across the batch: a
// small frame spreads better over the SMs as twice as many 16 x 8 tiles (the
// 16 x 16 tiny clip: 0.034 -> 0.027 ms).  Per frame, not per clip (see
// halo_choice).  The kernel-variant setting can force either.
int wide_choice(const ConvSpec &s, int halo) {
    if (!halo) return 0;
    const int v = g_variant[kVarWide].load(std::memory_order_relaxed);
    if (v == 0 || v == 1) return v;
    return s.H % 16 == 0 && s.W % 16 == 0 && (int64_t)s.B * (s.H / 16) * (s.W / 16) >= 16;
}

bool make_plan(const ConvSpec &s, Plan &pl, int pair, int halo, int wide) {
    pl.pair = pair;
    pl.halo = halo;
    // Wide halo tiles: 16 x 16 patches, two 128-row sub-tiles per CTA, so
    // every weight stage feeds twice the MMAs.  Two double-buffered
    // accumulators per CTA must fit TMEM (c_out <= 128); no shortcut segment.
    pl.nq = (halo && wide) ? 2 : 1;
    if (pl.nq == 2 && (s.sc_in || s.c_out > 128)) return false;
    pl.halo_w = 8 * pl.nq + 2;
    int sw = pick_sw(s.c_in);
    if (s.sc_in) {
        const int sw2 = pick_sw(s.c_sc);
        if (sw2 < sw) sw = sw2;
    }
    pl.sw = sw;
    // Halo layout: 64- and 32-channel chunks as one 128- or 64-byte swizzled
    // row per pixel, 16-channel ones as 8-channel planes of 16 bytes per
    // pixel.  TMA moves about one box row per clock per SM whatever its width
    // (measured: planes 16 B/clk, 64-byte rows 64, 128-byte rows ~108), so the
    // widest rows keep the halo loads off the critical path.  A rows region:
    // 18 x halo_w rows, aligned to its swizzle pattern (1024 B for 128-byte
    // rows, 512 B for 64-byte rows).
    pl.halo_rows = sw == 64 || sw == 32;
    {
        const uint32_t atom = sw == 64 ? 1023u : 511u;
        pl.sub_stride = ((uint32_t)(kHaloH * pl.halo_w) * (uint32_t)sw * 2u + atom) & ~atom;
    }
    // N split into equal pieces of at most 256 columns, each a multiple of
    // 16 * pair (a pair splits every piece's rows between its two CTAs).
    // Narrow layers (c_out < 16) pad N to 16 rows per CTA; their weight rows
    // past c_out are TMA out-of-bounds zeros and only c_out columns are stored.
    pl.narrow = s.c_out < 16;
    if (pl.narrow && (s.sc_in || s.epi != kEpiBias)) return false;
    pl.npad = pl.narrow ? 16 * pair : s.c_out;
    pl.n_pieces = 0;
    for (int np = 1; np <= pl.npad / 16; ++np) {
        if (pl.npad % np == 0 && (pl.npad / np) % (16 * pair) == 0 && pl.npad / np <= 256) {
            pl.n_pieces = np;
            break;
        }
    }
    if (!pl.n_pieces) return false;
    pl.piece_n = pl.npad / pl.n_pieces;
    pl.acc_cols = (pl.npad + 31) / 32 * 32;
    pl.acc_stride = pl.nq * pl.acc_cols;
    pl.nacc = 2 * pl.acc_stride <= 512 ? 2 : 1;
    if (pl.nq == 2 && pl.nacc != 2) return false;
    int cols = pl.nacc * pl.acc_stride;
    pl.tmem_cols = 32;
    while (pl.tmem_cols < cols) pl.tmem_cols *= 2;
    if (pl.tmem_cols > 512) return false;

    const uint32_t b_rows = (uint32_t)(pl.npad / pair);
    const int g_main = s.c_in / sw, g_sc = s.sc_in ? s.c_sc / sw : g_main;
    const int min_stages = pair == 2 ? 4 : 3;
    // Whole-tile staged epilogue when a single TMEM accumulator leaves the
    // tensor core idle during the epilogue (c_out > 256) and the bf16 tile
    // fits next to a 3-deep pipeline.
    const uint32_t stage_tile = (uint32_t)kBlockM * s.c_out * 2u;
    const uint32_t fixed = 1024 /*align*/ + 1024 /*bars+misc*/ + 2u * 4u * s.c_out +
                           4u * 4u * kBlockM /*norm partial sums*/;
    pl.staged = 0;
    if (s.up2d && pl.nacc != 2) return false;  // its scattered stores use the direct epilogue
    if (pl.nacc == 1 && s.c_out % 64 == 0) {
        const uint32_t sb1 = (kBlockM + b_rows) * (uint32_t)sw * 2u;
        if (3u * ((sb1 + 1023u) & ~1023u) + fixed + stage_tile <= (uint32_t)kSmemBudget)
            pl.staged = 1;
    }
    // Epilogue staging per warp: 32 rows x 32 channels, or for the
    // upsampler's phase-view stores on halo tiles the warp's whole channel
    // share of a sub-tile (its boxes leave by TMA after the last chunk).
    {
        const uint32_t c_split = (uint32_t)((s.c_out / 2 + 15) / 16 * 16);
        pl.stg_warp = (s.up2d && halo && 64u * c_split > kStageBytesPerWarp)
                          ? 64u * c_split
                          : kStageBytesPerWarp;
    }
    const uint32_t reserve = fixed + (pl.staged ? stage_tile : (uint32_t)kEpiWarps * pl.stg_warp);
    const int need_stages = pl.staged ? 3 : min_stages;
    if (halo) {
        // Halo ring (2 buffers of 18 x halo_w pixels x chunk channels) + a ring of
        // weight stages of tb spatial taps each.  Every stage costs the MMA
        // issuer one barrier access, so take the (chunk, tb) with the fewest
        // stages per tile among those that leave a deep enough ring (>= 3
        // stages of 3 taps, >= need_stages of one tap); 3-tap stages need the
        // weights of one CTA in one piece (n_pieces == 1).
        pl.nsub = 0;
        pl.tb = 1;
        pl.itb = 1;
        int best_waits = 0, best_stages = 0;
        for (int d = 4; d >= 1; --d) {
            if (d * sw > 128 || g_main % d || g_sc % d) continue;
            const uint32_t ha =
                pl.halo_rows ? (uint32_t)d * pl.sub_stride
                             : ((uint32_t)(pl.halo_w * kHaloH) * d * sw * 2u + 1023u) & ~1023u;
            // 3-tap stages (a row of the 3 x 3 taps), or for the upsampler
            // 4-tap stages (a phase's 2 x 2 taps); else one tap per stage
            for (int tb = s.up2d ? 4 : 3; tb >= 1; tb = tb > 1 ? 1 : 0) {
                if (tb > 1 && pl.n_pieces != 1) continue;
                const uint32_t bs = ((uint32_t)(tb * d) * b_rows * sw * 2u + 1023u) & ~1023u;
                if (2u * ha + reserve >= (uint32_t)kSmemBudget) continue;
                int st = (int)(((uint32_t)kSmemBudget - reserve - 2u * ha) / bs);
                if (st > 8) st = 8;
                if (st < (tb > 1 ? 3 : need_stages)) continue;
                const int waits = (s.up2d ? 4 : 27) * (g_main / d) / tb + (s.sc_in ? g_sc / d : 0);
                if (!pl.nsub || waits < best_waits || (waits == best_waits && st > best_stages)) {
                    pl.nsub = d;
                    pl.tb = tb;
                    best_waits = waits;
                    best_stages = st;
                }
            }
        }
        if (!pl.nsub) return false;
        const int d = pl.nsub;
        pl.kc_main = g_main / d;
        pl.kc_short = s.sc_in ? g_sc / d : 0;
        pl.a_sub = (uint32_t)kBlockM * sw * 2;  // one x-patch sub-tile (shortcut)
        pl.b_sub = b_rows * sw * 2;
        pl.a_tx = (uint32_t)(pl.halo_w * kHaloH) * d * sw * 2u;
        pl.a_stride = pl.halo_rows ? (uint32_t)d * pl.sub_stride : (pl.a_tx + 1023u) & ~1023u;
        pl.off_a = 0;
        pl.stage_bytes = (pl.b_sub * d * (uint32_t)pl.tb + 1023u) & ~1023u;
        // A halo of the upsampler feeds a single stage (one phase's four
        // taps), so two halo buffers would let its loads run only one stage
        // ahead of the MMAs: a third where three weight stages still fit.
        pl.na = 2;
        if (s.up2d && 3u * pl.a_stride + 3u * pl.stage_bytes + reserve <= (uint32_t)kSmemBudget)
            pl.na = 3;
        // the weight ring starts here, 1024-aligned (64-byte-row halos are
        // only 512-aligned)
        pl.a_bytes = ((uint32_t)pl.na * pl.a_stride + 1023u) & ~1023u;
        pl.stages = (int)((kSmemBudget - reserve - pl.a_bytes) / pl.stage_bytes);
        if (pl.stages > 8) pl.stages = 8;
        if (pl.stages < 2) return false;
        uint32_t off = pl.a_bytes + pl.stage_bytes * pl.stages;
        pl.off_stage = off;
        if (pl.staged) off += stage_tile;
        pl.off_bars = off;
        pl.off_misc = pl.off_bars + 8u * (2 * pl.stages + 14);
        pl.off_vec = (pl.off_misc + 24u + 15u) & ~15u;  // TMEM slot, abort flag, producer state
        pl.smem_bytes = 1024u + pl.off_vec + 2u * 4u * s.c_out + 4u * 4u * kBlockM +
                        (s.up2d ? 128u : 0u) /*staging alignment for TMA stores*/ +
                        (pl.staged ? 0u : (uint32_t)kEpiWarps * pl.stg_warp);
        // The input norm can ride on the halo loads when one chunk holds every
        // channel of a pixel (its norm is then complete in one halo), with no
        // shortcut segment and two accumulators (four epilogue warps keep up).
        // Only on request (set_kernel_variant): measured slower than the
        // separate pass, since every input voxel is normalised once per
        // temporal tap and halo it falls in (about 3.8 times) by four warps.
        {
            const int L = nact_lanes(s.c_in), vpt = (s.c_in / 8) / L;
            pl.fuse = s.norm_in && s.k == 3 && !s.up2d && !s.up_t && !s.sc_in &&
                      pl.kc_main == 1 && pl.nsub * sw == s.c_in && pl.nacc == 2 &&
                      !pl.staged && vpt <= kMaxNormVpt &&
                      g_variant[kVarFuse].load(std::memory_order_relaxed) == 1;
        }
        if (pl.smem_bytes < 120u * 1024u) pl.smem_bytes = 120u * 1024u;
        return pl.smem_bytes <= (uint32_t)kSmemBudget;
    }
    pl.off_a = 0;
    pl.a_stride = 0;
    pl.a_tx = 0;
    pl.na = 2;
    pl.tb = 1;
    pl.nsub = 1;
    pl.fuse = 0;
    for (int d = 4; d >= 1; --d) {
        if (d * sw > 128 || g_main % d || g_sc % d) continue;
        const uint32_t sb = (uint32_t)d * (kBlockM + b_rows) * sw * 2;
        if (need_stages * ((sb + 1023u) & ~1023u) + reserve <= (uint32_t)kSmemBudget) {
            pl.nsub = d;
            break;
        }
    }
    pl.kc_main = g_main / pl.nsub;
    pl.kc_short = s.sc_in ? g_sc / pl.nsub : 0;
    // Small c_in (one chunk of at most 32 channels): one k-step or two per tap
    // would cost the MMA issuer a barrier wait per one or two MMAs, so a stage
    // holds three consecutive taps (same K order as one tap per stage).
    // (The upsampler's four taps per phase: two or four per stage.)
    pl.itb = 1;
    if (s.k == 3 && !s.sc_in && !s.up_t && pl.kc_main == 1 && pl.nsub * sw <= 32) {
        for (int itb : {s.up2d ? 4 : 3, s.up2d ? 2 : 3}) {
            const uint32_t sbt = (uint32_t)itb * pl.nsub * (kBlockM + b_rows) * sw * 2u;
            if (pl.itb == 1 &&
                (uint32_t)need_stages * ((sbt + 1023u) & ~1023u) + reserve <=
                    (uint32_t)kSmemBudget) {
                pl.itb = itb;
                pl.nsub *= itb;
            }
        }
    }
    pl.a_sub = (uint32_t)kBlockM * sw * 2;
    pl.b_sub = b_rows * sw * 2;
    pl.a_bytes = pl.a_sub * pl.nsub;
    pl.stage_bytes = (pl.a_bytes + pl.b_sub * pl.nsub + 1023u) & ~1023u;
    pl.stages = (int)((kSmemBudget - reserve) / pl.stage_bytes);
    if (pl.stages > 8) pl.stages = 8;
    if (pl.stages < 2) return false;
    uint32_t off = pl.stage_bytes * pl.stages;
    pl.off_stage = off;
    if (pl.staged) off += stage_tile;
    pl.off_bars = off;
    pl.off_misc = pl.off_bars + 8u * (2 * pl.stages + 14);
    pl.off_vec = (pl.off_misc + 24u + 15u) & ~15u;  // TMEM slot, abort flag, producer state
    pl.smem_bytes = 1024u + pl.off_vec + 2u * 4u * s.c_out + 4u * 4u * kBlockM +
                    (pl.staged ? 0u : (uint32_t)kEpiWarps * pl.stg_warp);
    // One CTA per SM: the TMEM allocation assumes it has the SM to itself.
    if (pl.smem_bytes < 120u * 1024u) pl.smem_bytes = 120u * 1024u;
    return pl.smem_bytes <= (uint32_t)kSmemBudget;
}

// Per-device, per-kernel launch facts: the dynamic shared-memory opt-in and
// how many CTA-pair clusters can be resident at once.
struct KernelFacts {
    int dev;
    ConvKernelFn fn;
    int max_pairs;
};
std::mutex g_facts_mu;
KernelFacts g_facts[256];
int g_nfacts = 0;

cudaError_t kernel_facts(ConvKernelFn fn, bool pair, int &max_pairs) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(g_facts_mu);
    for (int i = 0; i < g_nfacts; ++i)
        if (g_facts[i].dev == dev && g_facts[i].fn == fn) {
            max_pairs = g_facts[i].max_pairs;
            return cudaSuccess;
        }
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBudget);
    if (e != cudaSuccess) return e;
    int n = 0;
    if (pair) {
        // Every launch uses >= 120 KB of shared memory, so one CTA per SM:
        // the resident-cluster count does not depend on the exact size.
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.gridDim = dim3(2, 1, 1);
        cfg.blockDim = dim3(kThreads, 1, 1);
        cfg.dynamicSmemBytes = (size_t)kSmemBudget;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaOccupancyMaxActiveClusters(&n, fn, &cfg);
        if (e != cudaSuccess) return e;
    }
    if (g_nfacts < 256) g_facts[g_nfacts++] = KernelFacts{dev, fn, n};
    max_pairs = n;
    return cudaSuccess;
}

// Halo tiles for a frame whose 16 x 8 patches do not tile it exactly: in a
// call of one frame per batch element (frame-by-frame decode, where they
// measured 7-8 % faster than im2col: 0.203 against 0.218 ms per 720p call)
// when the patches waste at most about a ninth of the MMA rows, and only
// when the halo plan and the im2col plan cut the channels into the same
// chunks -- im2col walks each temporal tap chunk by chunk, the spatial taps
// within a chunk, as the halo tiles do, so both tilings then add the same
// products in the same order and a clip run whole (im2col) and frame by frame
// (halo) give the same bits.
bool pick_ragged_halo(const ConvSpec &s, Plan &pl, int pair) {
    if (s.k != 3 || s.up2d || s.up_t || s.T != 1) return false;
    if (g_variant[kVarHalo].load(std::memory_order_relaxed) != -1) return false;
    if (s.H % 16 == 0 && s.W % 8 == 0) return false;  // (exact patches: halo_choice)
    const int64_t ph = (s.H + 15) / 16, pw = (s.W + 7) / 8;
    if (8 * ph * 16 * pw * 8 > 9 * (int64_t)s.H * s.W) return false;
    Plan hp, ip;
    if (!make_plan(s, hp, pair, 1, 0) || !make_plan(s, ip, pair, 0, 0)) return false;
    if (ip.itb != 1 || hp.nsub * hp.sw != ip.nsub * ip.sw || hp.kc_main != ip.kc_main ||
        hp.kc_short != ip.kc_short)
        return false;
    pl = hp;
    return true;
}

// The first plan that fits: the preferred CTA grouping with wide halo tiles,
// then plain halo tiles, then the same on single CTAs, then im2col.
bool pick_plan(const ConvSpec &s, Plan &pl, int pair) {
    if (pick_ragged_halo(s, pl, pair)) return true;
    const int hc = s.up_t ? 0 : halo_choice(s), wc = wide_choice(s, hc);  // (im2col: centre taps)
    return (wc && make_plan(s, pl, pair, hc, 1)) || make_plan(s, pl, pair, hc, 0) ||
           (wc && make_plan(s, pl, 1, hc, 1)) || make_plan(s, pl, 1, hc, 0) ||
           make_plan(s, pl, 1, 0, 0);
}

}  // namespace

int conv3d_supported(const ConvSpec &s) {
    if (s.k != 1 && s.k != 3) return -1;
    if (s.c_in < 16 || s.c_in % 16 || s.c_out < 1 || (s.c_out >= 16 && s.c_out % 16) ||
        s.c_out > 512)
        return -1;
    if (s.c_in > 4096) return -1;
    if (s.sc_in && (s.c_sc < 16 || s.c_sc % 16 || s.c_sc > 4096)) return -1;
    if (conv3d_narrow_supported(s) == 0) return 0;
    Plan pl;
    return pick_plan(s, pl, pair_choice()) ? 0 : -1;
}

bool conv3d_fuses_norm(const ConvSpec &s) {
    if (!s.norm_in || conv3d_narrow_supported(s) == 0) return false;
    Plan pl;
    return pick_plan(s, pl, pair_choice()) && pl.fuse;
}

void set_kernel_variant(int pair, int halo, int wide, int narrow, int fuse) {
    const int v[kNumVar] = {pair, halo, wide, narrow, fuse};
    for (int i = 0; i < kNumVar; ++i)
        g_variant[i].store(v[i] == 0 || v[i] == 1 || (i == kVarPair && v[i] == 2) ? v[i] : -1,
                           std::memory_order_relaxed);
}

int narrow_variant() { return g_variant[kVarNarrow].load(std::memory_order_relaxed); }

bool encode_tiled_bf16(CUtensorMap *m, int rank, const void *base, const cuuint64_t *dims,
                       const cuuint64_t *strides, const cuuint32_t *box, int swizzle_bytes) {
    if (!load_encoders()) return false;
    const CUtensorMapSwizzle sz = swizzle_bytes == 128   ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                  : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                        : CU_TENSOR_MAP_SWIZZLE_NONE;
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return g_encode_tiled(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank,
                          const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_conv3d(const ConvSpec &s, const LaunchCtx &ctx) {
    if (conv3d_narrow_supported(s) == 0) return launch_conv3d_narrow(s, ctx);
    Plan pl;
    if (!pick_plan(s, pl, pair_choice())) return cudaErrorInvalidValue;
    if (s.norm_in && !pl.fuse) return cudaErrorInvalidValue;  // (callers ask conv3d_fuses_norm)
    if (!load_encoders()) return cudaErrorInvalidValue;
    auto pick = [&](int pair) {
        if (s.up2d || s.up_t) return conv_kernel_up(pair, pl.sw / 16, pl.nsub, pl.n_pieces);
        if (pl.fuse) return conv_kernel_fuse(pair, pl.sw / 16, pl.nsub, pl.n_pieces);
        return conv_kernel_plain(pair, pl.sw / 16, pl.nsub, pl.n_pieces);
    };
    ConvKernelFn fn = pick(pl.pair);
    int max_pairs = 0;
    cudaError_t fe = kernel_facts(fn, pl.pair == 2, max_pairs);
    if (fe != cudaSuccess) return fe;
    if (pl.pair == 2 && max_pairs < 1) {
        if (!pick_plan(s, pl, 1) || (s.norm_in && !pl.fuse)) return cudaErrorInvalidValue;
        fn = pick(1);
        fe = kernel_facts(fn, false, max_pairs);
        if (fe != cudaSuccess) return fe;
    }

    const int HW = s.H * s.W;
    const int frames = s.B * s.T;
    const int64_t M = (int64_t)frames * HW;
    CUtensorMap mA, mC, mB, mSA, mSB, mY, mR;
    memset(&mY, 0, sizeof(mY));
    memset(&mR, 0, sizeof(mR));
    memset(&mC, 0, sizeof(mC));
    memset(&mSA, 0, sizeof(mSA));
    memset(&mSB, 0, sizeof(mSB));
    bool ok = true;
    if (pl.halo && pl.halo_rows) {
        ok = ok && encode_halo(&mA, s.in, s.c_in, s.W, s.H, frames, pl.sw, pl.halo_w);
        if (s.cache)
            ok = ok && encode_halo(&mC, s.cache, s.c_in, s.W, s.H, s.B * 2, pl.sw, pl.halo_w);
    } else if (pl.halo) {
        const int chunk = pl.nsub * pl.sw;
        ok = ok && encode_halo_planes(&mA, s.in, s.c_in, s.W, s.H, frames, chunk, pl.halo_w);
        if (s.cache)
            ok = ok && encode_halo_planes(&mC, s.cache, s.c_in, s.W, s.H, s.B * 2, chunk,
                                          pl.halo_w);
    } else if (s.k == 3) {
        ok = ok && encode_im2col(&mA, s.in, s.c_in, s.W, s.H, frames, pl.sw);
        if (s.cache) ok = ok && encode_im2col(&mC, s.cache, s.c_in, s.W, s.H, s.B * 2, pl.sw);
    } else {
        ok = ok && encode_2d(&mA, s.in, (uint64_t)s.c_in, (uint64_t)M, pl.sw, kBlockM, pl.sw);
    }
    if (pl.halo && pl.tb > 1)
        ok = ok && encode_weight_taps(&mB, s.w, (uint64_t)(s.up2d ? 4 : 27) * s.c_in, s.c_in,
                                      s.c_out, pl.pair, pl.sw, pl.nsub, pl.tb, pl.npad,
                                      s.up2d ? 4 : 1);
    else
        ok = ok && encode_weights(&mB, s.w,
                                  (uint64_t)(s.up2d ? 4 : s.up_t ? 2 : s.k * s.k * s.k) * s.c_in,
                                  s.c_out, pl.pair, pl.n_pieces, pl.sw, pl.halo ? pl.nsub : 0,
                                  pl.npad, s.up2d ? 4 : s.up_t ? 2 : 1);
    if (s.sc_in) {
        if (pl.halo)
            ok = ok && encode_patch(&mSA, s.sc_in, s.c_sc, s.W, s.H, frames, pl.sw, pl.sw);
        else
            ok = ok && encode_2d(&mSA, s.sc_in, (uint64_t)s.c_sc, (uint64_t)M, pl.sw, kBlockM,
                                 pl.sw);
        ok = ok && encode_weights(&mSB, s.sc_w, (uint64_t)s.c_sc, s.c_out, pl.pair, pl.n_pieces,
                                  pl.sw, pl.halo ? pl.nsub : 0);
    }
    if (pl.staged) {
        if (pl.halo) {
            ok = ok && encode_patch(&mY, s.out, s.c_out, s.W, s.H, frames, 64, 64);
            if (s.epi == kEpiResidual)
                ok = ok && encode_patch(&mR, s.resid, s.c_out, s.W, s.H, frames, 64, 64);
        } else {
            // (the temporal upsampler writes 2T frames: frame 2t + phase)
            ok = ok && encode_frames(&mY, s.out, s.c_out, HW, frames * (s.up_t ? 2 : 1));
            if (s.epi == kEpiResidual) ok = ok && encode_frames(&mR, s.resid, s.c_out, HW, frames);
        }
    }
    if (s.up2d && pl.halo)
        ok = ok && encode_phase_view(&mY, s.out, s.c_out, s.W, s.H, frames,
                                     up_box_channels(s.c_out));
    if (!ok) return cudaErrorInvalidValue;

    ConvArgs a;
    memset(&a, 0, sizeof(a));
    a.T = s.T;
    a.H = s.H;
    a.W = s.W;
    a.HW = HW;
    a.c_in = s.c_in;
    a.c_out = s.c_out;
    a.taps = s.k == 3 ? 27 : 1;
    a.has_cache = s.cache != nullptr && s.k == 3;
    a.sw = pl.sw;
    a.nsub = pl.nsub;
    a.itb = pl.halo ? 1 : pl.itb;
    a.kc_main = pl.kc_main;
    a.kc_short = pl.kc_short;
    a.n_pieces = pl.n_pieces;
    a.piece_n = pl.piece_n;
    a.layout = pl.sw == 64 ? kLayoutSw128 : (pl.sw == 32 ? kLayoutSw64 : kLayoutSw32);
    a.halo = pl.halo;
    a.nq = pl.halo ? pl.nq : 1;
    a.halo_w = pl.halo_w;
    a.halo_rows = pl.halo_rows;
    a.sub_stride = pl.sub_stride;
    a.plane_bytes = (uint32_t)(kHaloH * pl.halo_w * 16);
    a.patches_w = (s.W + 8 * a.nq - 1) / (8 * a.nq);
    a.tb = pl.tb;
    a.narrow = pl.narrow;
    a.bc_row = pl.narrow ? pl.npad / pl.pair : 0;
    a.bc_rank = pl.narrow ? 0 : 1;
    a.off_a = pl.off_a;
    a.a_stride = pl.a_stride;
    a.na = pl.na;
    a.up_tma = s.up2d && pl.halo;
    a.stg_warp = pl.stg_warp;
    a.up_box = up_box_channels(s.c_out);
    a.a_tx = pl.a_tx;
    a.tiles_per_frame = pl.halo ? ((s.H + 15) / 16) * a.patches_w : (HW + kBlockM - 1) / kBlockM;
    a.num_tiles = a.tiles_per_frame * frames;
    a.frames = frames;
    a.nphase = s.up2d ? 4 : s.up_t ? 2 : 1;
    a.tile_units = (a.num_tiles + pl.pair - 1) / pl.pair;
    a.wtap0 = s.up2d ? 18 : s.up_t ? 9 : 0;  // (temporal upsampler: taps kt = 1, 2)
    a.sp_taps = s.up2d ? 4 : s.up_t ? 1 : 9;
    a.sp_w = s.up2d ? 2 : s.up_t ? 1 : 3;
    a.up_t = s.up_t;
    a.segs_per_kt = a.sp_taps / (pl.halo ? 1 : pl.itb);  // (as a.itb)
    // which B box coordinate a phase moves: the rank dimension of the 3-tap
    // map (its pieces are one), else the piece dimension
    const bool taps_map = pl.halo && pl.tb > 1;
    a.ph_c2 = s.up2d && taps_map ? pl.pair : 0;
    a.ph_c3 = (s.up2d || s.up_t) && !taps_map ? pl.n_pieces : 0;
    a.stages = pl.stages;
    a.a_sub_bytes = pl.a_sub;
    a.b_sub_bytes = pl.b_sub;
    a.a_bytes = pl.a_bytes;
    a.stage_bytes = pl.stage_bytes;
    a.stage_tx = pl.halo ? pl.b_sub * pl.nsub * (uint32_t)pl.tb : (pl.a_sub + pl.b_sub) * pl.nsub;
    a.off_bars = pl.off_bars;
    a.off_misc = pl.off_misc;
    a.off_vec = pl.off_vec;
    a.staged = pl.staged;
    a.off_stage = pl.off_stage;
    a.acc_cols = pl.acc_cols;
    a.acc_stride = pl.acc_stride;
    a.nacc = pl.nacc;
    a.tmem_cols = pl.tmem_cols;
    a.epi = s.epi;
    a.eps = s.eps;
    a.sqrt_c = sqrtf((float)s.c_out);
    a.bias = s.bias;
    a.bias2 = s.bias2;
    a.gamma = s.gamma;
    a.resid = static_cast<const __nv_bfloat16 *>(s.resid);
    a.out = static_cast<__nv_bfloat16 *>(s.out);
    a.err = ctx.err;
    a.wait_ns = ctx.wait_ns;
    a.fuse = pl.fuse;
    a.epi_warps = pl.fuse ? 4 : kEpiWarps;
    // Two MMA issuers wherever the accumulators split in two: the sub-tiles
    // of a wide halo tile, or two N pieces.
    a.issuers = (a.nq == 2 || pl.n_pieces == 2) ? 2 : 1;
    // Two producers where a fill carries few MMAs: im2col stages, and halo
    // plans with one-tap weight stages (not with the fused input norm, whose
    // transform warps pace the halo stages).
    a.producers = !pl.halo || (pl.tb == 1 && !pl.fuse) ? 2 : 1;
    if (pl.fuse) {
        a.nl_L = nact_lanes(s.c_in);
        a.nl_vpt = (s.c_in / 8) / a.nl_L;
        a.sqrt_c_in = sqrtf((float)s.c_in);
        a.gamma_in = s.gamma_in;
        a.x_in = static_cast<const __nv_bfloat16 *>(s.in);
        a.cache_in = static_cast<const __nv_bfloat16 *>(s.cache);
    }

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    // programmatic dependent launch: the prologue (barriers, TMEM, descriptor
    // prefetch) overlaps the previous kernel's tail; the kernel waits for it
    // before its first global read
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    if (pl.pair == 1) {
        const int units = a.tile_units * a.nphase;
        const int grid = units < ctx.num_sms ? units : ctx.num_sms;
        cfg.gridDim = dim3((unsigned)grid, 1, 1);
        cfg.numAttrs = 1;
    } else {
        const int units = a.tile_units * a.nphase;
        const int pairs = units < max_pairs ? units : max_pairs;
        cfg.gridDim = dim3((unsigned)(2 * pairs), 1, 1);
        cfg.numAttrs = 2;
    }
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = pl.smem_bytes;
    cfg.stream = ctx.stream;
    return cudaLaunchKernelEx(&cfg, fn, mA, mC, mB, mSA, mSB, mY, mR, a);
}

}  // namespace wanvae
