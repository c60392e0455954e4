#pragma once
// conv3d_tcgen05.cuh -- device side of the CausalConv3d implicit GEMM (see
// conv3d_tcgen05.cu for the host side).  Included by the translation units
// that instantiate the kernel (conv3d_kernels_*.cu, compiled in parallel) and
// by the host code for the argument struct and the tiling constants.
//
// The operation ("Closing the gap: Wan 2.2 14B VAE decoder", sections 2 and 6;
// "Sharding of WAN 2.2 VAE", Conv3D strategy table):
//     out[b,t,y,x,o] = bias[o] + sum_{kt,kh,kw,c} w[o,kt,kh,kw,c]
//                                  * in[b, t+kt-2, y+kh-1, x+kw-1, c]
// with zeros (or the feat_cache frames) for t+kt-2 < 0 and zeros outside H, W.
// GEMM view: M = B*T*H*W output voxels, N = c_out, K = 27 * c_in; the K loop
// walks the three temporal taps, each in chunks of channels, and within a
// chunk the nine spatial taps (the same order for im2col and halo tiles).
//
// Tiling.  A CTA tile is 128 voxels of ONE frame (b, t): 128 consecutive ones
// (im2col; the last tile of a frame is ragged) or a 16 x 8 patch (halo) -- by all
// c_out channels (the accumulator is 128 TMEM lanes x c_out fp32 columns, so
// an epilogue thread owns every channel of one voxel, which is what lets the
// next RMS_norm run inside the epilogue).  Because a tile never spans frames,
// every tap of a tile reads a single source frame: the conv input, the
// feat_cache, or nothing (a zero causal-pad tap is skipped).
//
// A operand: one TMA im2col load per (tap, channel chunk) over the NHWC view
// [frames][H][W][C] of the input.  The map's bounding box is the H x W frame
// shrunk by the conv's one-element pad on each side; walking 128 pixels from
// the tile's first voxel and reading each at (pixel + (kw, kh)) gives exactly
// the tap-shifted rows, with out-of-frame reads filled with zeros by TMA (the
// spatial zero pad).  B operand: the weights as a K-major [c_out][27*c_in]
// matrix, one tiled TMA box per (chunk, N-piece).  Both land in smem with the
// hardware swizzle that the UMMA descriptors name.
//
// Warp roles (384 threads, one persistent CTA per SM): warp 0 = TMA producer,
// warp 1 = MMA issuer (and TMEM owner), warps 2-9 = epilogue, two per TMEM
// lane quarter, warp 10 = second MMA issuer where the accumulators split
// between two, warp 11 = second TMA producer where fills carry few MMAs
// (im2col tiles, one-tap halo stages).  An mbarrier ring of `stages` smem
// buffers links producers and MMA; up to two accumulators in TMEM let the
// epilogue of tile i overlap the MMAs of tile i+1 when 2 * c_out fits in
// TMEM's 512 columns.  Every wait is bounded (ptx.cuh).
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <string.h>

#include <type_traits>

#include "kernels.h"
#include "norm_act.cuh"
#include "ptx.cuh"

namespace wanvae {
namespace conv {

constexpr int kBlockM = 128;
constexpr int kEpiWarps = 8;  // two warps per TMEM lane quarter, each half the columns
// The second MMA issuer (after the producer, the first issuer and the
// epilogue warps).  Every shared-memory access by an issuing thread -- a
// barrier wait, even a plain load -- returns only after the operand reads of
// the MMAs it already issued, and the tensor core then runs dry until the
// thread issues again.  Two issuers that own separate accumulators (the two
// sub-tiles of a wide tile, or the two N pieces of a wide layer) each wait
// for every stage themselves, so one keeps the tensor core fed while the
// other waits.
constexpr int kIssuer2Warp = 2 + kEpiWarps;
// The second TMA producer of im2col tiles, for the same reason: each fill
// costs its producer a shared-memory round trip behind the tensor core's
// operand reads (the empty-slot wait), longer than the few MMAs of a
// one-tap stage, so two producers take alternate fills of the ring.
constexpr int kProducer2Warp = kIssuer2Warp + 1;
constexpr int kThreads = 32 * (kProducer2Warp + 1);
constexpr uint32_t kStageBytesPerWarp = 32 * 64;  // 32 rows x 32 bf16 channels
constexpr int kSmemBudget = 227 * 1024;
constexpr int kMaxItb = 4;  // im2col: most taps per stage (the upsampler's 2 x 2)
constexpr int kMaxNormVpt = 4;  // fused input norm: most 16-byte vectors a lane holds
constexpr uint64_t kDrainNs = 200ull * 1000 * 1000;  // cleanup waits after an abort


struct ConvArgs {
    int T, H, W, HW;
    int c_in, c_out;
    int taps;            // 27 or 1
    int has_cache;
    int sw;              // channels per swizzled sub-tile (64, 32 or 16)
    int nsub;            // sub-tiles per pipeline stage (im2col: itb taps x channel sub-tiles)
    int itb;             // im2col: taps per stage (3 for small c_in, else 1)
    int kc_main;         // stages per tap
    int kc_short;        // stages of the shortcut segment (0 = none)
    int n_pieces, piece_n;
    uint32_t layout;     // UMMA swizzle mode matching sw
    int tiles_per_frame, num_tiles;
    int frames;          // B * T
    int nphase;          // 4: upsampler conv (units = tile units x sub-pixel phases), else 1
    int tile_units;      // units per phase: ceil(num_tiles / pair)
    int wtap0;           // 9 x the temporal tap the weights start at (18: upsampler, kt = 2 only)
    int sp_taps, sp_w;   // spatial taps per temporal tap and per tap row: 9, 3 (upsampler: 4, 2)
    int segs_per_kt;     // im2col: stages per temporal tap and channel chunk, sp_taps / itb
    int na;              // halo mode: buffers in the A (halo) ring, 2 to 4
    int up_tma;          // upsampler on halo tiles: TMA stores through the phase view of y
    int up_box;          // channels per phase-view store box (48, else 16)
    uint32_t stg_warp;   // bytes of each epilogue warp's staging buffer
    int up_t;            // temporal upsampler: frame phases, taps t-1 and t at the centre pixel
    int fuse;            // input norm fused: warps 2 + epi_warps .. 9 build every halo
    int epi_warps;       // epilogue warps: 8 (two per TMEM lane quarter), 4 when fused
    int issuers;         // MMA issuers: 2 = one per sub-tile (nq = 2) or per N piece, else 1
    int producers;       // TMA producers: 2 (alternate fills) for im2col tiles, 1 for halo tiles
    int nl_L, nl_vpt;    // fused norm: lanes per pixel, 16-byte vectors per lane
    float sqrt_c_in;     // fused norm: sqrt(c_in)
    const float *gamma_in;
    const __nv_bfloat16 *x_in, *cache_in;  // fused: raw input x and the cache (normalised)
    int ph_c2, ph_c3;    // upsampler: B box coordinates 2 and 3 advance by phase x these
    int stages;
    uint32_t a_sub_bytes, b_sub_bytes, a_bytes, stage_bytes, stage_tx;
    uint32_t off_bars, off_misc, off_vec;
    int acc_cols;        // TMEM columns of one 128-row accumulator
    int acc_stride;      // columns of one accumulator buffer (nq accumulators)
    int nacc, tmem_cols;
    int staged;          // epilogue through a whole-tile smem buffer + TMA stores
    uint32_t off_stage;  // 1024-aligned offset of that buffer
    int halo;            // 16x8 patch tiles, one halo load per (kt, chunk) for 9 taps
    int patches_w;       // patches per frame row (halo mode)
    int nq;              // 128-row sub-tiles per CTA tile (halo mode: 1, or 2 for 16x16 patches)
    int halo_w;          // halo width in pixels: 8 * nq + 2
    int halo_rows;         // halo as swizzled pixel rows (sw = 64, 32) instead of 8-channel planes
    uint32_t sub_stride;   // rows: bytes between the halo's sw-channel regions (1024-aligned)
    uint32_t plane_bytes;  // planes: one 8-channel plane of the halo, 18 * halo_w * 16
    int tb;              // spatial taps per weight stage (halo mode: 1, 3)
    int narrow;          // c_out < 16: N padded to 16 per CTA, rows past c_out read as zeros
    int bc_row, bc_rank; // B box coordinates of this CTA's rows: (rank * bc_row, rank * bc_rank)
    uint32_t off_a, a_stride, a_tx;  // halo ring: 2 buffers, bytes per CTA per load
    int epi;
    float eps, sqrt_c;
    const float *bias, *bias2, *gamma;
    const __nv_bfloat16 *resid;
    __nv_bfloat16 *out;
    unsigned *err;
    uint64_t wait_ns;
};

struct TileInfo {
    int frame, pos, n, t, h0, w0, row0;
    bool dummy;  // a pair's second slot past the last tile: zero A, nothing stored
};

// Halo mode orders tiles patch-major, frame-minor: the tiles of the three
// output frames that read one input frame (its temporal taps) run side by
// side, so a frame is fetched from DRAM about once although it does not fit
// L2 three times over.  im2col mode orders them frame-major.
__device__ __forceinline__ int tile_frame(int tile, const ConvArgs &p) {
    return p.halo ? tile % p.frames : tile / p.tiles_per_frame;
}

__device__ __forceinline__ TileInfo tile_info(int tile, const ConvArgs &p) {
    TileInfo ti;
    ti.dummy = tile >= p.num_tiles;
    if (ti.dummy) tile = 0;
    ti.frame = tile_frame(tile, p);
    ti.pos = (p.halo ? tile / p.frames : tile - ti.frame * p.tiles_per_frame) * kBlockM;
    ti.n = ti.frame / p.T;
    ti.t = ti.frame - ti.n * p.T;
    if (p.halo) {
        // 16 x 8nq (H x W) patch of nq sub-tiles: row m of sub-tile s is
        // pixel (h0 + m / 8, w0 + 8 s + m % 8).
        const int pt = ti.pos / kBlockM;
        const int ph = pt / p.patches_w;
        ti.h0 = ph * 16;
        ti.w0 = (pt - ph * p.patches_w) * 8 * p.nq;
        ti.row0 = ti.frame * p.HW + ti.h0 * p.W + ti.w0;  // first pixel's voxel index
    } else {
        ti.h0 = ti.pos / p.W;
        ti.w0 = ti.pos - ti.h0 * p.W;
        ti.row0 = ti.frame * p.HW + ti.pos;
    }
    return ti;
}

// Halo mode: every smem halo is 18 x halo_w pixels (a 16 x 8nq patch grown
// by the 3x3 window; halo_w = 10 or 18), stored per sw-channel chunk as one
// swizzled row per pixel, row-major over the halo.  The MMA A operand of tap
// (kh, kw) for sub-tile s is the window starting at pixel (kh, kw + 8s):
// consecutive rows inside a patch row, 8-row groups one halo row (halo_w
// rows) apart -- a swizzled K-major operand whose start and group stride are
// not atom-aligned, which the tensor core reads correctly because it applies
// the swizzle by absolute address.
constexpr uint32_t kHaloH = 18;


// First temporal tap of a work unit (one tile, or the two tiles of a CTA
// pair, which share every B stage and so run the same taps): taps reading
// t+kt-2 < 0 are zero (skipped) unless a feat_cache supplies those frames.
// A pair member whose own frame needs a skipped-for-it tap loads zeros.
// Tile unit and sub-pixel phase of a work unit.  Upsampler: phase-minor, so
// the four phases of a tile run side by side on neighbouring CTAs and read
// its input from L2 rather than each from HBM.
__device__ __forceinline__ int unit_tile(int u, const ConvArgs &p) {
    return p.nphase > 1 ? u / p.nphase : u;
}
__device__ __forceinline__ int unit_phase(int u, const ConvArgs &p) {
    return p.nphase > 1 ? u % p.nphase : 0;
}
// Upsampler phase (a, b) = (ph >> 1, ph & 1): its sub-pixel kernel is the 2 x 2
// block of low-res taps whose corner is (a, b) in the 3 x 3 window; a plain
// conv's spatial taps start at (0, 0).
struct TapBase {
    int kh, kw;
};
__device__ __forceinline__ TapBase unit_tap_base(int u, const ConvArgs &p) {
    const int ph = unit_phase(u, p);
    return TapBase{ph >> 1, ph & 1};
}

template <int kPair>
__device__ __forceinline__ int unit_first_kt(int unit, const ConvArgs &p) {
    if (p.wtap0) return p.wtap0 / 9;  // upsampler: the current frame's taps only
    if (p.taps != 27 || p.has_cache) return 0;
    int kt0 = 3;
#pragma unroll
    for (int r = 0; r < kPair; ++r) {
        const int tile = unit * kPair + r;
        if (tile >= p.num_tiles) continue;
        const int t = tile_frame(tile, p) % p.T;
        const int k = t >= 2 ? 0 : 2 - t;
        kt0 = k < kt0 ? k : kt0;
    }
    return kt0;
}

template <int kPair>
__device__ __forceinline__ int unit_stages(int unit, const ConvArgs &p) {
    const int main_taps =
        p.taps == 27 ? (3 - unit_first_kt<kPair>(unit, p)) * p.segs_per_kt : 1;
    return main_taps * p.kc_main + p.kc_short;
}

struct Bars {
    uint32_t base;
    int stages;
    __device__ uint32_t full(int s) const { return base + 8u * s; }
    __device__ uint32_t empty(int s) const { return base + 8u * (stages + s); }
    __device__ uint32_t accf(int a) const { return base + 8u * (2 * stages + a); }
    __device__ uint32_t acce(int a) const { return base + 8u * (2 * stages + 2 + a); }
    __device__ uint32_t drain() const { return base + 8u * (2 * stages + 4); }
    __device__ uint32_t resf() const { return base + 8u * (2 * stages + 5); }
    __device__ uint32_t emptya(int i) const { return base + 8u * (2 * stages + 6 + i); }
    // fused norm in a CTA pair: the peer's halo in A buffer i is written
    __device__ uint32_t peer(int i) const { return base + 8u * (2 * stages + 10 + i); }
};

// The MMA issuer's view of the `full` ring.  Every barrier access by the
// issuing thread is slow while the tensor core streams its operands out of
// shared memory (the access queues behind them) and the few MMAs already
// queued run dry meanwhile, so the issuers wait once per stage and make the
// stages as large as shared memory allows.
template <bool kCluster>
struct FullRing {
    int stage = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ bool acquire(const Bars &bars, const WaitCtl &wc) {
        return mbar_wait<kCluster>(bars.full(stage), phase, wc);
    }
    __device__ __forceinline__ void advance(const Bars &bars) {
        if (++stage == bars.stages) {
            stage = 0;
            phase ^= 1u;
        }
    }
};

// A producer's exit: publish its last issued fill (prod[part]) and that it
// has stopped (prod[2 + part]), and after an abort (rank 0) let the newest
// fill of every stage it issued land before the CTA and its shared memory go
// away.  A fill is the newest of its stage unless a fill `stages` (or a
// multiple) later was issued, by either producer (fill f is producer f mod
// p.producers's); waiting on an older phase would never return.
template <int kPair>
__device__ void producer_finish(const ConvArgs &p, const Bars &bars, const WaitCtl &wc,
                                uint32_t rank, int part, int last_mine, volatile int *prod,
                                bool ok) {
    const int np = p.producers;
    prod[part] = last_mine;
    __threadfence_block();
    prod[2 + part] = 1;
    if ((ok && !*wc.abort) || rank != 0) return;
    volatile int no_abort = 0;
    const WaitCtl dc{kDrainNs, wc.err, &no_abort, kDevErrTimeout | kDevErrDrain};
    if (np == 2) {  // the other producer's last fill, once it has stopped
        const uint64_t t0 = globaltimer_ns();
        while (prod[2 + (1 - part)] == 0) {
            if (globaltimer_ns() - t0 >= kDrainNs) {
                atomicOr(wc.err, kDevErrTimeout | kDevErrDrain);
                break;
            }
        }
    }
    const int last0 = prod[0], last1 = np == 2 ? prod[1] : -1;
    const int newest = last0 > last1 ? last0 : last1;
    for (int f = last_mine; f >= 0 && f > last_mine - np * p.stages; f -= np) {
        bool superseded = false;
        for (int g = f + p.stages; g <= newest; g += p.stages)
            if (g <= ((g & 1) && np == 2 ? last1 : last0)) {
                superseded = true;
                break;
            }
        if (!superseded)
            mbar_wait<kPair == 2>(bars.full(f % p.stages), (uint32_t)(f / p.stages) & 1u, dc);
    }
}

// TMA producer (one thread per CTA).  In a CTA pair each CTA loads its own
// 128-row A tile and its half of every B piece; all loads complete on the
// leader CTA's `full` barrier, which the leader arms for both CTAs' bytes.
//
// With two producers (p.producers == 2) both walk the whole fill sequence and
// producer `part` issues the fills whose index is `part` modulo 2.  Each
// publishes the index of its last issued fill in prod[part] and then sets
// prod[2 + part]; after an abort both are needed to tell which fill is the
// newest of its stage, the one a drain may wait for.  A parity wait cannot
// tell phase m from phase m - 2, so a producer must never wait for fill f
// before fill f - 2 * stages is released: the issuers release fills in order
// and consume every stage, so the producer's own wait for fill f - 2 (which
// needed fill f - 2 - stages released) already implies it when stages >= 2.
template <int kPair, bool kUp>
__device__ void conv_producer(const CUtensorMap *mapA, const CUtensorMap *mapC,
                              const CUtensorMap *mapB, const CUtensorMap *mapSA,
                              const CUtensorMap *mapSB, const ConvArgs &p, uint32_t sbase,
                              const Bars &bars, const WaitCtl &wc, int unit0, int unit_stride,
                              int num_units, uint32_t rank, int part, volatile int *prod) {
    const int frames = p.num_tiles / p.tiles_per_frame;  // B*T
    const int M = frames * p.HW;
    const uint32_t np = (uint32_t)p.producers;
    int stage = 0;
    uint32_t phase = 0, fills = 0;
    int last_mine = -1;
    bool ok = true;
    // One fill with one tap per stage: weight tap wtap (of phase ph, for the
    // temporal upsampler) and the im2col rows of channel chunk kc at spatial
    // offset (kh, kw).
    auto fill_tap = [&](const CUtensorMap *am, int fidx, int wtap, int kh, int kw, int ph, int kc,
                        int w0, int h0) -> bool {
        if (!mbar_wait<kPair == 2>(bars.empty(stage), phase ^ 1u, wc)) return false;
        const uint32_t fb_local = bars.full(stage);
        if (rank == 0) mbar_arrive_expect_tx(fb_local, p.stage_tx * kPair);
        const uint32_t fb = kPair == 2 ? mapa_shared(fb_local, 0) : fb_local;
        const uint32_t sa = sbase + (uint32_t)stage * p.stage_bytes;
        const uint32_t sb = sa + p.a_bytes;
        for (int s2 = 0; s2 < p.nsub; ++s2) {
            const int c0 = (kc * p.nsub + s2) * p.sw;
            const uint32_t da = sa + (uint32_t)s2 * p.a_sub_bytes;
            const uint32_t db = sb + (uint32_t)s2 * p.b_sub_bytes;
            if (kPair == 2) {
                tma_load_im2col_4d_pair(da, am, fb, c0, w0 - 1, h0 - 1, fidx, (uint16_t)kw,
                                        (uint16_t)kh);
                tma_load_4d_pair(db, mapB, fb, wtap * p.c_in + c0, (int)rank * p.bc_row,
                                 (int)rank * p.bc_rank + ph * p.ph_c2, ph * p.ph_c3);
            } else {
                tma_load_im2col_4d(da, am, fb, c0, w0 - 1, h0 - 1, fidx, (uint16_t)kw,
                                   (uint16_t)kh);
                tma_load_4d(db, mapB, fb, wtap * p.c_in + c0, 0, ph * p.ph_c2, ph * p.ph_c3);
            }
        }
        last_mine = (int)fills;
        return true;
    };
    auto advance_fill = [&]() {
        ++fills;
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
        }
    };
    // Plain k = 3 convs with one tap per stage walk each temporal tap chunk by
    // chunk, the nine spatial taps within a chunk: the K order of the halo
    // tiles, so that either tiling gives the same sums (and the same bits).
    // The temporal upsampler walks its two taps (frames t - 1 and t, centre
    // pixel) within each chunk in the same way.
    const bool chunk_major = !kUp && p.taps == 27 && p.itb == 1;
    const bool chunk_major_t = kUp && p.up_t && p.taps == 27 && p.itb == 1;
    for (int u = unit0; ok && u < num_units; u += unit_stride) {
        const TileInfo ti = tile_info(unit_tile(u, p) * kPair + (int)rank, p);
        const int kt0 = unit_first_kt<kPair>(unit_tile(u, p), p);
        if (chunk_major) {
            for (int kt = kt0; ok && kt < 3; ++kt) {
                const int tt = ti.t + kt - 2;
                const CUtensorMap *am = mapA;
                int fidx = frames;  // out of range: zeros
                if (!ti.dummy) {
                    if (tt >= 0) {
                        fidx = ti.n * p.T + tt;
                    } else if (p.has_cache) {
                        am = mapC;
                        fidx = ti.n * 2 + tt + 2;
                    }
                }
                for (int kc = 0; ok && kc < p.kc_main; ++kc)
                    for (int sp = 0; ok && sp < 9; ++sp) {
                        const int tap = kt * 9 + sp;
                        if (fills % np == (uint32_t)part &&
                            !fill_tap(am, fidx, tap, (tap / 3) % 3, tap % 3, 0, kc, ti.w0, ti.h0)) {
                            ok = false;
                            break;
                        }
                        advance_fill();
                    }
            }
            if (!ok || p.kc_short == 0) continue;
        }
        if (chunk_major_t) {
            const CUtensorMap *am[2] = {mapA, mapA};
            int fidx[2] = {frames, frames};  // out of range: zeros
            for (int q = 0; q < 2; ++q) {
                const int tt = ti.t + q - 1;  // kt = 1 + q
                if (!ti.dummy) {
                    if (tt >= 0) {
                        fidx[q] = ti.n * p.T + tt;
                    } else if (p.has_cache) {
                        am[q] = mapC;
                        fidx[q] = ti.n * 2 + tt + 2;
                    }
                }
            }
            const int ph = unit_phase(u, p);
            for (int kc = 0; ok && kc < p.kc_main; ++kc)
                for (int q = 0; ok && q < 2; ++q) {
                    if (fills % np == (uint32_t)part &&
                        !fill_tap(am[q], fidx[q], q, 1, 1, ph, kc, ti.w0, ti.h0)) {
                        ok = false;
                        break;
                    }
                    advance_fill();
                }
            continue;  // (no shortcut segment)
        }
        // A segment is itb consecutive taps (one tap unless c_in is small),
        // each stage of it itb taps x nch channel sub-tiles.  (In chunk-major
        // order only the shortcut segment is left for this loop.)
        const int nseg = chunk_major ? 0 : (p.taps == 27 ? (3 - kt0) * p.segs_per_kt : 1);
        const TapBase tbase = kUp ? unit_tap_base(u, p) : TapBase{0, 0};
        const int segs = nseg + (p.kc_short > 0 ? 1 : 0);
        const int row0 = ti.dummy ? M : ti.row0;
        for (int seg = 0; ok && seg < segs; ++seg) {
            const bool shortcut = seg == nseg;
            const int ntap = shortcut ? 1 : p.itb, nch = shortcut ? p.nsub : p.nsub / p.itb;
            const int nkc = shortcut ? p.kc_short : p.kc_main;
            // The segment's taps, worked out once for all its channel-chunk
            // stages (this thread must keep ahead of the MMAs): weight tap,
            // spatial offset, source frame (out of range -> zeros) and map.
            int wtap[kMaxItb], kh[kMaxItb], kw[kMaxItb], fidx[kMaxItb];
            bool from_cache[kMaxItb];
#pragma unroll
            for (int j = 0; j < kMaxItb; ++j) {
                wtap[j] = 0;
                kh[j] = 1;
                kw[j] = 1;
                fidx[j] = frames;
                from_cache[j] = false;
                if (j < ntap && !shortcut && p.taps == 27) {
                    const int q = seg * p.itb + j;
                    int kt;
                    if (kUp && p.up_t) {  // frames t - 1 and t, centre pixel
                        kt = 1 + (q & 1);
                        wtap[j] = q & 1;
                    } else if (kUp) {  // the phase's 2 x 2 taps, current frame only
                        kt = 2;
                        kh[j] = tbase.kh + ((q >> 1) & 1);
                        kw[j] = tbase.kw + (q & 1);
                        wtap[j] = q & 3;
                    } else {
                        const int tap = kt0 * 9 + q;
                        kt = tap / 9;
                        kh[j] = (tap / 3) % 3;
                        kw[j] = tap % 3;
                        wtap[j] = tap;
                    }
                    const int tt = ti.t + kt - 2;
                    if (!ti.dummy) {
                        if (tt >= 0) {
                            fidx[j] = ti.n * p.T + tt;
                        } else if (p.has_cache) {
                            from_cache[j] = true;
                            fidx[j] = ti.n * 2 + tt + 2;
                        }
                    }
                }
            }
            const int ph = kUp ? unit_phase(u, p) : 0;  // upsampler: its weights
            const CUtensorMap *bm = shortcut ? mapSB : mapB;
            for (int kc = 0; kc < nkc; ++kc) {
                if (fills % np != (uint32_t)part) {  // the other producer's fill
                    ++fills;
                    if (++stage == p.stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    continue;
                }
                if (!mbar_wait<kPair == 2>(bars.empty(stage), phase ^ 1u, wc)) {
                    ok = false;
                    break;
                }
                const uint32_t fb_local = bars.full(stage);
                if (rank == 0) mbar_arrive_expect_tx(fb_local, p.stage_tx * kPair);
                const uint32_t fb = kPair == 2 ? mapa_shared(fb_local, 0) : fb_local;
                const uint32_t sa = sbase + (uint32_t)stage * p.stage_bytes;
                const uint32_t sb = sa + p.a_bytes;
#pragma unroll
                for (int j = 0; j < kMaxItb; ++j) {
                    if (j >= ntap) break;
                    const CUtensorMap *am = from_cache[j] ? mapC : mapA;
                    for (int s = 0; s < nch; ++s) {
                        const int c0 = (kc * nch + s) * p.sw;
                        const int idx = j * nch + s;  // sub-tile of the stage
                        const uint32_t da = sa + (uint32_t)idx * p.a_sub_bytes;
                        if (kPair == 2) {
                            if (shortcut)
                                tma_load_2d_pair(da, mapSA, fb, c0, row0);
                            else if (p.taps == 27)
                                tma_load_im2col_4d_pair(da, am, fb, c0, ti.w0 - 1, ti.h0 - 1,
                                                        fidx[j], (uint16_t)kw[j], (uint16_t)kh[j]);
                            else
                                tma_load_2d_pair(da, mapA, fb, c0, row0);
                        } else {
                            if (shortcut)
                                tma_load_2d(da, mapSA, fb, c0, row0);
                            else if (p.taps == 27)
                                tma_load_im2col_4d(da, am, fb, c0, ti.w0 - 1, ti.h0 - 1, fidx[j],
                                                   (uint16_t)kw[j], (uint16_t)kh[j]);
                            else
                                tma_load_2d(da, mapA, fb, c0, row0);
                        }
                        // This CTA's rows of every N-piece in one box: the weight
                        // map is viewed as [piece][pair rank][half_n rows][K].
                        const uint32_t db = sb + (uint32_t)idx * p.b_sub_bytes;
                        const int bk = shortcut ? c0 : wtap[j] * p.c_in + c0;
                        if (kPair == 2)
                            tma_load_4d_pair(db, bm, fb, bk, (int)rank * p.bc_row,
                                             (int)rank * p.bc_rank + ph * p.ph_c2,
                                             ph * p.ph_c3);
                        else
                            tma_load_4d(db, bm, fb, bk, 0, ph * p.ph_c2, ph * p.ph_c3);
                    }
                }
                last_mine = (int)fills;
                ++fills;
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    }
    producer_finish<kPair>(p, bars, wc, rank, part, last_mine, prod, ok);
}

// 5-D tiled load (x = c0 innermost).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap *m, uint32_t bar,
                                            int c0, int c1, int c2, int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(c4)
        : "memory");
}
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const CUtensorMap *m,
                                                 uint32_t cluster_bar, int c0, int c1, int c2,
                                                 int c3, int c4) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".cta_group::2 [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(m)), "r"(cluster_bar), "r"(c0), "r"(c1), "r"(c2),
        "r"(c3), "r"(c4)
        : "memory");
}

template <int kPair>
__device__ __forceinline__ void load5(uint32_t dst, const CUtensorMap *m, uint32_t bar, int c0,
                                      int c1, int c2, int c3, int c4) {
    if (kPair == 2)
        tma_load_5d_pair(dst, m, bar, c0, c1, c2, c3, c4);
    else
        tma_load_5d(dst, m, bar, c0, c1, c2, c3, c4);
}
template <int kPair>
__device__ __forceinline__ void load4(uint32_t dst, const CUtensorMap *m, uint32_t bar, int c0,
                                      int c1, int c2, int c3) {
    if (kPair == 2)
        tma_load_4d_pair(dst, m, bar, c0, c1, c2, c3);
    else
        tma_load_4d(dst, m, bar, c0, c1, c2, c3);
}

// Halo-mode producer.  Per unit, for each temporal tap kt and channel chunk:
// one halo load into the A ring (2 buffers) and 9 / tb weight stages of tb
// spatial taps each (B ring); the halo completes on the barrier of the first
// of those stages, so the MMA issuer waits once per stage.  Then the shortcut
// segment's chunks (x patch into the A ring + its weights, one stage each).
//
// With two producers (p.producers == 2: one-tap weight stages, whose few MMAs
// leave one producer's per-fill round trip exposed) producer `part` issues the
// fills whose index is `part` modulo 2, the halo load with the first fill of
// its (kt, chunk) group; both walk the whole sequence, stages and halo
// buffers alike (conv_producer has the same scheme).
template <int kPair, bool kUp, bool kFuse>
__device__ void conv_producer_halo(const CUtensorMap *mapA, const CUtensorMap *mapC,
                                   const CUtensorMap *mapB, const CUtensorMap *mapSA,
                                   const CUtensorMap *mapSB, const ConvArgs &p, uint32_t sbase,
                                   const Bars &bars, const WaitCtl &wc, int unit0,
                                   int unit_stride, int num_units, uint32_t rank, int part,
                                   volatile int *prod) {
    const int frames = p.num_tiles / p.tiles_per_frame;
    const int chunk = p.nsub * p.sw;  // channels per halo / per weight sub-stage
    const int groups = p.sp_taps / p.tb;
    const uint32_t np = (uint32_t)p.producers;
    int stage = 0, ia = 0;
    uint32_t phase = 0, pha = 0, fills = 0;
    int last_mine = -1;
    bool ok = true;
    auto mine = [&]() { return fills % np == (uint32_t)part; };
    auto skip_stage = [&]() {  // the other producer's fill
        ++fills;
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
        }
    };
    auto skip_abuf = [&]() {
        if (++ia == p.na) {
            ia = 0;
            pha ^= 1u;
        }
    };
    // Next B stage, armed for `tx` bytes per CTA (both CTAs' loads complete
    // on the leader's barrier).  With the input norm fused a stage completes
    // on two arrivals: a halo's first stage gets its second from the
    // transform warps once the pair's halos are written, the others get both
    // from here.
    auto next_stage = [&](uint32_t tx, bool second, uint32_t &dst, uint32_t &fb) -> bool {
        if (!mbar_wait<kPair == 2>(bars.empty(stage), phase ^ 1u, wc)) return false;
        const uint32_t fl = bars.full(stage);
        if (rank == 0) {
            mbar_arrive_expect_tx(fl, tx * kPair);
            if (second) mbar_arrive(fl);
        }
        fb = kPair == 2 ? mapa_shared(fl, 0) : fl;
        dst = sbase + p.a_bytes + (uint32_t)stage * p.stage_bytes;
        last_mine = (int)fills;
        ++fills;
        if (++stage == p.stages) {
            stage = 0;
            phase ^= 1u;
        }
        return true;
    };
    auto next_abuf = [&](uint32_t &dst) -> bool {
        if (!mbar_wait<kPair == 2>(bars.emptya(ia), pha ^ 1u, wc)) return false;
        dst = sbase + p.off_a + (uint32_t)ia * p.a_stride;
        if (++ia == p.na) {
            ia = 0;
            pha ^= 1u;
        }
        return true;
    };
    for (int u = unit0; ok && u < num_units; u += unit_stride) {
        const TileInfo ti = tile_info(unit_tile(u, p) * kPair + (int)rank, p);
        const int kt0 = unit_first_kt<kPair>(unit_tile(u, p), p);
        for (int kt = kt0; ok && kt < 3; ++kt) {
            const int tt = ti.t + kt - 2;
            const CUtensorMap *am = mapA;
            int fidx = frames;  // out of range: zeros
            if (!ti.dummy) {
                if (tt >= 0) {
                    fidx = ti.n * p.T + tt;
                } else if (p.has_cache) {
                    am = mapC;
                    fidx = ti.n * 2 + tt + 2;
                }
            }
            for (int cc = 0; ok && cc < p.kc_main; ++cc) {
                uint32_t da = 0;
                if (kFuse) {  // the transform warps fill the A buffer
                    skip_abuf();
                } else if (!mine()) {  // the group's first fill, so its halo: the other's
                    skip_abuf();
                } else if (!next_abuf(da)) {
                    ok = false;
                    break;
                }
                for (int g = 0; g < groups; ++g) {
                    if (!mine()) {
                        skip_stage();
                        continue;
                    }
                    uint32_t db, fb;
                    if (!next_stage(p.stage_tx + (g == 0 && !kFuse ? p.a_tx : 0u),
                                    kFuse && g > 0, db, fb)) {
                        ok = false;
                        break;
                    }
                    if (g == 0 && !kFuse) {
                        if (p.halo_rows) {
                            for (int s = 0; s < p.nsub; ++s)  // one region per sw channels
                                load4<kPair>(da + (uint32_t)s * p.sub_stride, am, fb,
                                             (cc * p.nsub + s) * p.sw, ti.w0 - 1, ti.h0 - 1, fidx);
                        } else {
                            load5<kPair>(da, am, fb, 0, ti.w0 - 1, ti.h0 - 1,
                                         cc * (chunk / 8), fidx);
                        }
                    }
                    // tb consecutive spatial taps of this chunk in one box
                    const int wtap = (kt - p.wtap0 / 9) * p.sp_taps + g * p.tb;
                    const int ph = kUp ? unit_phase(u, p) : 0;  // upsampler: its weights
                    load5<kPair>(db, mapB, fb, wtap * p.c_in + cc * chunk,
                                 (int)rank * p.bc_row, (int)rank * p.bc_rank + ph * p.ph_c2,
                                 ph * p.ph_c3, 0);
                }
            }
        }
        // shortcut segment: the patch's own pixels of x (no shift)
        const uint32_t sub_a = (uint32_t)kBlockM * p.sw * 2u;
        for (int cc = 0; ok && cc < p.kc_short; ++cc) {
            uint32_t da, db, fb;
            if (!mine()) {
                skip_abuf();
                skip_stage();
                continue;
            }
            if (!next_abuf(da) || !next_stage(p.nsub * (sub_a + p.b_sub_bytes), kFuse, db, fb)) {
                ok = false;
                break;
            }
            for (int s = 0; s < p.nsub; ++s)
                load4<kPair>(da + (uint32_t)s * sub_a, mapSA, fb, (cc * p.nsub + s) * p.sw, ti.w0,
                             ti.h0, ti.dummy ? frames : ti.frame);
            load5<kPair>(db, mapSB, fb, cc * chunk, 0, (int)rank, 0, 0);
        }
    }
    // (a halo load completes on its group's first stage, so draining the
    // newest fill of every stage covers the halos too)
    producer_finish<kPair>(p, bars, wc, rank, part, last_mine, prod, ok);
}

// Shared-memory address of the 16-byte vector j (channels 8j .. 8j + 7) of
// halo pixel `pix` in an A buffer: one swizzled row per pixel and sw-channel
// region -- 128-byte rows (sw = 64) with the 16-byte column XOR pix & 7, or
// 64-byte rows (sw = 32) with the column XOR (pix >> 1) & 3, the layouts
// TMA's 128- and 64-byte swizzles write into regions aligned to their
// 1024- and 512-byte pattern -- or 8-channel planes of 16 bytes per pixel.
__device__ __forceinline__ uint32_t halo_vec_addr(const ConvArgs &p, uint32_t abuf, int pix,
                                                  int j) {
    if (p.halo_rows && p.sw == 64)
        return abuf + (uint32_t)(j >> 3) * p.sub_stride + (uint32_t)pix * 128u +
               ((uint32_t)((j & 7) ^ (pix & 7)) << 4);
    if (p.halo_rows)
        return abuf + (uint32_t)(j >> 2) * p.sub_stride + (uint32_t)pix * 64u +
               ((uint32_t)((j & 3) ^ ((pix >> 1) & 3)) << 4);
    return abuf + (uint32_t)j * p.plane_bytes + (uint32_t)pix * 16u;
}

// The input norm fused into the halo loads (warps 2 + epi_warps .. 9, four
// warps).  For every halo of the unit sequence, in the producer's order, they
// read the pixels from global memory and write what the MMAs multiply into the
// A buffer: SiLU(RMS_norm(x)) for frames of the clip (every channel of a
// pixel is in the one chunk, so the norm is complete), the cache's frames as
// they are (the cache holds normalised frames), zeros outside the frame or
// the clip.  L lanes share a pixel as in the standalone norm pass, with the
// same arithmetic, so the values are bit for bit that pass's.  Then the
// halo's first weight stage gets its second arrival -- from the leader CTA,
// after the peer CTA reported its halo written and once the stage's previous
// phase has completed.
template <int kPair>
__device__ void conv_transform(const CUtensorMap *mapA, const CUtensorMap *mapC,
                               const ConvArgs &p, uint32_t sbase, const Bars &bars,
                               const WaitCtl &wc, int unit0, int unit_stride, int num_units,
                               uint32_t rank) {
    constexpr int NB = 3;  // pixel iterations whose loads are in flight together
    const int tw = (threadIdx.x >> 5) - 2 - p.epi_warps;  // 0 .. 3
    const int lane = threadIdx.x & 31;
    const int L = p.nl_L, vpt = p.nl_vpt;
    const int sub = lane & (L - 1), grp = lane / L, gpw = 32 / L;
    const int npix = (int)kHaloH * p.halo_w;
    const bool leader = tw == 0 && lane == 0;
    const int groups = p.sp_taps / p.tb;
    const float4 *g4 = reinterpret_cast<const float4 *>(p.gamma_in);
    // Source of the halo of unit u at temporal tap kt: frame index fidx of x
    // (norm) or of the cache, or none (zeros).
    struct Src {
        int fidx;
        bool cache, any;
    };
    auto source = [&](const TileInfo &t2, int kt) -> Src {
        const int tt = t2.t + kt - 2;
        if (t2.dummy) return Src{0, false, false};
        if (tt >= 0) return Src{t2.n * p.T + tt, false, true};
        if (p.has_cache) return Src{t2.n * 2 + tt + 2, true, true};
        return Src{0, false, false};
    };
    // L2 prefetch of a halo box (the loads below then hit L2, not DRAM)
    auto prefetch = [&](const TileInfo &t2, const Src &sr) {
        if (!sr.any) return;
        const CUtensorMap *m = sr.cache ? mapC : mapA;
        if (p.halo_rows) {
            for (int sidx = 0; sidx < p.nsub; ++sidx)
                tma_prefetch_l2_4d(m, sidx * p.sw, t2.w0 - 1, t2.h0 - 1, sr.fidx);
        } else {
            tma_prefetch_l2_5d(m, 0, t2.w0 - 1, t2.h0 - 1, 0, sr.fidx);
        }
    };
    int stage = 0, ia = 0;
    uint32_t phase = 0, pha = 0, peer_par = 0;
    bool ok = true;
    if (leader && unit0 < num_units) {  // the first halo
        const int u = unit0, kt = unit_first_kt<kPair>(unit_tile(u, p), p);
        const TileInfo t2 = tile_info(unit_tile(u, p) * kPair + (int)rank, p);
        prefetch(t2, source(t2, kt));
    }
    for (int u = unit0; ok && u < num_units; u += unit_stride) {
        const TileInfo ti = tile_info(unit_tile(u, p) * kPair + (int)rank, p);
        const int kt0 = unit_first_kt<kPair>(unit_tile(u, p), p);
        for (int kt = kt0; ok && kt < 3; ++kt) {
            const Src sr = source(ti, kt);
            const __nv_bfloat16 *src =
                !sr.any ? nullptr
                        : (sr.cache ? p.cache_in : p.x_in) + (size_t)sr.fidx * p.HW * p.c_in;
            const bool norm = sr.any && !sr.cache;
            if (leader) {  // the next halo, into L2 while this one is built
                int un = u, ktn = kt + 1;
                if (ktn == 3) {
                    un = u + unit_stride;
                    ktn = un < num_units ? unit_first_kt<kPair>(unit_tile(un, p), p) : 0;
                }
                if (un < num_units) {
                    const TileInfo tn = tile_info(unit_tile(un, p) * kPair + (int)rank, p);
                    prefetch(tn, source(tn, ktn));
                }
            }
            const int slot = ia;
            const uint32_t slot_par = pha;
            if (++ia == p.na) {
                ia = 0;
                pha ^= 1u;
            }
            const int s0 = stage;
            const uint32_t ph0 = phase;
            for (int g = 0; g < groups; ++g)
                if (++stage == p.stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            // the A buffer is free once the MMAs of its previous halo are done
            ok = mbar_wait_warp<kPair == 2>(bars.emptya(slot), slot_par ^ 1u, wc);
            if (bar_any(2, 128, !ok)) {
                ok = false;
                break;
            }
            const uint32_t abuf = sbase + p.off_a + (uint32_t)slot * p.a_stride;
            for (int pb = tw * gpw; pb < npix; pb += 4 * gpw * NB) {  // warp-uniform bound
                uint4 v[NB][kMaxNormVpt];
                bool in[NB];
#pragma unroll
                for (int b = 0; b < NB; ++b) {  // every load of NB iterations first
                    const int pix = pb + b * 4 * gpw + grp;
                    const int hy = pix / p.halo_w, hx = pix - hy * p.halo_w;
                    const int h = ti.h0 - 1 + hy, w = ti.w0 - 1 + hx;
                    in[b] = pix < npix && src && h >= 0 && h < p.H && w >= 0 && w < p.W;
                    const uint4 *pv = reinterpret_cast<const uint4 *>(
                        src + ((size_t)(in[b] ? h : 0) * p.W + (in[b] ? w : 0)) * p.c_in);
#pragma unroll
                    for (int i = 0; i < kMaxNormVpt; ++i)
                        if (i < vpt)
                            v[b][i] = in[b] ? __ldg(pv + sub + i * L) : make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int b = 0; b < NB; ++b) {
                    const int pix = pb + b * 4 * gpw + grp;
                    float ss = 0.f;
#pragma unroll
                    for (int i = 0; i < kMaxNormVpt; ++i)
                        if (i < vpt && norm) ss = nact_sumsq8(v[b][i], ss);
                    if (norm) ss = nact_group_sum(ss, L);  // (norm is uniform over the warp)
                    const float scale = nact_scale(ss, p.sqrt_c_in, p.eps);
#pragma unroll
                    for (int i = 0; i < kMaxNormVpt; ++i) {
                        if (i < vpt && pix < npix) {
                            const int j = sub + i * L;
                            const uint4 o = (norm && in[b])
                                                ? nact_apply8<true>(v[b][i], scale,
                                                                    __ldg(g4 + 2 * j),
                                                                    __ldg(g4 + 2 * j + 1))
                                                : v[b][i];
                            const uint32_t a = halo_vec_addr(p, abuf, pix, j);
                            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(a),
                                         "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w)
                                         : "memory");
                        }
                    }
                }
            }
            fence_proxy_async_smem();  // the tensor core reads the halo (async proxy)
            asm volatile("bar.sync 2, 128;" ::: "memory");
            if (leader) {
                if (kPair == 2 && rank == 1) {
                    mbar_arrive_cluster(mapa_shared(bars.peer(slot), 0));
                } else {
                    bool w = true;
                    if (kPair == 2) {
                        w = mbar_wait<true>(bars.peer(slot), (peer_par >> slot) & 1u, wc);
                        peer_par ^= 1u << slot;
                    }
                    // this arrival belongs to the stage's phase ph0: the one
                    // before must have completed
                    if (w) w = mbar_wait<kPair == 2>(bars.full(s0), ph0 ^ 1u, wc);
                    if (w) mbar_arrive_cluster(bars.full(s0));
                }
            }
        }
    }
}

// Halo-mode MMAs of one spatial tap and one 128-row sub-tile: k-step ks =
// s KK + kk reads the halo window at a0 + s a_sub16 + kk a_kk16 (descriptor
// units) and B sub-tile s (b_sub16 apart) at k-offset kk.
template <int kPair, int KK, int NSUB, int NP>
__device__ __forceinline__ void issue_tap_halo(const ConvArgs &p, uint32_t dacc, uint64_t a0,
                                               uint64_t b0, uint32_t b_sub16, uint32_t a_sub16,
                                               uint32_t a_kk16, uint32_t idesc, bool first,
                                               int np_run) {
    const uint32_t piece16 = (uint32_t)(p.piece_n / kPair) * (uint32_t)p.sw * 2u >> 4;
    auto mma = [&](int s, int kk, int ks, int j) {
        const uint64_t ad = a0 + (uint64_t)(s * a_sub16 + kk * a_kk16);
        const uint64_t bd = b0 + (uint64_t)(s * b_sub16 + j * piece16 + 2 * kk);
        const uint32_t accum = (first && ks == 0) ? 0u : 1u;
        const uint32_t d = dacc + (uint32_t)(j * p.piece_n);
        if (kPair == 2)
            mma_bf16_ss_pair(d, ad, bd, idesc, accum);
        else
            mma_bf16_ss(d, ad, bd, idesc, accum);
    };
    if (KK > 0) {
#pragma unroll
        for (int s = 0; s < NSUB; ++s)
#pragma unroll
            for (int kk = 0; kk < KK; ++kk)
#pragma unroll
                for (int j = 0; j < NP; ++j) mma(s, kk, s * KK + kk, j);
    } else {
        const int kk_n = p.sw / 16;
        for (int s = 0; s < p.nsub; ++s)
            for (int kk = 0; kk < kk_n; ++kk)
                for (int j = 0; j < np_run; ++j) mma(s, kk, s * kk_n + kk, j);
    }
}

// Issue the MMAs of one pipeline stage.  KK k-steps of 16 per swizzled
// sub-tile, NSUB sub-tiles, NP N-pieces: all compile-time, so the loop is fully
// unrolled and every descriptor is the stage's base plus a constant (the
// issuing thread must not spend more cycles between two MMAs than one MMA
// takes on the tensor core).  KK == 0 selects the run-time-bounded form for
// shapes without a specialisation, over np_run pieces.
template <int kPair, int KK, int NSUB, int NP>
__device__ __forceinline__ void issue_stage(const ConvArgs &p, uint32_t dacc, uint64_t a0,
                                            uint64_t b0, uint32_t idesc, bool first,
                                            int np_run) {
    const uint32_t a_sub16 = p.a_sub_bytes >> 4, b_sub16 = p.b_sub_bytes >> 4;
    const uint32_t piece16 = (uint32_t)(p.piece_n / kPair) * (uint32_t)p.sw * 2u >> 4;
    if (KK > 0) {
#pragma unroll
        for (int s = 0; s < NSUB; ++s) {
#pragma unroll
            for (int kk = 0; kk < KK; ++kk) {
                const uint64_t ad = a0 + (uint64_t)(s * a_sub16 + 2 * kk);
                const uint32_t accum = (first && s == 0 && kk == 0) ? 0u : 1u;
#pragma unroll
                for (int j = 0; j < NP; ++j) {
                    const uint64_t bd = b0 + (uint64_t)(s * b_sub16 + j * piece16 + 2 * kk);
                    const uint32_t d = dacc + (uint32_t)(j * p.piece_n);
                    if (kPair == 2)
                        mma_bf16_ss_pair(d, ad, bd, idesc, accum);
                    else
                        mma_bf16_ss(d, ad, bd, idesc, accum);
                }
            }
        }
    } else {
        for (int s = 0; s < p.nsub; ++s) {
            for (int kk = 0; kk < p.sw / 16; ++kk) {
                const uint64_t ad = a0 + (uint64_t)(s * a_sub16 + 2 * kk);
                const uint32_t accum = (first && s == 0 && kk == 0) ? 0u : 1u;
                for (int j = 0; j < np_run; ++j) {
                    const uint64_t bd = b0 + (uint64_t)(s * b_sub16 + j * piece16 + 2 * kk);
                    const uint32_t d = dacc + (uint32_t)(j * p.piece_n);
                    if (kPair == 2)
                        mma_bf16_ss_pair(d, ad, bd, idesc, accum);
                    else
                        mma_bf16_ss(d, ad, bd, idesc, accum);
                }
            }
        }
    }
}

// Halo-mode MMA issuer: per (kt, chunk), 9 / tb weight stages of tb spatial
// taps, each tap reading the halo through a window shifted by (kh, kw) for
// each of the nq sub-tiles (one TMEM accumulator each); the halo buffer is
// released after the ninth tap.  Descriptors are the ring bases plus
// offsets, so nothing but the stage bookkeeping sits between two stages'
// MMAs.  With two issuers (p.issuers == 2) issuer `part` runs every stage for
// sub-tile `part` (nq == 2) or for N piece `part`: the same MMAs, in the same
// order per accumulator, split by accumulator.
template <int kPair, int KK, int NSUB, int NP, bool kUp>
__device__ void conv_mma_halo(const ConvArgs &p, uint32_t sbase, uint32_t tmem_base,
                              const Bars &bars, const WaitCtl &wc, int unit0, int unit_stride,
                              int num_units, int part) {
    const uint32_t idesc = idesc_bf16_f32(kBlockM * kPair, p.piece_n);
    const uint32_t row_bytes = (uint32_t)p.sw * 2u;
    const uint32_t b_sub16 = p.b_sub_bytes >> 4;
    const uint32_t tap_b16 = (uint32_t)p.nsub * b_sub16;  // one tap's weights
    const uint32_t stage16 = p.stage_bytes >> 4, astride16 = p.a_stride >> 4;
    // Halo windows, 8-pixel groups one halo row apart.  Rows: one swizzled
    // row per pixel, sw-channel regions sub_stride apart, k-steps 32 B apart.
    // Planes: 16 bytes per pixel, k-steps two 8-channel planes apart.
    const uint32_t px16 = p.halo_rows ? row_bytes >> 4 : 1u;
    const uint32_t hrow16 = (uint32_t)p.halo_w * px16;
    const uint32_t a_kk16 = p.halo_rows ? 2u : (2u * p.plane_bytes) >> 4;
    const uint32_t a_sub16 = p.halo_rows ? p.sub_stride >> 4 : (uint32_t)(p.sw / 16) * a_kk16;
    const uint64_t bdesc0 = sdesc_kmajor(sbase + p.a_bytes, row_bytes, p.layout);
    const uint64_t adesc0 =
        p.halo_rows ? sdesc_kmajor_sbo(sbase + p.off_a, (uint32_t)p.halo_w * row_bytes, p.layout)
                    : sdesc_plain(sbase + p.off_a, p.plane_bytes, (uint32_t)p.halo_w * 16u);
    const bool tb3 = p.tb == 3, tb4 = kUp && p.tb == 4;
    const int nst = p.tb == 1 ? p.sp_taps : (tb3 ? 3 : 1);  // weight stages per (kt, chunk)
    // This issuer's share: a sub-tile (its accumulator and its halo window
    // 8 pixels along), or an N piece (its accumulator columns and its rows of
    // every weight stage).
    const bool split_q = p.issuers == 2 && p.nq == 2;
    const bool split_n = p.issuers == 2 && p.nq != 2;
    const int nq_run = split_q ? 1 : p.nq;
    const int np_run = split_n ? 1 : p.n_pieces;
    const uint32_t piece16 = (uint32_t)(p.piece_n / kPair) * row_bytes >> 4;
    const uint32_t d_part =
        split_q ? (uint32_t)(part * p.acc_cols) : (split_n ? (uint32_t)(part * p.piece_n) : 0u);
    const uint64_t a_part = split_q ? (uint64_t)(8 * part) * px16 : 0u;
    const uint64_t b_part = split_n ? (uint64_t)part * piece16 : 0u;
    FullRing<kPair == 2> ring;
    int ia = 0, it = 0;
    bool ok = true;
    auto commit = [&](uint32_t bar) {
        if (kPair == 2)
            mma_commit_pair_mc(bar, (uint16_t)0x3);
        else
            mma_commit(bar);
    };
    // One stage: NTAP taps from (kh, kw0), NW to a tap row (3 x 1 of a plain
    // conv's row, 2 x 2 of an upsampler phase, or one tap), for NQ sub-tiles
    // and NPc N pieces.  All compile-time, so the whole stage is one straight
    // run of MMAs.
    auto stage = [&](auto nq_c, auto ntap_c, auto nw_c, auto np_c, uint32_t dacc, uint64_t abase,
                     int kh, int kw0, bool first) {
        constexpr int NQ = decltype(nq_c)::value, NTAP = decltype(ntap_c)::value;
        constexpr int NW = decltype(nw_c)::value, NPc = decltype(np_c)::value;
        const uint64_t b0 = bdesc0 + (uint64_t)(ring.stage * stage16) + b_part;
        const uint64_t ah = abase + (uint64_t)(kh * hrow16 + kw0 * px16);
#pragma unroll
        for (int j = 0; j < NTAP; ++j)
#pragma unroll
            for (int sq = 0; sq < NQ; ++sq)
                issue_tap_halo<kPair, KK, NSUB, NPc>(
                    p, dacc + (uint32_t)(sq * p.acc_cols),
                    ah + (uint64_t)((j / NW) * hrow16 + (j % NW + 8 * sq) * px16),
                    b0 + (uint64_t)(j * tap_b16), b_sub16, a_sub16, a_kk16, idesc,
                    first && j == 0, np_run);
    };
    using I1 = std::integral_constant<int, 1>;
    using I2 = std::integral_constant<int, 2>;
    using I3 = std::integral_constant<int, 3>;
    using I4 = std::integral_constant<int, 4>;
    // (4-tap stages exist in the upsampler's kernels only)
    auto any_stage = [&](auto np_c, uint32_t dacc, uint64_t abase, int kh, int kw0, bool first) {
        if (nq_run == 2) {
            if (tb3) stage(I2{}, I3{}, I3{}, np_c, dacc, abase, kh, kw0, first);
            else if (kUp && tb4) stage(I2{}, I4{}, I2{}, np_c, dacc, abase, kh, kw0, first);
            else stage(I2{}, I1{}, I1{}, np_c, dacc, abase, kh, kw0, first);
        } else {
            if (tb3) stage(I1{}, I3{}, I3{}, np_c, dacc, abase, kh, kw0, first);
            else if (kUp && tb4) stage(I1{}, I4{}, I2{}, np_c, dacc, abase, kh, kw0, first);
            else stage(I1{}, I1{}, I1{}, np_c, dacc, abase, kh, kw0, first);
        }
    };
    for (int u = unit0; ok && u < num_units; u += unit_stride, ++it) {
        const int a = it % p.nacc;
        const uint32_t aph = (uint32_t)(it / p.nacc) & 1u;
        if (!mbar_wait<kPair == 2>(bars.acce(a), aph ^ 1u, wc)) break;
        tc_fence_after();
        const uint32_t dacc = tmem_base + (uint32_t)(a * p.acc_stride) + d_part;
        const int kt0 = unit_first_kt<kPair>(unit_tile(u, p), p);
        const TapBase tbase = kUp ? unit_tap_base(u, p) : TapBase{0, 0};
        bool first = true;
        for (int kt = kt0; ok && kt < 3; ++kt) {
            for (int cc = 0; ok && cc < p.kc_main; ++cc) {
                const uint64_t abase = adesc0 + (uint64_t)(ia * astride16) + a_part;
                // the first stage of (kt, cc) also carries the halo; the
                // stage's first tap (kh, kw0) steps by tb along rows of sp_w
                int kh = tbase.kh, kw0 = tbase.kw;
                for (int g = 0; g < nst; ++g) {
                    if (!ring.acquire(bars, wc)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if constexpr (NP == 2) {
                        if (split_n) any_stage(I1{}, dacc, abase, kh, kw0, first);
                        else any_stage(I2{}, dacc, abase, kh, kw0, first);
                    } else {
                        any_stage(std::integral_constant<int, NP>{}, dacc, abase, kh, kw0, first);
                    }
                    first = false;
                    commit(bars.empty(ring.stage));
                    ring.advance(bars);
                    kw0 += p.tb;
                    if (kw0 - tbase.kw >= p.sp_w) {  // tb is 1, a whole row or a whole phase
                        kw0 = tbase.kw;
                        kh += p.tb > p.sp_w ? 2 : 1;
                    }
                }
                if (!ok) break;
                commit(bars.emptya(ia));
                if (++ia == p.na) ia = 0;
            }
        }
        for (int cc = 0; ok && cc < p.kc_short; ++cc) {
            if (!ring.acquire(bars, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // x patch in the A buffer, swizzled like the weights: the stage
            // issue routine of the im2col path applies unchanged.  (Plans with
            // a shortcut have one sub-tile, so a split is by N piece.)
            const uint32_t abuf = sbase + p.off_a + (uint32_t)ia * p.a_stride;
            const uint32_t sb = sbase + p.a_bytes + (uint32_t)ring.stage * p.stage_bytes;
            const uint64_t ad = sdesc_kmajor(abuf, row_bytes, p.layout);
            const uint64_t bd = sdesc_kmajor(sb, row_bytes, p.layout) + b_part;
            if constexpr (NP == 2) {
                if (split_n) issue_stage<kPair, KK, NSUB, 1>(p, dacc, ad, bd, idesc, first, 1);
                else issue_stage<kPair, KK, NSUB, 2>(p, dacc, ad, bd, idesc, first, 2);
            } else {
                issue_stage<kPair, KK, NSUB, NP>(p, dacc, ad, bd, idesc, first, np_run);
            }
            first = false;
            commit(bars.empty(ring.stage));
            commit(bars.emptya(ia));
            ring.advance(bars);
            if (++ia == p.na) ia = 0;
        }
        if (!ok) break;
        commit(bars.accf(a));
    }
    volatile int no_abort = 0;
    const WaitCtl dc{kDrainNs, wc.err, &no_abort, kDevErrTimeout | kDevErrDrain};
    if (kPair == 2)
        mma_commit_pair(bars.drain());
    else
        mma_commit(bars.drain());
    mbar_wait<kPair == 2>(bars.drain(), 0u, dc);
}

// MMA issuer (one thread of the leader CTA).  With two issuers, issuer
// `part` runs every stage for N piece `part` (its accumulator columns and its
// rows of each weight stage).
template <int kPair, int KK, int NSUB, int NP>
__device__ void conv_mma(const ConvArgs &p, uint32_t sbase, uint32_t tmem_base, const Bars &bars,
                         const WaitCtl &wc, int unit0, int unit_stride, int num_units, int part) {
    const uint32_t idesc = idesc_bf16_f32(kBlockM * kPair, p.piece_n);
    const uint32_t row_bytes = (uint32_t)p.sw * 2u;
    const bool split_n = p.issuers == 2;
    const uint32_t d_part = split_n ? (uint32_t)(part * p.piece_n) : 0u;
    const uint64_t b_part =
        split_n ? (uint64_t)((uint32_t)(p.piece_n / kPair) * row_bytes >> 4) * (uint64_t)part : 0u;
    FullRing<kPair == 2> ring;
    int it = 0;
    bool ok = true;
    for (int u = unit0; ok && u < num_units; u += unit_stride, ++it) {
        const int a = it % p.nacc;
        const uint32_t aph = (uint32_t)(it / p.nacc) & 1u;
        if (!mbar_wait<kPair == 2>(bars.acce(a), aph ^ 1u, wc)) break;
        tc_fence_after();
        const uint32_t dacc = tmem_base + (uint32_t)(a * p.acc_stride) + d_part;
        const int nst = unit_stages<kPair>(unit_tile(u, p), p);
        for (int k = 0; k < nst; ++k) {
            if (!ring.acquire(bars, wc)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t sa = sbase + (uint32_t)ring.stage * p.stage_bytes;
            const uint64_t ad = sdesc_kmajor(sa, row_bytes, p.layout);
            const uint64_t bd = sdesc_kmajor(sa + p.a_bytes, row_bytes, p.layout) + b_part;
            if constexpr (NP == 2) {
                if (split_n) issue_stage<kPair, KK, NSUB, 1>(p, dacc, ad, bd, idesc, k == 0, 1);
                else issue_stage<kPair, KK, NSUB, 2>(p, dacc, ad, bd, idesc, k == 0, 2);
            } else {
                issue_stage<kPair, KK, NSUB, NP>(p, dacc, ad, bd, idesc, k == 0,
                                                 split_n ? 1 : p.n_pieces);
            }
            // Frees the smem stage (in both CTAs of a pair) when these MMAs finish.
            if (kPair == 2)
                mma_commit_pair_mc(bars.empty(ring.stage), (uint16_t)0x3);
            else
                mma_commit(bars.empty(ring.stage));
            ring.advance(bars);
        }
        if (!ok) break;
        // Accumulator ready for the epilogue (of both CTAs of a pair).
        if (kPair == 2)
            mma_commit_pair_mc(bars.accf(a), (uint16_t)0x3);
        else
            mma_commit(bars.accf(a));
    }
    // Every MMA issued above completes before TMEM is released.
    volatile int no_abort = 0;
    const WaitCtl dc{kDrainNs, wc.err, &no_abort, kDevErrTimeout | kDevErrDrain};
    if (kPair == 2)
        mma_commit_pair(bars.drain());
    else
        mma_commit(bars.drain());
    mbar_wait<kPair == 2>(bars.drain(), 0u, dc);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Where the 32 rows of one epilogue warp live in the output: consecutive
// voxels (im2col tiles; rows past the frame's end are invalid), or four patch
// rows of 8 pixels one frame row (W voxels) apart (halo tiles; rows and
// columns past the frame are invalid).
struct RowMap {
    int seg_rows;    // rows per contiguous segment (32 or 8)
    int64_t pitch;   // voxels between segments
    int nseg, ncol;  // valid segments, valid rows per segment
    __device__ __forceinline__ bool valid(int r) const {
        return r / seg_rows < nseg && r % seg_rows < ncol;
    }
    __device__ __forceinline__ int64_t offset(int r) const {
        return (int64_t)(r / seg_rows) * pitch + r % seg_rows;
    }
};

__device__ __forceinline__ RowMap warp_rows(const ConvArgs &p, const TileInfo &ti, int q,
                                            int sub = 0) {
    RowMap rm;
    if (p.halo) {
        rm.seg_rows = 8;
        rm.pitch = p.W;
        const int ns = p.H - ti.h0 - 4 * q, nc = p.W - ti.w0 - 8 * sub;
        rm.nseg = ti.dummy ? 0 : (ns < 0 ? 0 : (ns > 4 ? 4 : ns));
        rm.ncol = nc < 0 ? 0 : (nc > 8 ? 8 : nc);
    } else {
        rm.seg_rows = 32;
        rm.pitch = 0;
        const int nv = ti.dummy ? 0 : p.HW - ti.pos - q * 32;
        rm.nseg = 1;
        rm.ncol = nv < 0 ? 0 : (nv > 32 ? 32 : nv);
    }
    return rm;
}

// Write one warp's 32-row x n-channel (n = 16 or 32) bf16 chunk: each lane
// hands its row's n/8 16-byte pieces (o) to a swizzled shared buffer, then the
// warp writes the chunk back four lanes per row, so every store instruction
// covers eight whole 64-byte row segments instead of 32 scattered 16-byte
// pieces.  Rows at or past `nvalid` (the frame's end) are not written.
__device__ __forceinline__ void store_chunk(uint8_t *stg, const uint32_t (&o)[16], int n,
                                            __nv_bfloat16 *out_row0, int ldc, int c,
                                            const RowMap &rm) {
    const int lane = threadIdx.x & 31;
    const int np = n / 8;  // 16-byte pieces per row
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        if (k < np) {
            const int slot = k ^ ((lane >> 1) & 3);
            *reinterpret_cast<uint4 *>(stg + lane * 64 + slot * 16) =
                make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        }
    }
    __syncwarp();
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int r = j * 8 + (lane >> 2), q = lane & 3;
        if (q < np && rm.valid(r)) {
            const int slot = q ^ ((r >> 1) & 3);
            const uint4 v = *reinterpret_cast<const uint4 *>(stg + r * 64 + slot * 16);
            *reinterpret_cast<uint4 *>(out_row0 + rm.offset(r) * ldc + c + q * 8) = v;
        }
    }
    __syncwarp();
}

// Epilogue warps: warp w reads TMEM lane quarter (w % 4) -- the hardware's
// rule -- and owns half of the columns (half (w - 2) / 4), so two warps share
// every row.  The fused RMS_norm combines their two partial sums of squares
// through shared memory.
template <int kPair, bool kUp>
__device__ void conv_epilogue(const ConvArgs &p, uint32_t tmem_base, const float *s_bias,
                              const float *s_gamma, float *s_part, uint8_t *stg,
                              const CUtensorMap *mapY, const Bars &bars, const WaitCtl &wc,
                              int unit0, int unit_stride, int num_units, uint32_t rank) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;           // TMEM lane quarter this warp may read
    const int half = (warp - 2) >> 2; // 0 or 1: which column half
    const int row = q * 32 + lane;
    // eight epilogue warps: two per lane quarter, each half the columns;
    // four: one per lane quarter, all of them
    const int c_split = p.epi_warps == 8 ? ((p.c_out / 2) + 15) / 16 * 16 : p.c_out;
    const int c_begin = half ? c_split : 0, c_end = half ? p.c_out : c_split;
    int it = 0;
    for (int u = unit0; u < num_units; u += unit_stride, ++it) {
        const int a = it % p.nacc;
        const uint32_t aph = (uint32_t)(it / p.nacc) & 1u;
        // (the unit's tile, worked out while its MMAs still run)
        const TileInfo ti = tile_info(unit_tile(u, p) * kPair + (int)rank, p);
        bool handed_back = false;  // (the bias and residual epilogue hands back early)
        const bool got = mbar_wait_warp<kPair == 2>(bars.accf(a), aph, wc);
        if (p.epi == kEpiNormSilu) {
            // The norm's halves meet at a named barrier below, so all epilogue
            // warps take the same decision: stop if any of them gave up.
            if (bar_any(1, 32 * p.epi_warps, !got)) break;
        } else if (!got) {
            break;
        }
        tc_fence_after();
        for (int sub = 0; sub < p.nq; ++sub) {
        // This warp's 32 rows of sub-tile `sub`; rows outside the frame (or
        // of an empty pair slot) are not stored.
        const RowMap rm = warp_rows(p, ti, q, sub);
        const bool valid = rm.valid(lane);
        const int64_t wbase = p.halo ? (int64_t)ti.row0 + (int64_t)(4 * q) * p.W + 8 * sub
                                     : (int64_t)ti.row0 + q * 32;
        const int64_t g = wbase + rm.offset(lane);
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) +
                            (uint32_t)(a * p.acc_stride + sub * p.acc_cols);
        __nv_bfloat16 *out_w = p.out + wbase * p.c_out;
        float *part = s_part + sub * 2 * kBlockM;  // each sub-tile its own partial sums
        if (p.narrow) {
            // c_out < 16 (bias epilogue only): one 16-column TMEM load, then
            // each row's c_out channels as scalar bf16 stores.
            if (half == 0) {
                uint32_t r[32];
                tmem_ld_cols(tb, 16, r);
                if (valid) {
                    __nv_bfloat16 *o = p.out + g * p.c_out;
#pragma unroll
                    for (int c = 0; c < 16; ++c)  // constant indexes keep r in registers
                        if (c < p.c_out)
                            o[c] = __float2bfloat16_rn(__uint_as_float(r[c]) + s_bias[c]);
                }
            }
        } else if (p.epi == kEpiNormSilu) {
            // RMS_norm over all c_out channels of this voxel, then SiLU.  The
            // sum of squares is taken over two column halves and then added,
            // whether two warps share the row (eight epilogue warps) or one
            // warp has all of it (four): the same value either way.
            const int c_half = ((p.c_out / 2) + 15) / 16 * 16;
            float ssh[2] = {0.f, 0.f};
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int cb = hh ? c_half : 0, ce = hh ? p.c_out : c_half;
                if (p.epi_warps == 8 && hh != half) continue;
                float ss = 0.f;
                for (int c = cb; c < ce; c += 32) {
                    uint32_t r[32];
                    const int n = ce - c >= 32 ? 32 : 16;
                    tmem_ld_cols(tb + (uint32_t)c, n, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if (i < n) {
                            const float v = __fadd_rn(__uint_as_float(r[i]), s_bias[c + i]);
                            ss = __fmaf_rn(v, v, ss);
                        }
                    }
                }
                ssh[hh] = ss;
            }
            float tot = __fadd_rn(ssh[0], ssh[1]);
            if (p.epi_warps == 8) {
                part[half * kBlockM + row] = ssh[half];
                asm volatile("bar.sync 1, %0;" ::"r"(32 * p.epi_warps) : "memory");
                tot = __fadd_rn(part[row], part[kBlockM + row]);
            }
            const float scale = p.sqrt_c / fmaxf(sqrtf(tot), p.eps);
            for (int c = c_begin; c < c_end; c += 32) {
                uint32_t r[32];
                const int n = c_end - c >= 32 ? 32 : 16;
                tmem_ld_cols(tb + (uint32_t)c, n, r);
                uint32_t o[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (2 * i < n) {
                        float z0 = (__uint_as_float(r[2 * i]) + s_bias[c + 2 * i]) * scale *
                                   s_gamma[c + 2 * i];
                        float z1 = (__uint_as_float(r[2 * i + 1]) + s_bias[c + 2 * i + 1]) *
                                   scale * s_gamma[c + 2 * i + 1];
                        z0 = __fdividef(z0, 1.0f + __expf(-z0));
                        z1 = __fdividef(z1, 1.0f + __expf(-z1));
                        o[i] = pack_bf16x2(z0, z1);
                    }
                }
                store_chunk(stg, o, n, out_w, p.c_out, c, rm);
            }
            // A sub-tile's partial sums are rewritten only after the next
            // tile's bar_any, which every warp reaches after its last read.
        } else {
            const uint4 *res = p.epi == kEpiResidual
                                   ? reinterpret_cast<const uint4 *>(p.resid + g * p.c_out)
                                   : nullptr;
            for (int c = c_begin; c < c_end; c += 32) {
                uint32_t r[32];
                const int n = c_end - c >= 32 ? 32 : 16;
                // The bias and residual loads go out before the TMEM load
                // (whose wait the compiler cannot move them across), so
                // their latencies overlap instead of adding up.
                float v[32];
#pragma unroll
                for (int i = 0; i < 32; i += 4) {
                    if (i < n) {
                        const float4 b4 = *reinterpret_cast<const float4 *>(s_bias + c + i);
                        v[i] = b4.x;
                        v[i + 1] = b4.y;
                        v[i + 2] = b4.z;
                        v[i + 3] = b4.w;
                    }
                }
                uint4 x4[4];
                if (res && valid) {
#pragma unroll
                    for (int vv = 0; vv < 4; ++vv)
                        if (8 * vv < n) x4[vv] = res[c / 8 + vv];
                }
                tmem_ld_cols(tb + (uint32_t)c, n, r);
                if (sub == p.nq - 1 && c + 32 >= c_end) {
                    // The unit's last TMEM load: hand the accumulator back
                    // now, not after the stores -- the issuer's next MMAs
                    // into it wait for this, so the stores' latency would
                    // otherwise sit between two units' MMAs.
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        if (kPair == 2)
                            mbar_arrive_remote(mapa_shared(bars.acce(a), 0));
                        else
                            mbar_arrive(bars.acce(a));
                    }
                    handed_back = true;
                }
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    if (i < n) v[i] = __uint_as_float(r[i]) + v[i];
                if (res && valid) {
#pragma unroll
                    for (int vv = 0; vv < 4; ++vv) {
                        if (8 * vv < n) {
                            const uint32_t xs[4] = {x4[vv].x, x4[vv].y, x4[vv].z, x4[vv].w};
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                v[8 * vv + 2 * i] += __uint_as_float(xs[i] << 16);
                                v[8 * vv + 2 * i + 1] += __uint_as_float(xs[i] & 0xffff0000u);
                            }
                        }
                    }
                }
                uint32_t o[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) o[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
                if (kUp && p.up_tma) {
                    // Upsampler on halo tiles: the warp's 4 x 8 low-res pixels
                    // are boxes of the phase view of y (its pixels 2 apart),
                    // up_box channels each.  The whole sub-tile's channels are
                    // staged ([box][pixel][up_box channels]) and leave by TMA
                    // stores after its last chunk; the buffer is reused once
                    // the previous sub-tile's stores have read it.
                    if (c == c_begin) {
                        if (lane == 0) bulk_wait_read_all();
                        __syncwarp();
                    }
                    const int box_bytes = 64 * p.up_box;  // 32 pixels x up_box x 2 B
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (16 * h < n) {
                            const int cc = c - c_begin + 16 * h;
                            uint4 *d = reinterpret_cast<uint4 *>(
                                stg + (cc / p.up_box) * box_bytes + lane * 2 * p.up_box +
                                2 * (cc % p.up_box));
                            d[0] = make_uint4(o[8 * h], o[8 * h + 1], o[8 * h + 2], o[8 * h + 3]);
                            d[1] = make_uint4(o[8 * h + 4], o[8 * h + 5], o[8 * h + 6],
                                              o[8 * h + 7]);
                        }
                    }
                    if (c + 32 >= c_end) {  // the sub-tile's last chunk: store it
                        fence_proxy_async_smem();
                        __syncwarp();
                        const int ph = unit_phase(u, p);
                        if (lane == 0 && !ti.dummy && ti.h0 + 4 * q < p.H &&
                            ti.w0 + 8 * sub < p.W) {  // (a box past the frame: nothing)
                            for (int k = 0; k * p.up_box < c_end - c_begin; ++k) {
                                const uint32_t src = smem_u32(stg + k * box_bytes);
                                if (src & 127u) {  // a bulk tensor copy needs 128-byte alignment
                                    atomicOr(p.err, kDevErrAlign);
                                    break;
                                }
                                tma_store_5d(mapY, src,
                                             (ph & 1) * p.c_out + c_begin + k * p.up_box,
                                             ti.w0 + 8 * sub, ph >> 1, ti.h0 + 4 * q, ti.frame);
                            }
                            bulk_commit();
                        }
                    }
                } else if (kUp) {
                    // Spatial upsampler: low-res pixel (i, j) of this row is
                    // output pixel (2i + a, 2j + b) of the unit's phase (a, b).
                    // Temporal upsampler: frame t of batch element n is output
                    // frame 2t + a of the unit's phase a.
                    if (valid) {
                        const int64_t pos = g - (int64_t)ti.frame * p.HW;  // in the frame
                        const int ph = unit_phase(u, p);
                        int64_t dst;
                        if (p.up_t) {
                            dst = (((int64_t)ti.n * 2 * p.T + 2 * ti.t + ph) * p.HW + pos) *
                                      p.c_out + c;
                        } else {
                            const int64_t i = pos / p.W, j = pos - i * p.W;
                            dst = (((int64_t)ti.frame * 2 * p.H + 2 * i + (ph >> 1)) * 2 * p.W +
                                   2 * j + (ph & 1)) * p.c_out + c;
                        }
                        uint4 *d = reinterpret_cast<uint4 *>(p.out + dst);
#pragma unroll
                        for (int vv = 0; vv < 4; ++vv)
                            if (8 * vv < n)
                                d[vv] = make_uint4(o[4 * vv], o[4 * vv + 1], o[4 * vv + 2],
                                                   o[4 * vv + 3]);
                    }
                } else {
                    store_chunk(stg, o, n, out_w, p.c_out, c, rm);
                }
            }
        }
        }  // sub-tiles
        if (!handed_back) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                // Accumulator drained: tell the MMA issuer (in the leader CTA).
                if (kPair == 2)
                    mbar_arrive_remote(mapa_shared(bars.acce(a), 0));
                else
                    mbar_arrive(bars.acce(a));
            }
        }
    }
    if (kUp && p.up_tma && lane == 0) bulk_wait_all();  // stores done before the CTA leaves
}

// Whole-tile staged epilogue (one TMEM accumulator, c_out a multiple of 64).
// The epilogue warps turn the accumulator into the bf16 output tile inside a
// shared buffer laid out as TMA's 128-byte swizzle expects ([c_out/64] blocks
// of 128 rows x 64 channels), hand TMEM back to the MMA warp at once, and one
// thread drains the buffer to global memory with asynchronous bulk tensor
// stores while the next tile's MMAs run.  For the residual epilogue the x tile
// is brought into the same buffer by TMA during the mainloop (rows past the
// frame read as zeros and are never stored: the 3-D maps clip them).
template <int kPair>
__device__ void conv_epilogue_staged(const ConvArgs &p, uint32_t tmem_base, const float *s_bias,
                                     const float *s_gamma, float *s_part, uint8_t *buf,
                                     const CUtensorMap *mapY, const CUtensorMap *mapR,
                                     const Bars &bars, const WaitCtl &wc, int unit0,
                                     int unit_stride, int num_units, uint32_t rank) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    // eight epilogue warps: two per lane quarter, each half the columns;
    // four: one per lane quarter, all of them
    const int c_split = p.epi_warps == 8 ? ((p.c_out / 2) + 15) / 16 * 16 : p.c_out;
    const int c_begin = half ? c_split : 0, c_end = half ? p.c_out : c_split;
    const bool issuer = warp == 2 && lane == 0;
    const bool resid = p.epi == kEpiResidual;
    const int nblk = p.c_out / 64;
    const uint32_t buf_s = smem_u32(buf);
    const uint32_t res_bytes = (uint32_t)p.c_out * kBlockM * 2u;
    uint32_t res_phase = 0;
    bool res_pending = false;  // issuer: a residual load is in flight

    auto issue_residual = [&](int u) {
        const TileInfo tn = tile_info(unit_tile(u, p) * kPair + (int)rank, p);
        if (tn.dummy) return;
        mbar_arrive_expect_tx(bars.resf(), res_bytes);
        for (int b = 0; b < nblk; ++b) {
            if (p.halo)
                tma_load_4d(buf_s + (uint32_t)b * (kBlockM * 128u), mapR, bars.resf(), b * 64,
                            tn.w0, tn.h0, tn.frame);
            else
                tma_load_3d(buf_s + (uint32_t)b * (kBlockM * 128u), mapR, bars.resf(), b * 64,
                            tn.pos, tn.frame);
        }
        res_pending = true;
    };
    if (issuer && resid && unit0 < num_units) issue_residual(unit0);

    int it = 0;
    for (int u = unit0; u < num_units; u += unit_stride, ++it) {
        const TileInfo ti = tile_info(unit_tile(u, p) * kPair + (int)rank, p);
        bool got = mbar_wait_warp<kPair == 2>(bars.accf(0), (uint32_t)it & 1u, wc);
        if (got && resid && !ti.dummy) {
            got = mbar_wait_warp<false>(bars.resf(), res_phase, wc);
            res_phase ^= 1u;
            if (issuer) res_pending = false;
        }
        if (bar_any(1, 32 * p.epi_warps, !got)) break;  // same decision in every epilogue warp
        tc_fence_after();
        const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16);
        uint8_t *rowp = buf + row * 128;  // row `row` of block 0
        const int sw = row & 7;
        const bool norm = p.epi == kEpiNormSilu;
        // Pass 1: TMEM -> acc + bias (+ residual) -> bf16 tile in `buf`.  For
        // the fused norm this stores h = acc + bias and sums h^2 in fp32.
        float ss = 0.f;
        for (int c = c_begin; c < c_end; c += 32) {
            uint32_t r[32];
            const int n = c_end - c >= 32 ? 32 : 16;
            tmem_ld_cols(tb + (uint32_t)c, n, r);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (8 * k < n) {
                    const int ch = c + 8 * k;  // first channel of this 16-byte piece
                    uint4 *dst = reinterpret_cast<uint4 *>(
                        rowp + (ch >> 6) * (kBlockM * 128) + ((((ch & 63) >> 3) ^ sw) << 4));
                    float v[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[8 * k + i]) + s_bias[ch + i];
                    if (norm) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) ss += v[i] * v[i];
                    } else if (resid) {
                        const uint4 x4 = *dst;
                        const uint32_t xs[4] = {x4.x, x4.y, x4.z, x4.w};
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            v[2 * i] += __uint_as_float(xs[i] << 16);
                            v[2 * i + 1] += __uint_as_float(xs[i] & 0xffff0000u);
                        }
                    }
                    *dst = make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]),
                                      pack_bf16x2(v[4], v[5]), pack_bf16x2(v[6], v[7]));
                }
            }
        }
        if (norm) s_part[half * kBlockM + row] = ss;
        tc_fence_before();
        asm volatile("bar.sync 1, %0;" ::"r"(32 * p.epi_warps) : "memory");
        if (lane == 0) {
            // TMEM read out: the MMA warp may start the next tile now.
            if (kPair == 2)
                mbar_arrive_remote(mapa_shared(bars.acce(0), 0));
            else
                mbar_arrive(bars.acce(0));
        }
        if (norm) {
            // Pass 2, overlapping the next tile's MMAs: a2 = SiLU(h / max(|h|, eps)
            // * sqrt(C) * gamma), in place in `buf`.
            const float scale =
                p.sqrt_c / fmaxf(sqrtf(s_part[row] + s_part[kBlockM + row]), p.eps);
            for (int ch = c_begin; ch < c_end; ch += 8) {
                uint4 *dst = reinterpret_cast<uint4 *>(
                    rowp + (ch >> 6) * (kBlockM * 128) + ((((ch & 63) >> 3) ^ sw) << 4));
                const uint4 h4 = *dst;
                const uint32_t hs[4] = {h4.x, h4.y, h4.z, h4.w};
                uint32_t o[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float z0 = __uint_as_float(hs[i] << 16) * scale * s_gamma[ch + 2 * i];
                    float z1 = __uint_as_float(hs[i] & 0xffff0000u) * scale * s_gamma[ch + 2 * i + 1];
                    z0 = __fdividef(z0, 1.0f + __expf(-z0));
                    z1 = __fdividef(z1, 1.0f + __expf(-z1));
                    o[i] = pack_bf16x2(z0, z1);
                }
                *dst = make_uint4(o[0], o[1], o[2], o[3]);
            }
        }
        fence_proxy_async_smem();  // the tile in `buf` is visible to the TMA stores below
        asm volatile("bar.sync 1, %0;" ::"r"(32 * p.epi_warps) : "memory");
        if (issuer) {
            // output frame: the tile's own, or for the temporal upsampler frame
            // 2t + a of the unit's phase a
            const int out_frame =
                p.up_t ? (ti.n * 2 * p.T + 2 * ti.t + unit_phase(u, p)) : ti.frame;
            if (!ti.dummy) {
                for (int b = 0; b < nblk; ++b) {
                    if (p.halo)
                        tma_store_4d(mapY, buf_s + (uint32_t)b * (kBlockM * 128u), b * 64, ti.w0,
                                     ti.h0, ti.frame);
                    else
                        tma_store_3d(mapY, buf_s + (uint32_t)b * (kBlockM * 128u), b * 64,
                                     ti.pos, out_frame);
                }
                bulk_commit();
            }
            // The buffer is reused only after the stores have read it.
            bulk_wait_read_all();
            if (resid && u + unit_stride < num_units) issue_residual(u + unit_stride);
        }
    }
    if (issuer) {
        bulk_wait_all();
        if (res_pending) {  // aborted with a residual load in flight: let it land
            volatile int no_abort = 0;
            const WaitCtl dc{kDrainNs, wc.err, &no_abort, kDevErrTimeout | kDevErrDrain};
            mbar_wait(bars.resf(), res_phase, dc);
        }
    }
}

// (kThreads = 12 warps, one CTA per SM: three warps share a sub-partition's
// 16K registers, so at most 168 registers a thread)
template <int kPair, int KK, int NSUB, int NP, bool kUp, bool kFuse = false>
__global__ void __launch_bounds__(kThreads, 1)
conv3d_tcgen05_kernel(const __grid_constant__ CUtensorMap mapA,
                      const __grid_constant__ CUtensorMap mapC,
                      const __grid_constant__ CUtensorMap mapB,
                      const __grid_constant__ CUtensorMap mapSA,
                      const __grid_constant__ CUtensorMap mapSB,
                      const __grid_constant__ CUtensorMap mapY,
                      const __grid_constant__ CUtensorMap mapR, const ConvArgs p) {
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Bars bars{sbase + p.off_bars, p.stages};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + p.off_misc);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + p.off_misc + 4);
    // the producers' last issued fills and done flags (conv_producer)
    volatile int *prod_state = reinterpret_cast<volatile int *>(smem + p.off_misc + 8);
    float *s_bias = reinterpret_cast<float *>(smem + p.off_vec);
    float *s_gamma = s_bias + p.c_out;
    float *s_part = s_gamma + p.c_out;  // [2 sub-tiles][2][128] partial sums of squares
    // output staging; 128-byte aligned where the upsampler's TMA stores read it
    // (the plan reserves the slack for that case only)
    const uintptr_t stg0 = reinterpret_cast<uintptr_t>(s_part + 4 * kBlockM);
    uint8_t *s_stage = reinterpret_cast<uint8_t *>(
        p.up_tma ? (stg0 + 127) & ~static_cast<uintptr_t>(127) : stg0);

    // Work units: single tiles, or pairs of consecutive tiles per cluster.
    const uint32_t rank = kPair == 2 ? cluster_ctarank() : 0u;
    const int unit0 = kPair == 2 ? (int)cluster_id_x() : (int)blockIdx.x;
    const int unit_stride = kPair == 2 ? (int)cluster_count_x() : (int)gridDim.x;
    const int num_units = p.tile_units * p.nphase;

    if (threadIdx.x == 0) {
        // every issuer's commit arrives on the barriers the MMAs release
        const uint32_t ni = (uint32_t)p.issuers;
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(bars.full(s), kFuse ? 2 : 1);  // (fused: the weights' and the halo's)
            mbar_init(bars.empty(s), ni);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bars.accf(a), ni);
            mbar_init(bars.acce(a), p.epi_warps * kPair);
        }
        mbar_init(bars.drain(), ni);
        mbar_init(bars.resf(), 1);
        for (int i = 0; i < 4; ++i) mbar_init(bars.emptya(i), ni);
        if (kFuse)
            for (int i = 0; i < 4; ++i) mbar_init(bars.peer(i), 1);
        *abort_flag = 0;
        prod_state[0] = prod_state[1] = -1;
        prod_state[2] = prod_state[3] = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&mapA);
        tma_prefetch_desc(&mapB);
        if (p.has_cache) tma_prefetch_desc(&mapC);
        if (p.kc_short) {
            tma_prefetch_desc(&mapSA);
            tma_prefetch_desc(&mapSB);
        }
        if (p.staged) {
            tma_prefetch_desc(&mapY);
            if (p.epi == kEpiResidual) tma_prefetch_desc(&mapR);
        }
    }
    if (warp == 1) {
        if (kPair == 2) {
            tmem_alloc_pair(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
            tmem_relinquish();
        }
    }
    griddep_wait();  // the previous kernel's outputs (and anything before it) are visible
    for (int i = threadIdx.x; i < p.c_out; i += kThreads) {
        float b = p.bias ? p.bias[i] : 0.f;
        if (p.bias2) b += p.bias2[i];
        s_bias[i] = b;
        s_gamma[i] = p.gamma ? p.gamma[i] : 1.f;
    }
    tc_fence_before();
    if (kPair == 2)
        cluster_sync_all();  // barriers of both CTAs initialised before any cross-CTA use
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtl wc{p.wait_ns, p.err, abort_flag, 0u};

    if (warp == 0 || warp == kProducer2Warp) {
        const int part = warp == 0 ? 0 : 1;
        if (lane == 0 && part < p.producers) {
            if (p.halo)
                conv_producer_halo<kPair, kUp, kFuse>(&mapA, &mapC, &mapB, &mapSA, &mapSB, p,
                                                      sbase, bars, wc, unit0, unit_stride,
                                                      num_units, rank, part, prod_state);
            else
                conv_producer<kPair, kUp>(&mapA, &mapC, &mapB, &mapSA, &mapSB, p, sbase, bars, wc,
                                          unit0, unit_stride, num_units, rank, part, prod_state);
        }
    } else if (warp == 1 || warp == kIssuer2Warp) {
        const int part = warp == 1 ? 0 : 1;
        if (lane == 0 && rank == 0 && part < p.issuers) {
            if (p.halo)
                conv_mma_halo<kPair, KK, NSUB, NP, kUp>(p, sbase, tmem_base, bars, wc, unit0,
                                                        unit_stride, num_units, part);
            else
                conv_mma<kPair, KK, NSUB, NP>(p, sbase, tmem_base, bars, wc, unit0, unit_stride,
                                              num_units, part);
        }
    } else if (kFuse && warp >= 2 + p.epi_warps) {
        conv_transform<kPair>(&mapA, &mapC, p, sbase, bars, wc, unit0, unit_stride, num_units,
                              rank);
    } else {
        if (p.staged)
            conv_epilogue_staged<kPair>(p, tmem_base, s_bias, s_gamma, s_part,
                                        smem + p.off_stage, &mapY, &mapR, bars, wc, unit0,
                                        unit_stride, num_units, rank);
        else
            conv_epilogue<kPair, kUp>(p, tmem_base, s_bias, s_gamma, s_part,
                                 s_stage + (threadIdx.x / 32 - 2) * p.stg_warp, &mapY,
                                 bars, wc, unit0, unit_stride, num_units, rank);
    }
    __syncwarp();
    tc_fence_before();
    if (kPair == 2)
        cluster_sync_all();  // no CTA leaves while its peer may still touch it
    else
        __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        if (kPair == 2)
            tmem_dealloc_pair(tmem_base, (uint32_t)p.tmem_cols);
        else
            tmem_dealloc(tmem_base, (uint32_t)p.tmem_cols);
    }
}


typedef void (*ConvKernelFn)(const CUtensorMap, const CUtensorMap, const CUtensorMap,
                             const CUtensorMap, const CUtensorMap, const CUtensorMap,
                             const CUtensorMap, const ConvArgs);

// The kernel for a plan (conv3d_kernels_misc.cu, from the translation units
// that instantiate it): unrolled MMA issue for every (k-steps per sub-tile
// kk, sub-tiles per stage nsub, N pieces np) the planner produces, run-time
// loops otherwise.  pair = 1 or 2 (CTA pairs); conv_kernel_up gives the
// upsamplers' instantiations.
ConvKernelFn conv_kernel_plain(int pair, int kk, int nsub, int np);
ConvKernelFn conv_kernel_up(int pair, int kk, int nsub, int np);
ConvKernelFn conv_kernel_fuse(int pair, int kk, int nsub, int np);

}  // namespace conv
}  // namespace wanvae
