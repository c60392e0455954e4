// conv3d_narrow.cu -- CausalConv3d k=3 for very narrow outputs (c_out <= 3:
// the decoder's conv_out from 96 channels to RGB, "Sharding of WAN 2.2 VAE",
// decoder tree).
//
// As an implicit GEMM with N = c_out, every MMA would carry 3 useful columns
// of at least 16 and the 27 shifted taps would need 27 MMAs per k-step: the
// issue rate, not the math, would bound it.  Instead the taps go into N:
//
//   Z_f[p, (o, kt, kh, kw)] = sum_c a_f[p, c] * W[o, kt, kh, kw, c]
//
// is one dense GEMM per input frame f over the halo pixels p of a 16 x 16
// patch (M = 18 x 18 = 324 pixels in three 128-row tiles, N = 27 c_out padded
// to 16, K = c_in), and the conv is the stencil sum
//
//   y_t[q, o] = b[o] + sum_{kt,kh,kw} Z_{t-2+kt}[q + (kh, kw), (o, kt, kh, kw)]
//
// over the three input frames that output frame t reads.  A CTA owns one
// patch and marches along T: each input frame is loaded once (one TMA halo
// box per 64- or 32-channel chunk, 128-/64-byte swizzled rows of one pixel
// each), multiplied once, and its Z adds into the three output frames it
// feeds (running sums in registers); an output frame is stored as soon as
// its last input frame (kt = 2) is in.  Frames before t = 0 are the causal
// zeros (skipped) or, with a feat_cache, the cache's two frames.
#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <string.h>

#include "kernels.h"
#include "ptx.cuh"

namespace wanvae {
namespace {

constexpr int kThreadsN = 256;           // 8 warps; thread q owns output pixel q of the patch
constexpr int kHalo = 18;                // halo width and height (16 x 16 patch + the 3x3 window)
constexpr int kHaloPx = kHalo * kHalo;   // 324 pixels = M rows (three 128-row MMA tiles)
constexpr int kHaloRows = 328;           // halo rows in smem: the third M tile (rows 200..327)
                                         // reads 4 slack rows past the 324 pixels
constexpr uint64_t kDrainNsN = 200ull * 1000 * 1000;

struct NarrowArgs {
    int B, T, H, W, c_in, c_out;
    int npad;               // MMA N: 27 c_out rounded up to 16
    int nch;                // channel chunks: 64 channels each, then a last one of 32
    int patches_w, patches_h, num_items;
    int has_cache;
    uint32_t off_a0, off_a1, off_b0, off_b1;  // per chunk (at most two): halo rows, B rows
    uint32_t off_z, off_bars;
    uint32_t b_tx;          // bytes of the whole B operand
    uint32_t halo_tx;       // bytes of one halo load
    const float *bias;
    __nv_bfloat16 *out;
    unsigned *err;
    uint64_t wait_ns;
};

// Bars: halo full, MMA done, weights loaded.
struct NBars {
    uint32_t base;
    __device__ uint32_t full() const { return base; }
    __device__ uint32_t mmad() const { return base + 8; }
    __device__ uint32_t wld() const { return base + 16; }
};

// First halo pixel of each 128-row M tile (the third overlaps the second so
// that it needs only 4 slack rows).
__device__ __forceinline__ int tile_row(int j) { return j == 0 ? 0 : (j == 1 ? 128 : 200); }

// Chunk k holds channels [64 k, 64 k + width): width 64 (128-B rows, 128-B
// swizzle) except a last chunk of 32 (64-B rows, 64-B swizzle).
__device__ __forceinline__ int chunk_w(const NarrowArgs &p, int k) {
    return (k == p.nch - 1 && p.c_in % 64) ? 32 : 64;
}

template <int CO>
__global__ void __launch_bounds__(kThreadsN, 1)
conv3d_narrow_kernel(const __grid_constant__ CUtensorMap mapX64,
                     const __grid_constant__ CUtensorMap mapX32,
                     const __grid_constant__ CUtensorMap mapC64,
                     const __grid_constant__ CUtensorMap mapC32,
                     const __grid_constant__ CUtensorMap mapW64,
                     const __grid_constant__ CUtensorMap mapW32, const NarrowArgs p) {
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const NBars bars{sbase + p.off_bars};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + p.off_bars + 32);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + p.off_bars + 36);
    float *zs = reinterpret_cast<float *>(smem + p.off_z);

    if (tid == 0) {
        mbar_init(bars.full(), 1);
        mbar_init(bars.mmad(), 1);
        mbar_init(bars.wld(), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mapX64);
        tma_prefetch_desc(&mapX32);
        tma_prefetch_desc(&mapW64);
        tma_prefetch_desc(&mapW32);
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{p.wait_ns, p.err, abort_flag, 0u};
    griddep_wait();  // the previous kernel's outputs are visible from here on

    // The whole B operand (27 c_out rows, rows up to npad read as zeros) once.
    if (tid == 0) {
        mbar_arrive_expect_tx(bars.wld(), p.b_tx);
        for (int k = 0; k < p.nch; ++k)
            tma_load_2d(sbase + (k == 0 ? p.off_b0 : p.off_b1), chunk_w(p, k) == 64 ? &mapW64 : &mapW32, bars.wld(),
                        64 * k, 0);
    }
    bool ok = mbar_wait_warp(bars.wld(), 0u, wc);
    ok = !bar_any(1, kThreadsN, !ok);

    const uint32_t idesc = idesc_bf16_f32(128, p.npad);
    const int qh = tid >> 4, qw = tid & 15;       // this thread's output pixel in the patch
    const int qd = warp & 3, jw = warp >> 2;       // TMEM lane quarter; first M tile copied
    const int f0 = p.has_cache ? -2 : 0;
    uint32_t ph_full = 0, ph_mma = 0;
    int pending_full = 0;                          // halo loads issued but not waited for
    int pending_mma = 0;                           // MMAs committed but not waited for
    int lost_full = -1;  // thread 0: phase of a halo load whose wait gave up (still in flight)

    // halo of frame f (f < 0: cache frame f + 2): one box of 18 x 18 pixels per
    // channel chunk, one swizzled row per pixel (out-of-frame pixels: zeros)
    auto load_halo = [&](int b, int f, int h0, int w0) {
        mbar_arrive_expect_tx(bars.full(), p.halo_tx);
        const int frame = f < 0 ? b * 2 + f + 2 : b * p.T + f;
        for (int k = 0; k < p.nch; ++k) {
            const bool w64 = chunk_w(p, k) == 64;
            const CUtensorMap *m = f < 0 ? (w64 ? &mapC64 : &mapC32) : (w64 ? &mapX64 : &mapX32);
            tma_load_4d(sbase + (k == 0 ? p.off_a0 : p.off_a1), m, bars.full(), 64 * k, w0 - 1, h0 - 1, frame);
        }
    };

    constexpr int kZS = (27 * CO) | 1;  // floats per halo pixel of Z in smem (odd: conflict-free)
    // Z of one input frame, all c_out x 27 columns of every halo pixel:
    // TMEM -> shared memory, so TMEM is free for the next frame's MMAs.
    auto copy_z = [&]() {
        for (int j = jw; j < 3; j += 2) {
            const int px = tile_row(j) + qd * 32 + lane;
            const bool mine = px < kHaloPx && (j < 2 || px >= 256);  // tile 2 overlaps tile 1
#pragma unroll
            for (int c0 = 0; c0 < 27 * CO; c0 += 32) {
                uint32_t r[32];
                tmem_ld_cols(tmem + ((uint32_t)(qd * 32) << 16) + (uint32_t)(j * p.npad + c0), 32,
                             r);
                if (mine) {
#pragma unroll
                    for (int c = 0; c < 32; ++c)
                        if (c0 + c < 27 * CO) zs[px * kZS + c0 + c] = __uint_as_float(r[c]);
                }
            }
        }
    };
    auto issue_mma = [&]() {
        // Z_f for the three 128-row tiles of the halo (rows = consecutive halo
        // pixels), K in 16-channel steps of 32 bytes through each chunk.
        for (int j = 0; j < 3; ++j) {
            for (int k = 0; k < p.nch; ++k) {
                const int cw = chunk_w(p, k);
                const uint32_t rowb = (uint32_t)cw * 2u, lay = cw == 64 ? kLayoutSw128 : kLayoutSw64;
                const uint64_t a0 =
                    sdesc_kmajor(sbase + (k == 0 ? p.off_a0 : p.off_a1) + (uint32_t)tile_row(j) * rowb, rowb, lay);
                const uint64_t b0 = sdesc_kmajor(sbase + (k == 0 ? p.off_b0 : p.off_b1), rowb, lay);
                for (int ks = 0; ks < cw / 16; ++ks)
                    mma_bf16_ss(tmem + (uint32_t)(j * p.npad), a0 + (uint64_t)(2 * ks),
                                b0 + (uint64_t)(2 * ks), idesc, (k > 0 || ks > 0) ? 1u : 0u);
            }
        }
        mma_commit(bars.mmad());
    };

    for (int item = blockIdx.x; ok && item < p.num_items; item += gridDim.x) {
        const int per_clip = p.patches_h * p.patches_w;
        const int b = item / per_clip, pr = item - b * per_clip;
        const int h0 = (pr / p.patches_w) * 16, w0 = (pr % p.patches_w) * 16;
        float cur[CO], nxt[CO], nx2[CO];  // output frames f, f+1, f+2
#pragma unroll
        for (int o = 0; o < CO; ++o) cur[o] = nxt[o] = nx2[o] = 0.f;
        // Prologue: Z of the first input frame into shared memory.
        if (tid == 0) load_halo(b, f0, h0, w0);
        pending_full = 1;
        ok = mbar_wait_warp(bars.full(), ph_full, wc);
        if (bar_any(1, kThreadsN, !ok)) {
            ok = false;
            break;
        }
        ph_full ^= 1u;
        pending_full = 0;
        tc_fence_after();
        if (tid == 0) issue_mma();
        pending_mma = 1;
        ok = mbar_wait_warp(bars.mmad(), ph_mma, wc);
        if (bar_any(1, kThreadsN, !ok)) {
            ok = false;
            break;
        }
        ph_mma ^= 1u;
        pending_mma = 0;
        tc_fence_after();
        if (tid == 0 && f0 + 1 < p.T) load_halo(b, f0 + 1, h0, w0);
        pending_full = f0 + 1 < p.T ? 1 : 0;
        copy_z();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        for (int f = f0; f < p.T; ++f) {
            const bool next = f + 1 < p.T;
            // Frame f+1's MMAs run on the tensor core while frame f's stencil
            // sums run on the CUDA cores (TMEM was emptied into smem).
            if (next && tid == 0) {
                if (mbar_wait(bars.full(), ph_full, wc)) {
                    tc_fence_after();
                    issue_mma();
                } else {
                    lost_full = (int)ph_full;  // the abort flag is up: the wait below gives up
                }
            }
            // the 3x3 spatial stencil of Z_f for each temporal tap and channel
            const float *zq = zs + (qh * kHalo + qw) * kZS;
#pragma unroll
            for (int o = 0; o < CO; ++o) {
                float s0 = 0.f, s1 = 0.f, s2 = 0.f;
#pragma unroll
                for (int kh = 0; kh < 3; ++kh)
#pragma unroll
                    for (int kw = 0; kw < 3; ++kw) {
                        const float *z = zq + (kh * kHalo + kw) * kZS + o * 27 + kh * 3 + kw;
                        s0 += z[0];   // kt = 0: output frame f + 2
                        s1 += z[9];   // kt = 1: output frame f + 1
                        s2 += z[18];  // kt = 2: output frame f
                    }
                cur[o] += s2;
                nxt[o] += s1;
                nx2[o] += s0;
            }
            if (f >= 0) {
                const int h = h0 + qh, w = w0 + qw;
                if (h < p.H && w < p.W) {
                    __nv_bfloat16 *y =
                        p.out + ((((int64_t)b * p.T + f) * p.H + h) * p.W + w) * CO;
#pragma unroll
                    for (int o = 0; o < CO; ++o)
                        y[o] = __float2bfloat16_rn(cur[o] + (p.bias ? p.bias[o] : 0.f));
                }
            }
#pragma unroll
            for (int o = 0; o < CO; ++o) {
                cur[o] = nxt[o];
                nxt[o] = nx2[o];
                nx2[o] = 0.f;
            }
            if (!next) break;
            ph_full ^= 1u;  // frame f+1's halo was consumed by its MMAs
            pending_full = 0;
            pending_mma = lost_full < 0 ? 1 : 0;
            ok = mbar_wait_warp(bars.mmad(), ph_mma, wc);
            // (the reduction is also the barrier that ends every read of Z_f)
            if (bar_any(1, kThreadsN, !ok)) {
                ok = false;
                break;
            }
            ph_mma ^= 1u;
            pending_mma = 0;
            tc_fence_after();
            if (tid == 0 && f + 2 < p.T) load_halo(b, f + 2, h0, w0);
            pending_full = f + 2 < p.T ? 1 : 0;
            copy_z();
            tc_fence_before();
            __syncthreads();
            tc_fence_after();
        }
    }
    // Aborted: let a halo load in flight land and committed MMAs finish before
    // the CTA's shared memory and TMEM go away.
    if (!ok && tid == 0) {
        volatile int no_abort = 0;
        const WaitCtl dc{kDrainNsN, p.err, &no_abort, kDevErrTimeout | kDevErrDrain};
        if (pending_full) mbar_wait(bars.full(), ph_full, dc);
        if (lost_full >= 0) mbar_wait(bars.full(), (uint32_t)lost_full, dc);
        if (pending_mma) mbar_wait(bars.mmad(), ph_mma, dc);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 512);
}

// The dynamic shared-memory opt-in of each instantiation, made once per
// device (it does not change between launches).
template <int CO>
cudaError_t launch_narrow(const NarrowArgs &a, const CUtensorMap *m, uint32_t smem,
                          const LaunchCtx &ctx) {
    auto kern = conv3d_narrow_kernel<CO>;
    constexpr int kMaxDev = 64;
    static std::atomic<uint32_t> opted[kMaxDev];  // bytes opted in per device (0 = not yet)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    if (opted[dev].load(std::memory_order_acquire) < smem) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        opted[dev].store(smem, std::memory_order_release);
    }
    const int grid = a.num_items < ctx.num_sms ? a.num_items : ctx.num_sms;
    return launch_pdl(kern, dim3((unsigned)grid), dim3(kThreadsN), smem, ctx, m[0], m[1], m[2],
                      m[3], m[4], m[5], a);
}

// The kernel-variant setting (set_kernel_variant) can route narrow layers to
// the implicit-GEMM kernel instead.
bool narrow_enabled() { return narrow_variant() != 0; }

}  // namespace

int conv3d_narrow_supported(const ConvSpec &s) {
    if (!narrow_enabled()) return -1;
    if (s.k != 3 || s.c_out < 1 || s.c_out > 3 || s.sc_in || s.epi != kEpiBias) return -1;
    if (s.up2d || s.up_t) return -1;  // plain convs only
    if (s.c_in < 32 || s.c_in % 32 || s.c_in > 128) return -1;
    return 0;
}

cudaError_t launch_conv3d_narrow(const ConvSpec &s, const LaunchCtx &ctx) {
    NarrowArgs a;
    memset(&a, 0, sizeof(a));
    a.B = s.B;
    a.T = s.T;
    a.H = s.H;
    a.W = s.W;
    a.c_in = s.c_in;
    a.c_out = s.c_out;
    a.npad = (27 * s.c_out + 15) / 16 * 16;
    a.nch = (s.c_in + 63) / 64;
    a.patches_w = (s.W + 15) / 16;
    a.patches_h = (s.H + 15) / 16;
    a.num_items = s.B * a.patches_w * a.patches_h;
    a.has_cache = s.cache != nullptr;
    // Shared memory per chunk: 328 halo rows and npad B rows of the chunk's
    // width (1024-aligned: the swizzle atoms), then Z and the barriers.
    uint32_t off = 0;
    for (int k = 0; k < a.nch; ++k) {
        const uint32_t rowb = (k == a.nch - 1 && s.c_in % 64) ? 64u : 128u;
        (k == 0 ? a.off_a0 : a.off_a1) = off;
        off += ((uint32_t)kHaloRows * rowb + 1023u) & ~1023u;
    }
    for (int k = 0; k < a.nch; ++k) {
        const uint32_t rowb = (k == a.nch - 1 && s.c_in % 64) ? 64u : 128u;
        (k == 0 ? a.off_b0 : a.off_b1) = off;
        off += ((uint32_t)a.npad * rowb + 1023u) & ~1023u;
    }
    a.halo_tx = (uint32_t)kHaloPx * (uint32_t)s.c_in * 2u;
    a.b_tx = (uint32_t)a.npad * (uint32_t)s.c_in * 2u;
    a.off_z = off;
    const uint32_t zs_floats = (uint32_t)((27 * s.c_out) | 1);
    a.off_bars = (a.off_z + (uint32_t)kHaloPx * zs_floats * 4u + 15u) & ~15u;
    uint32_t smem = 1024u + a.off_bars + 64u;
    if (smem < 120u * 1024u) smem = 120u * 1024u;  // one CTA per SM (it holds 512 TMEM columns)
    a.bias = s.bias;
    a.out = static_cast<__nv_bfloat16 *>(s.out);
    a.err = ctx.err;
    a.wait_ns = ctx.wait_ns;

    // NHWC input as (C, W, H, frames); boxes of 64 or 32 channels x 18 x 18
    // pixels land as one swizzled row per pixel.  Weights [c_out][27][c_in] =
    // a [27 c_out][c_in] K-major matrix; boxes of npad rows (rows past 27 c_out
    // read as zeros).  Maps: X64, X32, C64, C32, W64, W32 (unused ones repeat
    // a valid one).
    const int frames = s.B * s.T;
    CUtensorMap m[6];
    memset(m, 0, sizeof(m));
    cuuint64_t dx[4] = {(cuuint64_t)s.c_in, (cuuint64_t)s.W, (cuuint64_t)s.H, (cuuint64_t)frames};
    cuuint64_t sx[3] = {(cuuint64_t)s.c_in * 2, (cuuint64_t)s.W * s.c_in * 2,
                        (cuuint64_t)s.H * s.W * s.c_in * 2};
    cuuint64_t dw[2] = {(cuuint64_t)s.c_in, (cuuint64_t)(27 * s.c_out)};
    cuuint64_t sw[1] = {(cuuint64_t)s.c_in * 2};
    bool ok = true;
    for (int w = 0; w < 2; ++w) {
        const uint32_t cw = w == 0 ? 64u : 32u;
        if ((w == 0 && s.c_in < 64) || (w == 1 && s.c_in % 64 == 0)) continue;
        cuuint32_t bx[4] = {cw, kHalo, kHalo, 1};
        ok = ok && encode_tiled_bf16(&m[w], 4, s.in, dx, sx, bx, (int)cw * 2);
        if (s.cache) {
            cuuint64_t dc[4] = {dx[0], dx[1], dx[2], (cuuint64_t)s.B * 2};
            ok = ok && encode_tiled_bf16(&m[2 + w], 4, s.cache, dc, sx, bx, (int)cw * 2);
        }
        cuuint32_t bw[2] = {cw, (cuuint32_t)a.npad};
        ok = ok && encode_tiled_bf16(&m[4 + w], 2, s.w, dw, sw, bw, (int)cw * 2);
    }
    if (!ok) return cudaErrorInvalidValue;
    const int have = s.c_in >= 64 ? 0 : 1;  // a map that exists, for the unused slots
    for (int w = 0; w < 2; ++w) {
        if ((w == 0 && s.c_in < 64) || (w == 1 && s.c_in % 64 == 0)) {
            m[w] = m[have];
            m[4 + w] = m[4 + have];
        }
        if (!s.cache) m[2 + w] = m[w];
        else if ((w == 0 && s.c_in < 64) || (w == 1 && s.c_in % 64 == 0)) m[2 + w] = m[2 + have];
    }
    switch (s.c_out) {
        case 1: return launch_narrow<1>(a, m, smem, ctx);
        case 2: return launch_narrow<2>(a, m, smem, ctx);
        case 3: return launch_narrow<3>(a, m, smem, ctx);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace wanvae
