// attn_tcgen05.cu -- the mid-block's spatial self-attention core on tcgen05:
// O = softmax(Q K^T / sqrt(D)) V per frame, one head of width D.
//
// "Closing the gap: Wan 2.2 14B VAE decoder", section 5: the decoder's one
// attention block lets every position of a frame attend to every other; the
// sequence is the frame's H x W grid and each (batch, frame) is an
// independent problem.  The projections around this core (RMS_norm, 1x1
// q/k/v, 1x1 output with the residual) run on the conv kernel.
//
// One CTA owns a tile of 128 queries of one frame and sweeps the frame's keys
// in blocks of 128 (a flash-style pass: the scores never reach memory):
//   S = Q K_j^T           (tcgen05, S in TMEM columns [0, 128))
//   P = exp2(S' - m)      (4 softmax warps, one query row per thread; P in
//                          shared memory as the next MMA's A operand)
//   O += P V_j            (tcgen05, O in TMEM columns [128, 128 + D))
// The running max m moves only when a block's max exceeds it by more than
// 2^8 (then O and the row sum are rescaled), so P stays <= 256 and the rescale
// is rare.  Q stays in shared memory for the tile; K and V^T stream through a
// 3-stage ring of 32 KB stages (128 keys x 128 dims).  S_{j+1} is issued as
// soon as the softmax warps have read S_j, so it overlaps their exponentials;
// P_j waits for PV_{j-1} to finish reading the P buffer.
//
// Warp roles: warp 0 = TMA producer (one thread), warp 1 = TMEM allocation and
// the MMA issuer (one thread), warps 2-5 = softmax and epilogue (warp w reads
// TMEM lane quarter w % 4).  Every wait is bounded; on expiry the kernel raises
// the device error bit, drains its copies and MMAs, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <math.h>
#include <string.h>

#include <atomic>

#include "kernels.h"
#include "ptx.cuh"

namespace wanvae {
namespace {

constexpr int kAThreads = 192;
constexpr int kBlk = 128;                 // queries per tile, keys per block
constexpr int kAStages = 3;
constexpr uint32_t kAtom = 128u * 128u;   // one swizzled atom column: 128 rows x 64 bf16
constexpr uint32_t kStage = 2u * kAtom;   // 128 rows x 128 bf16
constexpr uint64_t kADrainNs = 200ull * 1000 * 1000;

struct AttnArgs {
    int F, N, D;          // frames, positions per frame, head width (128, 256 or 384)
    int q_tiles, nkb;     // 128-query tiles and 128-key blocks per frame
    float scale_log2;     // log2(e) / sqrt(D)
    uint32_t off_p, off_ring, off_bars;
    __nv_bfloat16 *out;   // [F][N][D]
    unsigned *err;
    uint64_t wait_ns;
};

struct ABars {
    uint32_t base;
    __device__ uint32_t full(int s) const { return base + 8u * s; }
    __device__ uint32_t empty(int s) const { return base + 8u * (kAStages + s); }
    __device__ uint32_t q_full() const { return base + 8u * (2 * kAStages); }
    __device__ uint32_t q_empty() const { return base + 8u * (2 * kAStages + 1); }
    __device__ uint32_t s_full() const { return base + 8u * (2 * kAStages + 2); }
    __device__ uint32_t s_free() const { return base + 8u * (2 * kAStages + 3); }
    __device__ uint32_t p_full() const { return base + 8u * (2 * kAStages + 4); }
    __device__ uint32_t o_done() const { return base + 8u * (2 * kAStages + 5); }
    __device__ uint32_t o_free() const { return base + 8u * (2 * kAStages + 6); }
    __device__ uint32_t drain() const { return base + 8u * (2 * kAStages + 7); }
};
constexpr int kANumBars = 2 * kAStages + 8;

// 32 columns of this warp's TMEM lane quarter <- r (then wait for the store).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Byte offset of element (row r, k) in a K-major operand stored as 128-byte
// swizzled atom columns of 64 bf16 (the layout TMA's 128-byte swizzle writes
// into a 1024-byte aligned buffer): the 16-byte chunk index is XORed with
// the row's position in its 8-row group.
__device__ __forceinline__ uint32_t sw128_off(int r, int k) {
    return (uint32_t)(k >> 6) * kAtom + (uint32_t)r * 128u +
           ((uint32_t)(((k & 63) >> 3) ^ (r & 7)) << 4) + (uint32_t)(k & 7) * 2u;
}

// TMA producer (one thread).  Per tile: Q (D / 64 boxes of 64 dims x 128
// queries) on q_full, then K and V^T blocks through the ring in the order the
// issuer consumes them: S_0, then S_{j+1} and PV_j for every block j.
__device__ void attn_producer(const CUtensorMap *mQ, const CUtensorMap *mK,
                              const CUtensorMap *mVt, const AttnArgs &p, uint32_t sbase,
                              const ABars &bars, const WaitCtl &wc, int item0, int istride,
                              int items) {
    const int nd = p.D / 64, nc = p.D / 128;
    int stage = 0, it = 0;
    uint32_t phase = 0, fills = 0, qloads = 0;
    bool ok = true;
    auto next = [&](uint32_t &dst, uint32_t &fb) -> bool {
        if (!mbar_wait<false>(bars.empty(stage), phase ^ 1u, wc)) return false;
        fb = bars.full(stage);
        mbar_arrive_expect_tx(fb, kStage);
        dst = sbase + p.off_ring + (uint32_t)stage * kStage;
        ++fills;
        if (++stage == kAStages) {
            stage = 0;
            phase ^= 1u;
        }
        return true;
    };
    // 128 keys x 128 dims of K (dims c*128 ..) or of V^T (the same keys, as
    // rows of 128 dims), each as two 64-wide swizzled boxes
    auto load_k = [&](int f, int j) -> bool {
        for (int c = 0; c < nc; ++c) {
            uint32_t dst, fb;
            if (!next(dst, fb)) return false;
            for (int h = 0; h < 2; ++h)
                tma_load_3d(dst + (uint32_t)h * kAtom, mK, fb, c * 128 + h * 64, j * kBlk, f);
        }
        return true;
    };
    auto load_v = [&](int f, int j) -> bool {
        for (int c = 0; c < nc; ++c) {
            uint32_t dst, fb;
            if (!next(dst, fb)) return false;
            for (int h = 0; h < 2; ++h)
                tma_load_3d(dst + (uint32_t)h * kAtom, mVt, fb, j * kBlk + h * 64, c * 128, f);
        }
        return true;
    };
    for (int item = item0; ok && item < items; item += istride, ++it) {
        const int f = item / p.q_tiles, qt = item % p.q_tiles;
        if (!mbar_wait<false>(bars.q_empty(), ((uint32_t)it & 1u) ^ 1u, wc)) {
            ok = false;
            break;
        }
        mbar_arrive_expect_tx(bars.q_full(), (uint32_t)nd * kAtom);
        for (int a = 0; a < nd; ++a)
            tma_load_3d(sbase + (uint32_t)a * kAtom, mQ, bars.q_full(), a * 64, qt * kBlk, f);
        ++qloads;
        ok = load_k(f, 0);
        for (int j = 0; ok && j < p.nkb; ++j) {
            if (j + 1 < p.nkb) ok = load_k(f, j + 1);
            if (ok) ok = load_v(f, j);
        }
    }
    if (!ok) {
        // Aborted: let every copy in flight land before shared memory goes away.
        volatile int no_abort = 0;
        const WaitCtl dc{kADrainNs, wc.err, &no_abort, kDevErrTimeout | kDevErrDrain};
        const uint32_t n = fills < (uint32_t)kAStages ? fills : (uint32_t)kAStages;
        for (uint32_t f = fills - n; f < fills; ++f)
            mbar_wait<false>(bars.full((int)(f % kAStages)), (f / kAStages) & 1u, dc);
        if (qloads) mbar_wait<false>(bars.q_full(), (qloads - 1) & 1u, dc);
    }
}

// MMA issuer (one thread).  Descriptors are the buffers' bases plus constant
// offsets (k-step kk of a 128-wide chunk: atom column kk / 4, 32 bytes x
// (kk % 4) into it), so nothing but the stage bookkeeping sits between MMAs.
__device__ void attn_mma(const AttnArgs &p, uint32_t sbase, uint32_t tmem, const ABars &bars,
                         const WaitCtl &wc, int item0, int istride, int items) {
    const uint32_t idesc = idesc_bf16_f32(128, 128);
    const int nc = p.D / 128;
    const uint64_t q0 = sdesc_kmajor(sbase, 128u, kLayoutSw128);
    const uint64_t p0 = sdesc_kmajor(sbase + p.off_p, 128u, kLayoutSw128);
    const uint64_t r0 = sdesc_kmajor(sbase + p.off_ring, 128u, kLayoutSw128);
    const uint32_t atom16 = kAtom >> 4, stage16 = kStage >> 4;
    int stage = 0, it = 0;
    uint32_t phase = 0, gs = 0, gp = 0;  // ring position; S and PV blocks issued so far
    bool ok = true;
    auto acquire = [&]() -> bool {
        if (!mbar_wait<false>(bars.full(stage), phase, wc)) return false;
        tc_fence_after();
        return true;
    };
    auto release = [&]() {
        mma_commit(bars.empty(stage));
        if (++stage == kAStages) {
            stage = 0;
            phase ^= 1u;
        }
    };
    // S = Q K_j^T, once the softmax warps have read the previous S
    auto issue_s = [&]() -> bool {
        if (gs > 0 && !mbar_wait<false>(bars.s_free(), (gs - 1) & 1u, wc)) return false;
        tc_fence_after();
        for (int c = 0; c < nc; ++c) {
            if (!acquire()) return false;
            const uint64_t b = r0 + (uint64_t)((uint32_t)stage * stage16);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad =
                    q0 + (uint64_t)((uint32_t)(2 * c + (kk >> 2)) * atom16 + (kk & 3) * 2);
                const uint64_t bd = b + (uint64_t)((uint32_t)(kk >> 2) * atom16 + (kk & 3) * 2);
                mma_bf16_ss(tmem, ad, bd, idesc, (c == 0 && kk == 0) ? 0u : 1u);
            }
            release();
        }
        mma_commit(bars.s_full());
        ++gs;
        return true;
    };
    // O[:, c*128 ..] += P V_j[:, c*128 ..], once P_j is in shared memory
    auto issue_pv = [&](bool first) -> bool {
        if (!mbar_wait<false>(bars.p_full(), gp & 1u, wc)) return false;
        tc_fence_after();
        for (int c = 0; c < nc; ++c) {
            if (!acquire()) return false;
            const uint64_t b = r0 + (uint64_t)((uint32_t)stage * stage16);
            const uint32_t d = tmem + 128u + (uint32_t)(c * 128);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t ad = p0 + (uint64_t)((uint32_t)(kk >> 2) * atom16 + (kk & 3) * 2);
                const uint64_t bd = b + (uint64_t)((uint32_t)(kk >> 2) * atom16 + (kk & 3) * 2);
                mma_bf16_ss(d, ad, bd, idesc, (first && kk == 0) ? 0u : 1u);
            }
            release();
        }
        mma_commit(bars.o_done());
        ++gp;
        return true;
    };
    for (int item = item0; ok && item < items; item += istride, ++it) {
        if (!mbar_wait<false>(bars.q_full(), (uint32_t)it & 1u, wc)) break;
        tc_fence_after();
        ok = issue_s();
        for (int j = 0; ok && j < p.nkb; ++j) {
            if (j + 1 < p.nkb) ok = issue_s();
            // the previous tile's epilogue must have read O before PV_0 overwrites it
            if (ok && j == 0 && it > 0)
                ok = mbar_wait<false>(bars.o_free(), (uint32_t)(it - 1) & 1u, wc);
            if (ok) ok = issue_pv(j == 0);
        }
        if (ok) mma_commit(bars.q_empty());  // Q is free once the tile's MMAs are done
    }
    // Every MMA issued above completes before TMEM is released.
    volatile int no_abort = 0;
    const WaitCtl dc{kADrainNs, wc.err, &no_abort, kDevErrTimeout | kDevErrDrain};
    mma_commit(bars.drain());
    mbar_wait<false>(bars.drain(), 0u, dc);
}

// Softmax and epilogue warps (warps 2-5, one query row per thread: row
// (warp % 4) * 32 + lane, the TMEM lane quarter the warp may access).  The
// decisions that steer warp-collective TMEM accesses are made warp-uniform.
__device__ void attn_softmax(const AttnArgs &p, uint8_t *pbuf, uint32_t tmem, const ABars &bars,
                             const WaitCtl &wc, int item0, int istride, int items) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int qd = warp & 3;
    const int row = qd * 32 + lane;
    const uint32_t trow = tmem + ((uint32_t)(qd * 32) << 16);
    uint32_t gs = 0, gp = 0;  // S blocks read and P blocks written so far
    int it = 0;
    bool ok = true;
    for (int item = item0; ok && item < items; item += istride, ++it) {
        const int f = item / p.q_tiles, qt = item % p.q_tiles;
        float m = -INFINITY, l = 0.f;
        for (int j = 0; ok && j < p.nkb; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait_warp<false>(bars.s_full(), gs & 1u, wc));
            if (!ok) break;
            tc_fence_after();
            float s[kBlk];
#pragma unroll
            for (int c0 = 0; c0 < kBlk; c0 += 32) {
                uint32_t r[32];
                tmem_ld_cols(trow + (uint32_t)c0, 32, r);
#pragma unroll
                for (int i = 0; i < 32; ++i) s[c0 + i] = __uint_as_float(r[i]);
            }
            tc_fence_before();
            mbar_arrive(bars.s_free());  // S may be overwritten by the next block's MMAs
            ++gs;
            // scores in log2 units; keys past the frame's end do not exist
            const int kvalid = p.N - j * kBlk;
            float mx = -INFINITY;
#pragma unroll
            for (int c = 0; c < kBlk; ++c) {
                s[c] = c < kvalid ? s[c] * p.scale_log2 : -INFINITY;
                mx = fmaxf(mx, s[c]);
            }
            float factor = 1.f;
            if (mx > m + 8.f) {  // the running max moves only by more than 2^8
                if (m != -INFINITY) factor = exp2f(m - mx);
                m = mx;
            }
            float sum = 0.f;
            uint32_t pk[kBlk / 2];
#pragma unroll
            for (int c = 0; c < kBlk; c += 2) {
                const float a = exp2f(s[c] - m), b = exp2f(s[c + 1] - m);
                sum += a + b;
                pk[c / 2] = pack2(a, b);
            }
            l = l * factor + sum;
            // P's buffer and O are free once PV of the previous block is done
            if (gp > 0) {
                ok = __all_sync(0xffffffffu,
                                mbar_wait_warp<false>(bars.o_done(), (gp - 1) & 1u, wc));
                if (!ok) break;
            }
            tc_fence_after();
            if (__any_sync(0xffffffffu, factor != 1.f)) {
                for (int c0 = 0; c0 < p.D; c0 += 32) {
                    uint32_t r[32];
                    tmem_ld_cols(trow + 128u + (uint32_t)c0, 32, r);
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        r[i] = __float_as_uint(__uint_as_float(r[i]) * factor);
                    tmem_st32(trow + 128u + (uint32_t)c0, r);
                }
            }
#pragma unroll
            for (int ch = 0; ch < kBlk / 8; ++ch)
                *reinterpret_cast<uint4 *>(pbuf + sw128_off(row, ch * 8)) =
                    make_uint4(pk[4 * ch], pk[4 * ch + 1], pk[4 * ch + 2], pk[4 * ch + 3]);
            fence_proxy_async_smem();  // P is read by the tensor core (async proxy)
            tc_fence_before();
            mbar_arrive(bars.p_full());
            ++gp;
        }
        if (!ok) break;
        // epilogue: O / l of this row -> bf16, then O is free for the next tile
        ok = __all_sync(0xffffffffu, mbar_wait_warp<false>(bars.o_done(), (gp - 1) & 1u, wc));
        if (!ok) break;
        tc_fence_after();
        const float inv = 1.f / l;
        const int q = qt * kBlk + row;
        __nv_bfloat16 *dst = p.out + ((int64_t)f * p.N + q) * p.D;
        for (int c0 = 0; c0 < p.D; c0 += 32) {
            uint32_t r[32];
            tmem_ld_cols(trow + 128u + (uint32_t)c0, 32, r);
            if (q < p.N) {
                uint4 *d = reinterpret_cast<uint4 *>(dst + c0);
#pragma unroll
                for (int v = 0; v < 4; ++v)
                    d[v] = make_uint4(
                        pack2(__uint_as_float(r[8 * v]) * inv, __uint_as_float(r[8 * v + 1]) * inv),
                        pack2(__uint_as_float(r[8 * v + 2]) * inv,
                              __uint_as_float(r[8 * v + 3]) * inv),
                        pack2(__uint_as_float(r[8 * v + 4]) * inv,
                              __uint_as_float(r[8 * v + 5]) * inv),
                        pack2(__uint_as_float(r[8 * v + 6]) * inv,
                              __uint_as_float(r[8 * v + 7]) * inv));
            }
        }
        tc_fence_before();
        mbar_arrive(bars.o_free());
    }
}

__global__ void __launch_bounds__(kAThreads, 1)
attn_tcgen05_kernel(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mVt, const AttnArgs p) {
    griddep_launch_dependents();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const ABars bars{sbase + p.off_bars};
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + p.off_bars + 8 * kANumBars);
    volatile int *abort_flag =
        reinterpret_cast<volatile int *>(smem + p.off_bars + 8 * kANumBars + 4);
    if (threadIdx.x == 0) {
        for (int s = 0; s < kAStages; ++s) {
            mbar_init(bars.full(s), 1);
            mbar_init(bars.empty(s), 1);
        }
        mbar_init(bars.q_full(), 1);
        mbar_init(bars.q_empty(), 1);
        mbar_init(bars.s_full(), 1);
        mbar_init(bars.s_free(), 128);
        mbar_init(bars.p_full(), 128);
        mbar_init(bars.o_done(), 1);
        mbar_init(bars.o_free(), 128);
        mbar_init(bars.drain(), 1);
        *abort_flag = 0;
        fence_mbar_init();
        tma_prefetch_desc(&mQ);
        tma_prefetch_desc(&mK);
        tma_prefetch_desc(&mVt);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512u);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const WaitCtl wc{p.wait_ns, p.err, abort_flag, 0u};
    griddep_wait();  // q, k and V^T written by the previous kernels are visible
    const int items = p.F * p.q_tiles;
    if (warp == 0) {
        if (lane == 0)
            attn_producer(&mQ, &mK, &mVt, p, sbase, bars, wc, blockIdx.x, gridDim.x, items);
    } else if (warp == 1) {
        if (lane == 0) attn_mma(p, sbase, tmem, bars, wc, blockIdx.x, gridDim.x, items);
    } else {
        attn_softmax(p, smem + p.off_p, tmem, bars, wc, blockIdx.x, gridDim.x, items);
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512u);
}

// v [F][N][D] -> vt [F][D][ldn] (ldn >= N, a multiple of 8 so that rows
// start on 16 bytes): V as the K-major B operand of O += P V, keys along K.
// A CTA moves a 64 (positions) x 64 (dims) tile: 16-byte loads of 8 dims of
// a position into shared memory, then 16-byte stores of 8 positions of a dim
// (gathered from the tile's column).  Positions past N are not written.
constexpr int kTp = 64;
__global__ void __launch_bounds__(256)
transpose_v_kernel(const __nv_bfloat16 *__restrict__ v, __nv_bfloat16 *__restrict__ vt, int N,
                   int D, int ldn) {
    griddep_launch_dependents();
    griddep_wait();
    __shared__ uint16_t tile[kTp][kTp + 2];  // [position][dim], padded rows
    const int f = blockIdx.z;
    const int n0 = blockIdx.x * kTp, d0 = blockIdx.y * kTp;
    const uint16_t *src = reinterpret_cast<const uint16_t *>(v) + (int64_t)f * N * D;
    uint16_t *dst = reinterpret_cast<uint16_t *>(vt) + (int64_t)f * D * ldn;
    for (int e = threadIdx.x; e < kTp * kTp / 8; e += blockDim.x) {
        const int i = e >> 3, c8 = (e & 7) * 8;  // position row, first dim
        const int n = n0 + i;
        uint4 w = make_uint4(0u, 0u, 0u, 0u);
        if (n < N) w = __ldg(reinterpret_cast<const uint4 *>(src + (int64_t)n * D + d0 + c8));
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            tile[i][c8 + 2 * k] = (uint16_t)(ws[k] & 0xffffu);
            tile[i][c8 + 2 * k + 1] = (uint16_t)(ws[k] >> 16);
        }
    }
    __syncthreads();
    for (int e = threadIdx.x; e < kTp * kTp / 8; e += blockDim.x) {
        const int j = e >> 3, p8 = (e & 7) * 8;  // dim row, first position
        const int n = n0 + p8;
        if (n >= N) continue;
        uint16_t *out = dst + (int64_t)(d0 + j) * ldn + n;
        if (n + 8 <= N) {
            uint32_t ws[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                ws[k] = (uint32_t)tile[p8 + 2 * k][j] | ((uint32_t)tile[p8 + 2 * k + 1][j] << 16);
            *reinterpret_cast<uint4 *>(out) = make_uint4(ws[0], ws[1], ws[2], ws[3]);
        } else {
            for (int k = 0; n + k < N; ++k) out[k] = tile[p8 + k][j];
        }
    }
}

}  // namespace

int frame_attention_ldn(int N) { return (N + 7) / 8 * 8; }

cudaError_t launch_transpose_v(const void *v, void *vt, int F, int N, int D,
                               const LaunchCtx &ctx) {
    if (D % kTp) return cudaErrorInvalidValue;  // (D is 128, 256 or 384)
    const dim3 grid((unsigned)((N + kTp - 1) / kTp), (unsigned)(D / kTp), (unsigned)F);
    return launch_pdl(transpose_v_kernel, grid, dim3(256), 0, ctx,
                      static_cast<const __nv_bfloat16 *>(v), static_cast<__nv_bfloat16 *>(vt), N, D,
                      frame_attention_ldn(N));
}

cudaError_t launch_attention_core(const void *q, const void *k, const void *vt, void *out, int F,
                                  int N, int D, const LaunchCtx &ctx) {
    if (F < 1 || N < 1 || (D != 128 && D != 256 && D != 384)) return cudaErrorInvalidValue;
    const int ldn = frame_attention_ldn(N);
    CUtensorMap mQ, mK, mV;
    // Q and K: [F][N][D] as (D, N, F), boxes of 64 dims x 128 positions
    const cuuint64_t dq[3] = {(cuuint64_t)D, (cuuint64_t)N, (cuuint64_t)F};
    const cuuint64_t sq[2] = {(cuuint64_t)D * 2, (cuuint64_t)N * D * 2};
    const cuuint32_t bq[3] = {64, (cuuint32_t)kBlk, 1};
    // V^T: [F][D][ldn] as (N, D, F), boxes of 64 keys x 128 dims
    const cuuint64_t dv[3] = {(cuuint64_t)N, (cuuint64_t)D, (cuuint64_t)F};
    const cuuint64_t sv[2] = {(cuuint64_t)ldn * 2, (cuuint64_t)D * ldn * 2};
    const cuuint32_t bv[3] = {64, 128, 1};
    if (!encode_tiled_bf16(&mQ, 3, q, dq, sq, bq, 128) ||
        !encode_tiled_bf16(&mK, 3, k, dq, sq, bq, 128) ||
        !encode_tiled_bf16(&mV, 3, vt, dv, sv, bv, 128))
        return cudaErrorInvalidValue;
    AttnArgs a;
    memset(&a, 0, sizeof(a));
    a.F = F;
    a.N = N;
    a.D = D;
    a.q_tiles = (N + kBlk - 1) / kBlk;
    a.nkb = a.q_tiles;
    a.scale_log2 = 1.4426950408889634f / sqrtf((float)D);
    a.off_p = (uint32_t)(D / 64) * kAtom;          // Q: D / 64 atom columns
    a.off_ring = a.off_p + kStage;                 // P: 128 x 128
    a.off_bars = a.off_ring + kAStages * kStage;   // K / V^T ring
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.err = ctx.err;
    a.wait_ns = ctx.wait_ns;
    const size_t smem = 1024 + a.off_bars + 8 * kANumBars + 16;
    // The shared-memory opt-in, once per device (every launch asks for <= 227 KB).
    constexpr int kMaxDev = 64;
    static std::atomic<bool> attr_set[kMaxDev];
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return de;
    if (dev < 0 || dev >= kMaxDev) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        cudaError_t e = cudaFuncSetAttribute(attn_tcgen05_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             227 * 1024);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    if (smem > 227 * 1024) return cudaErrorInvalidValue;
    const int items = F * a.q_tiles;
    const int grid = items < ctx.num_sms ? items : ctx.num_sms;
    return launch_pdl(attn_tcgen05_kernel, dim3((unsigned)grid), dim3(kAThreads), smem, ctx, mQ,
                      mK, mV, a);
}

}  // namespace wanvae
