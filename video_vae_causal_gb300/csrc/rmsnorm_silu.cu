// rmsnorm_silu.cu -- fused RMS_norm over channels + SiLU on NDHWC voxels, and
// the feat_cache frame update.  Both are HBM-bound streaming passes.
//
// RMS_norm follows "Closing the gap: Wan 2.2 14B VAE decoder", section 4:
// the L2 norm over the channels of one voxel, clamped below by eps, divides
// the voxel, which is then scaled by sqrt(C) * gamma; tt-metal's fused
// rms_norm + SiLU kernel is the model for doing the activation in the same
// pass.  SiLU(z) = z * sigmoid(z).
#include <cuda_bf16.h>

#include "kernels.h"
#include "norm_act.cuh"
#include "ptx.cuh"

namespace wanvae {
namespace {

__device__ __forceinline__ float bf16lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// The pass is bound by issue slots, not DRAM, at 8 channels per 16-byte
// vector, so SiLU uses the fast reciprocal-based divide (for z below about
// -87 the denominator overflows and the result is the limit 0).
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// The pass's activation: SiLU, or none (the attention block's norm).
template <bool kSilu>
__device__ __forceinline__ float act(float z) {
    return kSilu ? silu(z) : z;
}

// One group of L lanes owns one voxel; each lane holds VPT 16-byte vectors
// of it (vector j of the voxel lives in lane j % L, slot j / L), so every
// warp-wide load covers 32 consecutive 16-byte vectors of (32 / L) voxels.
// A warp works on U such voxel groups per iteration and issues all their
// loads before the first reduction, so U * VPT loads per lane are in flight
// (the pass is bound by DRAM latency x bytes in flight).  The channel sum of
// squares is reduced with xor-shuffles inside the group.
template <bool F32, int VPT, int U, bool kSilu>
__global__ void __launch_bounds__(256)
rmsnorm_silu_kernel(const uint4 *__restrict__ x, uint4 *__restrict__ y,
                    const float *__restrict__ gamma, int64_t n, int C, int L, float eps,
                    float sqrt_c) {
    griddep_launch_dependents();
    griddep_wait();
    constexpr int E = F32 ? 4 : 8;  // channels per 16-byte vector
    const int V = C / E;            // vectors per voxel
    const int lane = threadIdx.x & 31;
    const int sub = lane & (L - 1);
    const int grp = lane / L;
    const int gpw = 32 / L;
    const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;

    for (int64_t v0 = warp_id * gpw * U; v0 < n; v0 += nwarps * gpw * U) {
        uint4 buf[U][VPT];
        float ss[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = v0 + u * gpw + grp;
#pragma unroll
            for (int i = 0; i < VPT; ++i)
                if (v < n) buf[u][i] = __ldg(x + v * V + sub + i * L);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = v0 + u * gpw + grp;
            ss[u] = 0.f;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                if (v >= n) continue;
                if (F32) {
                    float a = __uint_as_float(buf[u][i].x), b = __uint_as_float(buf[u][i].y);
                    float c = __uint_as_float(buf[u][i].z), d = __uint_as_float(buf[u][i].w);
                    ss[u] += a * a + b * b + c * c + d * d;
                } else {
                    ss[u] = nact_sumsq8(buf[u][i], ss[u]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (F32) {
                for (int off = L >> 1; off > 0; off >>= 1)
                    ss[u] += __shfl_xor_sync(0xffffffffu, ss[u], off);
            } else {
                ss[u] = nact_group_sum(ss[u], L);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = v0 + u * gpw + grp;
            if (v >= n) continue;
            const float scale = F32 ? sqrt_c / fmaxf(sqrtf(ss[u]), eps)
                                    : nact_scale(ss[u], sqrt_c, eps);
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int j = sub + i * L;
                const float4 *g4 = reinterpret_cast<const float4 *>(gamma + j * E);
                const uint4 b = buf[u][i];
                uint4 o;
                if (F32) {
                    const float4 g = __ldg(g4);
                    o.x = __float_as_uint(act<kSilu>(__uint_as_float(b.x) * scale * g.x));
                    o.y = __float_as_uint(act<kSilu>(__uint_as_float(b.y) * scale * g.y));
                    o.z = __float_as_uint(act<kSilu>(__uint_as_float(b.z) * scale * g.z));
                    o.w = __float_as_uint(act<kSilu>(__uint_as_float(b.w) * scale * g.w));
                } else {
                    o = nact_apply8<kSilu>(b, scale, __ldg(g4), __ldg(g4 + 1));
                }
                y[v * V + j] = o;
            }
        }
    }
}

template <bool F32, bool kSilu = true>
cudaError_t dispatch_norm(const void *x, void *y, const float *gamma, int64_t n, int C, float eps,
                          const LaunchCtx &ctx) {
    constexpr int E = F32 ? 4 : 8;
    const int V = C / E;
    int L = 1;
    while (L < 32 && V % (2 * L) == 0) L *= 2;  // largest power of two dividing V
    const int vpt = V / L;
    const int threads = 256;
    const int64_t voxels_per_block = (threads / 32) * (32 / L) * (vpt <= 4 ? 2 : 1);
    const int64_t blocks = (n + voxels_per_block - 1) / voxels_per_block;
    const float sqrt_c = sqrtf((float)C);
    auto *xi = static_cast<const uint4 *>(x);
    auto *yo = static_cast<uint4 *>(y);
    // One resident wave (grid-stride beyond it): as many CTAs per SM as the
    // instantiation's registers allow, looked up once per instantiation.
#define WANVAE_NORM_CASE(K)                                                              \
    case K: {                                                                            \
        auto *kern = rmsnorm_silu_kernel<F32, K, (K <= 4 ? 2 : 1), kSilu>;               \
        static int per_sm = 0;                                                           \
        if (per_sm == 0 &&                                                               \
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, 0) !=  \
                cudaSuccess)                                                             \
            per_sm = 2;                                                                  \
        if (per_sm < 1) per_sm = 1;                                                      \
        const int64_t cap = (int64_t)ctx.num_sms * per_sm;                               \
        const cudaError_t le = launch_pdl(kern, dim3((unsigned)(blocks < cap ? blocks : cap)), \
                                          dim3(threads), 0, ctx, xi, yo, gamma, n, C, L, eps,   \
                                          sqrt_c);                                              \
        if (le != cudaSuccess) return le;                                                \
        break;                                                                           \
    }
    switch (vpt) {
        WANVAE_NORM_CASE(1)
        WANVAE_NORM_CASE(2)
        WANVAE_NORM_CASE(3)
        WANVAE_NORM_CASE(4)
        WANVAE_NORM_CASE(5)
        WANVAE_NORM_CASE(6)
        WANVAE_NORM_CASE(7)
        WANVAE_NORM_CASE(8)
        WANVAE_NORM_CASE(9)
        WANVAE_NORM_CASE(10)
        WANVAE_NORM_CASE(11)
        WANVAE_NORM_CASE(12)
        WANVAE_NORM_CASE(13)
        WANVAE_NORM_CASE(14)
        WANVAE_NORM_CASE(15)
        WANVAE_NORM_CASE(16)
        default:
            return cudaErrorInvalidValue;
    }
#undef WANVAE_NORM_CASE
    return cudaGetLastError();
}

// cache[b] <- last two frames of concat(cache[b], src[b]).  For T >= 2 both
// frames come from src; for T == 1 frame 1 moves to frame 0 and src's only
// frame becomes frame 1 (each element is read before it is overwritten by
// the same thread, so the in-place shift has no race).
__global__ void cache_update_kernel(uint4 *__restrict__ cache, const uint4 *__restrict__ src,
                                    int B, int T, int64_t fv) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t total = (int64_t)B * fv;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / fv, e = i - b * fv;
        uint4 *c = cache + b * 2 * fv + e;
        const uint4 *s = src + b * (int64_t)T * fv + e;
        if (T >= 2) {
            c[0] = s[(int64_t)(T - 2) * fv];
            c[fv] = s[(int64_t)(T - 1) * fv];
        } else {
            const uint4 keep = c[fv];
            c[0] = keep;
            c[fv] = s[0];
        }
    }
}

// Both convs' feat_cache updates in one launch (blockIdx.y picks the pair):
// the same copy as cache_update_kernel for (cache0, src0) and (cache1, src1).
__global__ void cache_update2_kernel(uint4 *__restrict__ cache0, const uint4 *__restrict__ src0,
                                     int64_t fv0, uint4 *__restrict__ cache1,
                                     const uint4 *__restrict__ src1, int64_t fv1, int B, int T) {
    griddep_launch_dependents();
    griddep_wait();
    uint4 *cache = blockIdx.y ? cache1 : cache0;
    const uint4 *src = blockIdx.y ? src1 : src0;
    const int64_t fv = blockIdx.y ? fv1 : fv0;
    const int64_t total = (int64_t)B * fv;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t b = i / fv, e = i - b * fv;
        uint4 *c = cache + b * 2 * fv + e;
        const uint4 *sp = src + b * (int64_t)T * fv + e;
        if (T >= 2) {
            c[0] = sp[(int64_t)(T - 2) * fv];
            c[fv] = sp[(int64_t)(T - 1) * fv];
        } else {
            const uint4 keep = c[fv];
            c[0] = keep;
            c[fv] = sp[0];
        }
    }
}

// feat_cache update of a conv whose input norm is fused (its input a1 =
// SiLU(RMS_norm(x)) is never written out): cache[b] <- the last two frames of
// concat(cache[b], a1(src[b])).  A group of L lanes owns a pixel, lane `sub`
// its vectors sub, sub + L, ..., the grouping and arithmetic of the
// standalone pass, so the frames are bit for bit those that pass (and the
// conv's fused transform) produce.  T == 1: frame 1 moves to frame 0 and a1 of
// src's frame becomes frame 1; each lane copies its own vectors of a pixel
// before it overwrites them, so the in-place shift has no race.
template <int VPT>
__global__ void __launch_bounds__(256)
cache_update_norm_kernel(uint4 *__restrict__ cache, const uint4 *__restrict__ src,
                         const float *__restrict__ gamma, int B, int T, int64_t HW, int C, int L,
                         float eps, float sqrt_c) {
    griddep_launch_dependents();
    griddep_wait();
    const int V = C / 8;  // 16-byte vectors per pixel
    const int lane = threadIdx.x & 31;
    const int sub = lane & (L - 1), grp = lane / L, gpw = 32 / L;
    const int64_t warp_id = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t npix = (int64_t)B * HW;
    const float4 *g4 = reinterpret_cast<const float4 *>(gamma);
    for (int64_t p0 = warp_id * gpw; p0 < npix; p0 += nwarps * gpw) {  // warp-uniform
        const int64_t pix = p0 + grp;
        const bool valid = pix < npix;
        const int64_t b = valid ? pix / HW : 0, q = valid ? pix - b * HW : 0;
        uint4 *c0 = cache + ((b * 2 + 0) * HW + q) * V;
        uint4 *c1 = cache + ((b * 2 + 1) * HW + q) * V;
        // frames of src that become cache frames: T >= 2: T-2 -> 0 and T-1 -> 1
        for (int f = (T >= 2 ? 0 : 1); f < 2; ++f) {
            const int tsrc = T - 2 + f;
            const uint4 *ps = src + ((b * T + tsrc) * HW + q) * V;
            uint4 v[VPT];
            float ss = 0.f;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                v[i] = valid ? __ldg(ps + sub + i * L) : make_uint4(0u, 0u, 0u, 0u);
                ss = nact_sumsq8(v[i], ss);
            }
            ss = nact_group_sum(ss, L);
            const float scale = nact_scale(ss, sqrt_c, eps);
            if (!valid) continue;
            uint4 *dst = f == 0 ? c0 : c1;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int j = sub + i * L;
                if (T == 1) c0[j] = c1[j];  // (f == 1 only: move frame 1 first)
                dst[j] = nact_apply8<true>(v[i], scale, __ldg(g4 + 2 * j), __ldg(g4 + 2 * j + 1));
            }
        }
    }
}

// Sub-pixel weights of the upsampler conv.  Nearest 2x upsampling then a 3x3
// conv gives output pixel (2i + a, 2j + b) as a conv over the low-res input
// around (i, j): tap (kh, kw) of the upsampled grid reads low-res row
// i + floor((a + kh - 1) / 2) (offsets -1, 0, 0 for a = 0 and 0, 0, 1 for
// a = 1), likewise for columns, so each phase (a, b) touches only the 2 x 2
// low-res offsets (a + e - 1, b + f - 1), e, f in {0, 1}, and its tap (e, f)
// is the sum of the original taps that land there.
// w [Co][3][3][Ci] -> w2 [4 = 2a + b][Co][2][2][Ci], fp32 sums rounded to bf16.
__global__ void expand_up2d_weights_kernel(const __nv_bfloat16 *__restrict__ w,
                                           __nv_bfloat16 *__restrict__ w2, int Co, int Ci) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t total = (int64_t)4 * Co * 4 * Ci;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(idx % Ci);
        int64_t r = idx / Ci;
        const int f = (int)(r & 1);
        const int e = (int)((r >> 1) & 1);
        r >>= 2;
        const int o = (int)(r % Co);
        const int ph = (int)(r / Co), a = ph >> 1, b = ph & 1;
        float acc = 0.f;
        for (int kh = 0; kh < 3; ++kh) {
            if (((a + kh + 1) >> 1) != a + e) continue;  // floor((a + kh - 1) / 2) + 1
            for (int kw = 0; kw < 3; ++kw) {
                if (((b + kw + 1) >> 1) != b + f) continue;
                acc += __bfloat162float(w[((int64_t)(o * 3 + kh) * 3 + kw) * Ci + c]);
            }
        }
        w2[idx] = __float2bfloat16_rn(acc);
    }
}

// Phase weights of the temporal upsampler conv.  Nearest 2x in T then a
// causal 3-tap conv gives output frame 2t + a as a conv over input frames
// t - 1 and t: tap kt of the upsampled sequence reads upsampled frame
// 2t + a + kt - 2, i.e. input frame t - 1 + ((a + kt) >> 1).  So phase a's tap
// e in {0, 1} (frame t - 1 + e) is the sum of the taps kt with
// (a + kt) >> 1 == e: w0 + w1 and w2 for a = 0, w0 and w1 + w2 for a = 1.
// w [Co][3][Ci] -> w2 [2 = a][Co][2 = e][Ci], fp32 sums rounded to bf16.
__global__ void expand_time_up_weights_kernel(const __nv_bfloat16 *__restrict__ w,
                                              __nv_bfloat16 *__restrict__ w2, int Co, int Ci) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t total = (int64_t)2 * Co * 2 * Ci;
    for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
         idx += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(idx % Ci);
        int64_t r = idx / Ci;
        const int e = (int)(r & 1);
        r >>= 1;
        const int o = (int)(r % Co);
        const int a = (int)(r / Co);
        float acc = 0.f;
        for (int kt = 0; kt < 3; ++kt)
            if (((a + kt) >> 1) == e) acc += __bfloat162float(w[((int64_t)o * 3 + kt) * Ci + c]);
        w2[idx] = __float2bfloat16_rn(acc);
    }
}

}  // namespace

cudaError_t launch_expand_time_up_weights(const void *w, void *w2, int Co, int Ci,
                                          const LaunchCtx &ctx) {
    const int64_t total = (int64_t)2 * Co * 2 * Ci;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)ctx.num_sms * 8) blocks = (int64_t)ctx.num_sms * 8;
    if (blocks < 1) blocks = 1;
    return launch_pdl(expand_time_up_weights_kernel, dim3((unsigned)blocks), dim3(256), 0, ctx,
                      static_cast<const __nv_bfloat16 *>(w), static_cast<__nv_bfloat16 *>(w2),
                      Co, Ci);
}

cudaError_t launch_expand_up2d_weights(const void *w, void *w2, int Co, int Ci,
                                       const LaunchCtx &ctx) {
    const int64_t total = (int64_t)4 * Co * 4 * Ci;
    int64_t blocks = (total + 255) / 256;
    if (blocks > (int64_t)ctx.num_sms * 8) blocks = (int64_t)ctx.num_sms * 8;
    return launch_pdl(expand_up2d_weights_kernel, dim3((unsigned)blocks), dim3(256), 0, ctx,
                      static_cast<const __nv_bfloat16 *>(w), static_cast<__nv_bfloat16 *>(w2),
                      Co, Ci);
}

cudaError_t launch_rmsnorm(const void *x, void *y, const float *gamma, int64_t n, int C,
                           float eps, const LaunchCtx &ctx) {
    return dispatch_norm<false, false>(x, y, gamma, n, C, eps, ctx);
}

cudaError_t launch_rmsnorm_silu(const void *x, void *y, const float *gamma, bool is_f32,
                                int64_t n, int C, float eps, const LaunchCtx &ctx) {
    return is_f32 ? dispatch_norm<true>(x, y, gamma, n, C, eps, ctx)
                  : dispatch_norm<false>(x, y, gamma, n, C, eps, ctx);
}

cudaError_t launch_cache_update_norm(void *cache, const void *src, const float *gamma, int B,
                                     int T, int64_t HW, int C, float eps, const LaunchCtx &ctx) {
    const int L = nact_lanes(C), vpt = (C / 8) / L;
    const int threads = 256;
    int64_t blocks = ((int64_t)B * HW * L + threads - 1) / threads;
    const int64_t cap = (int64_t)ctx.num_sms * 4;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    auto *c = static_cast<uint4 *>(cache);
    auto *x = static_cast<const uint4 *>(src);
    const float sc = sqrtf((float)C);
    switch (vpt) {
        case 1: return launch_pdl(cache_update_norm_kernel<1>, dim3((unsigned)blocks),
                                  dim3(threads), 0, ctx, c, x, gamma, B, T, HW, C, L, eps, sc);
        case 2: return launch_pdl(cache_update_norm_kernel<2>, dim3((unsigned)blocks),
                                  dim3(threads), 0, ctx, c, x, gamma, B, T, HW, C, L, eps, sc);
        case 3: return launch_pdl(cache_update_norm_kernel<3>, dim3((unsigned)blocks),
                                  dim3(threads), 0, ctx, c, x, gamma, B, T, HW, C, L, eps, sc);
        case 4: return launch_pdl(cache_update_norm_kernel<4>, dim3((unsigned)blocks),
                                  dim3(threads), 0, ctx, c, x, gamma, B, T, HW, C, L, eps, sc);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_cache_update2(void *cache0, const void *src0, int64_t frame_bytes0,
                                 void *cache1, const void *src1, int64_t frame_bytes1, int B,
                                 int T, const LaunchCtx &ctx) {
    const int64_t fv0 = frame_bytes0 / 16, fv1 = frame_bytes1 / 16;
    const int threads = 256;
    const int64_t fv = fv0 > fv1 ? fv0 : fv1;
    int64_t blocks = ((int64_t)B * fv + threads - 1) / threads;
    const int64_t cap = (int64_t)ctx.num_sms * 4;  // x 2 pairs
    if (blocks > cap) blocks = cap;
    return launch_pdl(cache_update2_kernel, dim3((unsigned)blocks, 2), dim3(threads), 0, ctx,
                      static_cast<uint4 *>(cache0), static_cast<const uint4 *>(src0), fv0,
                      static_cast<uint4 *>(cache1), static_cast<const uint4 *>(src1), fv1, B, T);
}

cudaError_t launch_cache_update(void *cache, const void *src, int B, int T, int64_t frame_bytes,
                                const LaunchCtx &ctx) {
    const int64_t fv = frame_bytes / 16;
    const int threads = 256;
    int64_t blocks = ((int64_t)B * fv + threads - 1) / threads;
    const int64_t cap = (int64_t)ctx.num_sms * 8;
    if (blocks > cap) blocks = cap;
    return launch_pdl(cache_update_kernel, dim3((unsigned)blocks), dim3(threads), 0, ctx,
                      static_cast<uint4 *>(cache), static_cast<const uint4 *>(src), B, T, fv);
}

}  // namespace wanvae
