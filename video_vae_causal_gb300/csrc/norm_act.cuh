// norm_act.cuh -- the RMS_norm (+ SiLU) arithmetic on bf16 voxels, shared by
// the standalone norm pass, the conv kernel's fused input transform and the
// feat_cache kernel that writes normalised frames.  Every step is an
// explicitly rounded operation (no contraction left to the compiler), so all
// three produce the same bits for the same voxel when they use the same lane
// grouping (L lanes per voxel, lane `sub` holding the voxel's 16-byte vectors
// sub, sub + L, ...).
//
// RMS_norm ("Closing the gap: Wan 2.2 14B VAE decoder", section 4): the L2
// norm over the voxel's channels, clamped below by eps, divides the voxel,
// which is then scaled by sqrt(C) * gamma.  SiLU(z) = z / (1 + exp(-z)).
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

namespace wanvae {

__device__ __forceinline__ float nact_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float nact_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t nact_pack(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// ss plus the squares of the 8 bf16 channels of v, in channel order.
__device__ __forceinline__ float nact_sumsq8(const uint4 &v, float ss) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float a = nact_lo(w[k]), b = nact_hi(w[k]);
        ss = __fmaf_rn(a, a, ss);
        ss = __fmaf_rn(b, b, ss);
    }
    return ss;
}

// Sum over the L lanes of a group (L a power of two, every lane of the warp
// taking part).
__device__ __forceinline__ float nact_group_sum(float ss, int L) {
    for (int off = L >> 1; off > 0; off >>= 1)
        ss = __fadd_rn(ss, __shfl_xor_sync(0xffffffffu, ss, off));
    return ss;
}

// sqrt(C) / max(||v||, eps)
__device__ __forceinline__ float nact_scale(float ss, float sqrt_c, float eps) {
    return __fdiv_rn(sqrt_c, fmaxf(__fsqrt_rn(ss), eps));
}

// SiLU with the fast reciprocal-based divide; for z below about -87 the
// denominator overflows and the result is the limit 0.
__device__ __forceinline__ float nact_silu(float z) {
    return __fdividef(z, __fadd_rn(1.0f, __expf(-z)));
}

template <bool kSilu>
__device__ __forceinline__ float nact_act(float x, float scale, float g) {
    const float z = __fmul_rn(__fmul_rn(x, scale), g);
    return kSilu ? nact_silu(z) : z;
}

// The 8 channels of v normalised (gamma ga = channels 0-3, gb = 4-7) and,
// with kSilu, passed through SiLU; bf16 round to nearest even.
template <bool kSilu>
__device__ __forceinline__ uint4 nact_apply8(const uint4 &v, float scale, const float4 &ga,
                                            const float4 &gb) {
    uint4 o;
    o.x = nact_pack(nact_act<kSilu>(nact_lo(v.x), scale, ga.x),
                    nact_act<kSilu>(nact_hi(v.x), scale, ga.y));
    o.y = nact_pack(nact_act<kSilu>(nact_lo(v.y), scale, ga.z),
                    nact_act<kSilu>(nact_hi(v.y), scale, ga.w));
    o.z = nact_pack(nact_act<kSilu>(nact_lo(v.z), scale, gb.x),
                    nact_act<kSilu>(nact_hi(v.z), scale, gb.y));
    o.w = nact_pack(nact_act<kSilu>(nact_lo(v.w), scale, gb.z),
                    nact_act<kSilu>(nact_hi(v.w), scale, gb.w));
    return o;
}

// Lanes per voxel for C channels: the largest power of two (at most 32)
// dividing the voxel's C / 8 vectors.
__host__ __device__ __forceinline__ int nact_lanes(int C) {
    const int V = C / 8;
    int L = 1;
    while (L < 32 && V % (2 * L) == 0) L *= 2;
    return L;
}

}  // namespace wanvae
