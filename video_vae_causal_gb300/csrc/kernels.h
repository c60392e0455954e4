// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernels (rmsnorm_silu.cu, conv3d_tcgen05.cu).  Not installed, not exported.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace wanvae {

// Per-launch context every kernel needs: the device error word and the
// bound on device-side waits.
struct LaunchCtx {
    cudaStream_t stream;
    unsigned *err;      // device address of the error word
    uint64_t wait_ns;   // bound of every device-side wait
    int num_sms;
};

// Launch `kern` on ctx.stream with programmatic dependent launch allowed (the
// kernel must call griddep_wait before reading what earlier work wrote).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       const LaunchCtx &ctx, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = ctx.stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// SiLU(RMS_norm(x)) over C channels of n voxels; is_f32 selects fp32 in/out
// (else bf16).  Returns a cudaError_t.
cudaError_t launch_rmsnorm_silu(const void *x, void *y, const float *gamma, bool is_f32,
                                int64_t n, int C, float eps, const LaunchCtx &ctx);

// RMS_norm alone (no activation), bf16 in and out: the attention block's norm.
cudaError_t launch_rmsnorm(const void *x, void *y, const float *gamma, int64_t n, int C,
                           float eps, const LaunchCtx &ctx);

// The attention core (attn_tcgen05.cu): out = softmax(q k^T / sqrt(D)) v per
// frame, q, k, out bf16 [F][N][D], vt bf16 [F][D][frame_attention_ldn(N)]
// (V transposed by launch_transpose_v); D = 128, 256 or 384.
int frame_attention_ldn(int N);
cudaError_t launch_transpose_v(const void *v, void *vt, int F, int N, int D, const LaunchCtx &ctx);
cudaError_t launch_attention_core(const void *q, const void *k, const void *vt, void *out, int F,
                                  int N, int D, const LaunchCtx &ctx);

// cache[b] <- last two frames of concat(cache[b], src[b]) along T, for bf16
// tensors of frame_bytes bytes per frame (a multiple of 16).
cudaError_t launch_cache_update(void *cache, const void *src, int B, int T, int64_t frame_bytes,
                                const LaunchCtx &ctx);
// The same for two (cache, src) pairs in one launch.
cudaError_t launch_cache_update2(void *cache0, const void *src0, int64_t frame_bytes0,
                                 void *cache1, const void *src1, int64_t frame_bytes1, int B,
                                 int T, const LaunchCtx &ctx);

// Sub-pixel weights of the upsampler conv: w [Co][3][3][Ci] ->
// w2 [4 phases][Co][2][2][Ci] (bf16), see rmsnorm_silu.cu.
cudaError_t launch_expand_up2d_weights(const void *w, void *w2, int Co, int Ci,
                                       const LaunchCtx &ctx);

// Phase weights of the temporal upsampler conv: w [Co][3][Ci] ->
// w2 [2 phases][Co][2][Ci] (bf16), see rmsnorm_silu.cu.
cudaError_t launch_expand_time_up_weights(const void *w, void *w2, int Co, int Ci,
                                          const LaunchCtx &ctx);

// Epilogue of the implicit-GEMM conv.
enum EpiMode : int {
    kEpiBias = 0,      // out = acc + bias (+ bias2)
    kEpiNormSilu = 1,  // out = SiLU(RMS_norm(acc + bias) * gamma) over all c_out
    kEpiResidual = 2,  // out = acc + bias (+ bias2) + resid  (resid: [M][c_out])
};

// One CausalConv3d as an implicit GEMM on tcgen05 (M = voxels, N = c_out,
// K = taps * c_in), optionally followed in the same accumulator by a 1x1x1
// shortcut segment (K += c_sc over sc_in with weights sc_w).
struct ConvSpec {
    const void *in;      // bf16 [B][T][H][W][c_in]
    const void *cache;   // bf16 [B][2][H][W][c_in] frames t-2, t-1, or NULL (zeros)
    const void *w;       // bf16 [c_out][k][k][k][c_in]
    const float *bias;   // [c_out] or NULL
    const float *bias2;  // [c_out] or NULL (added to bias)
    const float *gamma;  // [c_out], kEpiNormSilu only
    float eps;
    const void *resid;   // bf16 [M][c_out], kEpiResidual only
    const void *sc_in;   // bf16 [M][c_sc] or NULL (no shortcut segment)
    const void *sc_w;    // bf16 [c_out][c_sc]
    void *out;           // bf16 [B][T][H][W][c_out]
    int B, T, H, W;
    int c_in, c_out, c_sc;
    int k;               // 3 or 1
    int epi;             // EpiMode
    // Spatial upsampler conv: nearest 2x in H and W then a 3x3 conv, as four
    // sub-pixel phases over the low-res input (H x W here), each a 2 x 2 conv.
    // w holds the sub-pixel weights [4][c_out][2][2][c_in] (the current
    // frame's taps only), out is [B][T][2H][2W][c_out]; k = 3, no cache, bias
    // epilogue.
    int up2d;
    // Temporal upsampler conv (upsample3d's temporal half): nearest 2x in T
    // then a causal 3x1x1 conv, as two frame phases over the input frames:
    // output frame 2t + a is a 2-tap conv of input frames t - 1 and t.  w holds
    // the phase weights [2][c_out][2][c_in]; out is [B][2T][H][W][c_out];
    // k = 3, no cache, bias epilogue.
    int up_t;
    // Fused input norm (the block's conv A): the conv reads the raw block
    // input x as `in` and applies SiLU(RMS_norm(x; gamma_in, eps)) to every
    // halo pixel on its way to shared memory, so a1 is never written out.
    // `cache` then holds normalised frames, as without fusion.  Honoured only
    // where conv3d_fuses_norm() says the plan allows it.
    int norm_in;
    const float *gamma_in;  // [c_in]
};

// Whether launch_conv3d runs `s` (with norm_in set) with the input norm fused
// into the conv: halo tiles whose one channel chunk holds all c_in channels
// (c_in <= 128), no shortcut segment, double-buffered accumulators.
bool conv3d_fuses_norm(const ConvSpec &s);

// feat_cache update for a fused conv: cache[b] <- the last two frames of
// concat(cache[b], SiLU(RMS_norm(src[b]; gamma, eps))), src bf16
// [B][T][HW][C]; the same arithmetic and lane grouping as the standalone
// norm pass (bit-identical frames).
cudaError_t launch_cache_update_norm(void *cache, const void *src, const float *gamma, int B,
                                     int T, int64_t HW, int C, float eps, const LaunchCtx &ctx);

// Host-side validation of a ConvSpec the library can run (channel counts,
// sizes); returns 0 if supported.
int conv3d_supported(const ConvSpec &s);

// Enqueue the conv; returns a cudaError_t (cudaErrorInvalidValue when a
// tensor map cannot be encoded).
cudaError_t launch_conv3d(const ConvSpec &s, const LaunchCtx &ctx);

// The k=3 conv for very narrow outputs (c_out <= 3, a decoder's conv_out to
// RGB) as one GEMM over all 27 taps at once plus a 3x3x3 stencil sum
// (conv3d_narrow.cu).  conv3d_narrow_supported returns 0 when it applies.
int conv3d_narrow_supported(const ConvSpec &s);
cudaError_t launch_conv3d_narrow(const ConvSpec &s, const LaunchCtx &ctx);

// Kernel-variant overrides, process-wide (wanvae_set_kernel_variant): each
// argument 0 or 1 forces that choice, anything else restores the automatic
// choice.  pair: 1 = single-CTA kernel, else CTA pairs; halo: halo tiles (1)
// or im2col tiles (0); wide: 16 x 16 halo patches (1) or 16 x 8 (0); narrow:
// the GEMM-plus-stencil kernel for c_out <= 3 (1) or the implicit GEMM (0);
// fuse: 1 = fuse the block's input norm into conv A where possible, else never.
void set_kernel_variant(int pair, int halo, int wide, int narrow, int fuse);
int narrow_variant();

// cuTensorMapEncodeTiled for a bf16 tensor of `rank` dimensions (driver
// entry point looked up once); swizzle_bytes 0, 32, 64 or 128.  False when
// the entry point is missing or the encoding is rejected.
bool encode_tiled_bf16(CUtensorMap *m, int rank, const void *base, const cuuint64_t *dims,
                       const cuuint64_t *strides, const cuuint32_t *box, int swizzle_bytes);

}  // namespace wanvae
