/*
 * wanvae.h -- C ABI of libwanvae.so: the Wan 2.2 VAE decoder ResidualBlock
 * forward pass on one NVIDIA GB300 (sm_103a), NDHWC bf16 end to end.
 *
 * The block ("Sharding of WAN 2.2 VAE", section "Channel sharding (in
 * Megatron style)", ResidualBlock listing and op-sequence figure):
 *
 *     a1 = SiLU(RMS_norm(x;  gamma1))            RMS over channels, C = c_in
 *     h  = CausalConv3d_A(a1)                    3x3x3, c_in  -> c_out
 *     a2 = SiLU(RMS_norm(h;  gamma2))            C = c_out
 *     r  = CausalConv3d_B(a2)                    3x3x3, c_out -> c_out
 *     y  = r + shortcut(x)                       1x1x1 conv, or Identity when
 *                                                c_in == c_out and no wS given
 *
 * RMS_norm ("Closing the gap: Wan 2.2 14B VAE decoder", section 4) is
 *     RMS_norm(v)[c] = v[c] / max(||v||_2, eps) * sqrt(C) * gamma[c]
 * with the L2 norm taken over the channels of one voxel and no bias.
 * CausalConv3d ("Closing the gap", section 2; "Sharding of WAN 2.2 VAE",
 * Conv3D strategy table) is a stride-1 3x3x3 convolution that pads two
 * leading frames in T (zeros, or the feat_cache frames) and one element on
 * each side of H and W (zeros):
 *     out[b,t,y,x,o] = bias[o] + sum_{kt,kh,kw,c} w[o,kt,kh,kw,c]
 *                          * in[b, t+kt-2, y+kh-1, x+kw-1, c].
 * kt = 2 is the current frame, kt = 0 is frame t-2.
 *
 * Conventions for every call:
 *  - Layout: activations are NDHWC ([B][T][H][W][C], C fastest, densely
 *    packed); conv weights are [c_out][kT][kH][kW][c_in] bf16 (k = 3 or 1);
 *    gammas and biases are fp32.  bf16 pointers are typed `void *` so that
 *    the header needs no CUDA include; they hold IEEE bfloat16 bit patterns.
 *  - Memory: every pointer argument is DEVICE memory owned by the caller,
 *    except where a comment says "host".  The library never allocates,
 *    frees or synchronises on these calls; all work is enqueued on `stream`
 *    (a cudaStream_t; NULL is the legacy default stream).
 *  - Requirements: C (each of c_in, c_out) a multiple of 16 and at most 512;
 *    all device pointers 16-byte aligned; outputs must not alias inputs;
 *    every dimension >= 1 and B*T*H*W < 2^31 voxels.
 *  - Errors: argument errors are returned synchronously, before any launch,
 *    and nothing is enqueued.  A failed launch returns WANVAE_ERR_CUDA.
 *    Every device-side wait is bounded; a wait that runs out sets a device
 *    flag that wanvae_sync_status() reports as WANVAE_ERR_TIMEOUT.
 *  - The library never prints and never exits the process.
 */
#ifndef WANVAE_H
#define WANVAE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    WANVAE_OK = 0,
    WANVAE_ERR_INVALID_ARG = 1, /* null pointer, bad size, aliasing, bad enum */
    WANVAE_ERR_UNSUPPORTED = 2, /* legal block, but a size the library rejects */
    WANVAE_ERR_MISALIGNED = 3,  /* a pointer is not 16-byte aligned */
    WANVAE_ERR_WORKSPACE = 4,   /* workspace NULL or smaller than required */
    WANVAE_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed */
    WANVAE_ERR_TIMEOUT = 6,     /* a device-side bounded wait ran out */
    WANVAE_ERR_UNDRAINED = 7    /* a wait ran out, and then so did the kernel's wait
                                   for its own in-flight copies or MMAs: they may
                                   have landed after it returned, so the CUDA context
                                   should not be reused */
} wanvae_status;

typedef enum { WANVAE_BF16 = 0, WANVAE_F32 = 1 } wanvae_dtype;

/* The CUDA stream type, declared without including the CUDA headers
 * (identical to cudaStream_t). */
typedef struct CUstream_st *wanvae_stream;

/* Clip extent; the channel count is passed separately. */
typedef struct {
    int64_t B, T, H, W;
} wanvae_dims;

/* ResidualBlock parameters (all device pointers, caller-owned). */
typedef struct {
    int64_t c_in, c_out;
    float eps;            /* RMS_norm clamp; 1e-12 reproduces F.normalize */
    const float *gamma1;  /* [c_in]  RMS_norm 1 scale */
    const float *gamma2;  /* [c_out] RMS_norm 2 scale */
    const void *wA;       /* bf16 [c_out][3][3][3][c_in]  conv A */
    const float *bA;      /* [c_out] */
    const void *wB;       /* bf16 [c_out][3][3][3][c_out] conv B */
    const float *bB;      /* [c_out] */
    const void *wS;       /* bf16 [c_out][1][1][1][c_in] shortcut, or NULL =
                             Identity (then c_in must equal c_out) */
    const float *bS;      /* [c_out] shortcut bias, or NULL (= zeros) */
} wanvae_resblock_params;

/* feat_cache of one ResidualBlock for frame-by-frame decode ("Sharding of
 * WAN 2.2 VAE", section "Why depth sharding is not beneficial": the cache
 * holds the last frames of each CausalConv3d's input).  Each buffer holds
 * the two frames that precede the call's first frame, of that conv's input
 * (post norm+SiLU): convA_in bf16 [B][2][H][W][c_in], convB_in bf16
 * [B][2][H][W][c_out], frame 0 = t-2, frame 1 = t-1.  The caller zero-fills
 * both before the clip's first frame.  A call reads them and then replaces
 * them, in stream order, with the last two frames of concat(cache, this
 * call's conv input). */
typedef struct {
    void *convA_in;
    void *convB_in;
} wanvae_resblock_cache;

/* Human-readable name of a status (static string, never NULL). */
const char *wanvae_status_string(wanvae_status s);

/* Library ABI version: 100 * major + minor. */
int wanvae_version(void);

/* SiLU(RMS_norm(x)) over the channels of n_voxels voxels ("Closing the gap",
 * section 4: one fused norm + SiLU kernel).
 *   x, y    : [n_voxels][C] of type dt (bf16 or fp32), y may not alias x.
 *   gamma   : fp32 [C].
 *   Math in fp32; bf16 outputs are rounded to nearest-even.
 * Errors: INVALID_ARG (null, n_voxels < 1, C < 16 or C % 16, C > 4096, bad
 * dt), MISALIGNED, CUDA. */
wanvae_status wanvae_rmsnorm_silu(const void *x, void *y, const float *gamma,
                                  wanvae_dtype dt, int64_t n_voxels, int64_t C,
                                  float eps, wanvae_stream stream);

/* One CausalConv3d (definition above), bf16 in/out, fp32 accumulate.
 *   x     : bf16 [B][T][H][W][c_in]      y: bf16 [B][T][H][W][c_out]
 *   w     : bf16 [c_out][k][k][k][c_in]  bias: fp32 [c_out] (NULL = zeros)
 *   k     : 3 (causal 3x3x3) or 1 (pointwise; cache must be NULL)
 *   cache : NULL for a whole clip (zero causal pad), or bf16 [B][2][H][W][c_in]
 *           holding the two frames before x (read, then replaced in stream
 *           order by the last two frames of concat(cache, x)).
 *   c_in  : a multiple of 16, at most 512.  c_out: 1 to 15 (a decoder's
 *           conv_out, e.g. 96 -> 3; the kernel pads N internally) or a
 *           multiple of 16 up to 512.
 * Errors: INVALID_ARG, UNSUPPORTED (other channel counts), MISALIGNED, CUDA. */
wanvae_status wanvae_causal_conv3d(const void *x, const void *w, const float *bias,
                                   void *y, wanvae_dims d, int64_t c_in, int64_t c_out,
                                   int k, void *cache, wanvae_stream stream);

/* The decoder's spatial upsampler ("Sharding of WAN 2.2 VAE", decoder tree:
 * WanUpBlock(..., upsample2d); its resample[1] is the conv): every frame is
 * upsampled 2x in H and W by nearest neighbour, then convolved 3x3 with one
 * pixel of zero pad and a bias (the pages give no more; this is the plainest
 * reading).
 *   x     : bf16 [B][T][H][W][c_in]  (d gives the low-res B, T, H, W)
 *   w     : bf16 [c_out][3][3][c_in] bias: fp32 [c_out] (NULL = zeros)
 *   y     : bf16 [B][T][2H][2W][c_out]
 *   workspace : device buffer of wanvae_upsample2d_workspace_size(c_in, c_out)
 *           bytes, 256-byte aligned, for the weights of the four sub-pixel
 *           phases: each phase of the output is a 2 x 2 conv of x whose taps
 *           are bf16 sums of the 3 x 3 taps it folds together (one more
 *           rounding of the weights than the plain definition).
 *   c_in  : a multiple of 16 up to 512; c_out: a multiple of 16 up to 256.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA. */
size_t wanvae_upsample2d_workspace_size(int64_t c_in, int64_t c_out);
wanvae_status wanvae_upsample2d_conv(const void *x, const void *w, const float *bias, void *y,
                                     wanvae_dims d, int64_t c_in, int64_t c_out,
                                     void *workspace, size_t ws_bytes, wanvae_stream stream);

/* The temporal half of the decoder's upsample3d ("Sharding of WAN 2.2 VAE",
 * decoder tree: WanUpBlock(..., upsample3d); the graph's 3x1x1 conv kernels,
 * "Closing the gap", section 3): every frame repeated twice in T (nearest
 * neighbour), then a causal conv with a 3x1x1 kernel (two zero frames before
 * the first) and a bias.  The pages give no more; this is the plainest
 * reading.  The spatial half is wanvae_upsample2d_conv on this call's output.
 *   x     : bf16 [B][T][H][W][c_in]
 *   w     : bf16 [c_out][3][c_in] (tap 2 reads the current upsampled frame)
 *   bias  : fp32 [c_out] (NULL = zeros)
 *   y     : bf16 [B][2T][H][W][c_out]
 *   workspace : device buffer of wanvae_time_upsample_workspace_size(c_in,
 *           c_out) bytes, 256-byte aligned, for the two frame phases'
 *           weights: output frame 2t + a is a 2-tap conv of input frames
 *           t - 1 and t whose taps are bf16 sums of the 3 taps (one more
 *           rounding of the weights than the plain definition).
 *   c_in, c_out : multiples of 16 up to 512.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA. */
size_t wanvae_time_upsample_workspace_size(int64_t c_in, int64_t c_out);
wanvae_status wanvae_time_upsample_conv(const void *x, const void *w, const float *bias,
                                        void *y, wanvae_dims d, int64_t c_in, int64_t c_out,
                                        void *workspace, size_t ws_bytes, wanvae_stream stream);

/* The decoder's whole upsample3d as read from the pages: the temporal half
 * (wanvae_time_upsample_conv, c_in -> c_mid) and then the spatial upsampler
 * (wanvae_upsample2d_conv, c_mid -> c_out) on every frame of its output.
 *   x : bf16 [B][T][H][W][c_in];  y : bf16 [B][2T][2H][2W][c_out]
 *   w_t : bf16 [c_mid][3][c_in], b_t : fp32 [c_mid] or NULL
 *   w_s : bf16 [c_out][3][3][c_mid], b_s : fp32 [c_out] or NULL
 *   workspace : wanvae_upsample3d_workspace_size(d, c_in, c_mid, c_out) bytes,
 *           256-byte aligned (the [B][2T][H][W][c_mid] intermediate and both
 *           calls' weight workspaces).
 * Errors: those of the two calls; WORKSPACE if ws_bytes is short. */
size_t wanvae_upsample3d_workspace_size(wanvae_dims d, int64_t c_in, int64_t c_mid,
                                        int64_t c_out);
wanvae_status wanvae_upsample3d(const void *x, const void *w_t, const float *b_t, const void *w_s,
                                const float *b_s, void *y, wanvae_dims d, int64_t c_in,
                                int64_t c_mid, int64_t c_out, void *workspace, size_t ws_bytes,
                                wanvae_stream stream);
/* The decoder's mid-block attention ("Closing the gap: Wan 2.2 14B VAE
 * decoder", section 5: a spatial self-attention within each frame; the
 * sequence is the H x W grid and each (batch, frame) is an independent
 * problem).  The pages give no more; the plainest reading is computed:
 *   y = x + Wo (softmax(q k^T / sqrt(C)) v) + bo,  [q; k; v] = Wqkv n + bqkv,
 *   n = RMS_norm(x) (as in the ResidualBlock, no SiLU), one head of width C.
 *   x, y  : bf16 [B][T][H][W][C] (y may not alias x)
 *   gamma : fp32 [C];  wqkv : bf16 [3C][C] (rows q, k, v);  bqkv : fp32 [3C]
 *           or NULL;  wo : bf16 [C][C];  bo : fp32 [C] or NULL;  eps > 0
 *   workspace : device buffer of wanvae_frame_attention_workspace_size(d, C)
 *           bytes, 256-byte aligned (the normed input, q, k, v, V transposed
 *           and the attention output).
 *   C : 128, 256 or 384.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA. */
size_t wanvae_frame_attention_workspace_size(wanvae_dims d, int64_t c);
wanvae_status wanvae_frame_attention(const void *x, const float *gamma, const void *wqkv,
                                     const float *bqkv, const void *wo, const float *bo, void *y,
                                     wanvae_dims d, int64_t c, float eps, void *workspace,
                                     size_t ws_bytes, wanvae_stream stream);

/* Bytes of device workspace wanvae_resblock_forward needs for these sizes
 * (the bf16 conv inputs a1 and a2, 256-byte aligned).  0 on invalid sizes. */
size_t wanvae_resblock_workspace_size(wanvae_dims d, int64_t c_in, int64_t c_out);

/* The whole ResidualBlock forward.
 *   x : bf16 [B][T][H][W][c_in];  y : bf16 [B][T][H][W][c_out]
 *   cache : NULL for full-T (the whole clip at once, zero causal pad), or a
 *           feat_cache (see wanvae_resblock_cache) for one streaming call of
 *           T frames (T = 1 for frame-by-frame decode).
 *   workspace : device buffer of at least
 *               wanvae_resblock_workspace_size(d, c_in, c_out) bytes, 256-byte
 *               aligned; contents on entry are ignored.
 * Kernels: fused RMS_norm1+SiLU; conv A with RMS_norm2+SiLU fused into its
 * epilogue; conv B with bias, shortcut GEMM and residual add fused into it.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA. */
wanvae_status wanvae_resblock_forward(const wanvae_resblock_params *p, const void *x,
                                      void *y, wanvae_dims d,
                                      const wanvae_resblock_cache *cache,
                                      void *workspace, size_t ws_bytes,
                                      wanvae_stream stream);

/* Same as wanvae_resblock_forward, and records four caller-created CUDA
 * events (cudaEvent_t values passed as void *, host array of 4) on `stream`:
 * [0] before RMS_norm1, [1] before conv A, [2] before conv B, [3] after the
 * last kernel.  Used to time each kernel inside a whole step. */
wanvae_status wanvae_resblock_forward_profiled(const wanvae_resblock_params *p,
                                               const void *x, void *y, wanvae_dims d,
                                               const wanvae_resblock_cache *cache,
                                               void *workspace, size_t ws_bytes,
                                               void *const *events, wanvae_stream stream);

/* Bytes of device workspace wanvae_resblock_forward_host needs: two chunks of
 * x and of y (chunk_T frames each), the two feat_caches, and the block
 * workspace of one chunk.  0 on invalid sizes. */
size_t wanvae_resblock_forward_host_workspace_size(wanvae_dims d, int64_t c_in, int64_t c_out,
                                                   int64_t chunk_T);

/* The whole-clip ResidualBlock forward for a clip held in HOST memory.  The
 * clip runs as consecutive chunks of chunk_T frames carried by the
 * feat_cache ("Sharding of WAN 2.2 VAE", "Why depth sharding is not
 * beneficial": frame-wise decode with a cache of the previous frames), which
 * gives exactly the full-T result, and the chunks are pipelined over three
 * streams: chunk i+1 is copied in on `copy_in` while chunk i computes on
 * `compute` and chunk i-1 is copied out on `copy_out`.
 *   x_host : bf16 [B][T][H][W][c_in], y_host : bf16 [B][T][H][W][c_out], host
 *            memory (page-locked for the copies to overlap; pageable memory
 *            gives the same result without the overlap).
 *   chunk_T : frames per chunk, 1 <= chunk_T (the last chunk may be shorter).
 *   workspace : device buffer of wanvae_resblock_forward_host_workspace_size()
 *            bytes, 256-byte aligned; contents on entry are ignored.
 *   compute, copy_in, copy_out : CUDA streams (may coincide: then nothing
 *            overlaps).  The call returns once everything is enqueued; y_host
 *            is complete when copy_out has drained (synchronise it).  Work
 *            enqueued on copy_in / copy_out before this call is not waited for.
 * Kernels and numerics: those of wanvae_resblock_forward on each chunk.
 * Errors: INVALID_ARG, UNSUPPORTED, MISALIGNED, WORKSPACE, CUDA. */
wanvae_status wanvae_resblock_forward_host(const wanvae_resblock_params *p, const void *x_host,
                                           void *y_host, wanvae_dims d, int64_t chunk_T,
                                           void *workspace, size_t ws_bytes,
                                           wanvae_stream compute, wanvae_stream copy_in,
                                           wanvae_stream copy_out);

/* Size of the library's own device workspace used by
 * wanvae_resblock_forward_static: 32 MiB, enough for one frame-by-frame call
 * (T = 1) of a 384-channel block on a 90 x 160 latent frame. */
#define WANVAE_STATIC_WORKSPACE_BYTES (32u << 20)

/* wanvae_resblock_forward without a caller workspace, for callers that cannot
 * allocate device memory where they run the block (for example a plugin that
 * is handed only its input and output buffers, or a real-time decode loop in
 * which cudaMalloc would synchronise the device).  The source pages have no
 * counterpart: this is a packaging variant, the computation is the same.
 *   The workspace is a 256-byte aligned array of WANVAE_STATIC_WORKSPACE_BYTES
 *   inside the library, one per device, kept until the process exits.  Calls
 *   whose wanvae_resblock_workspace_size() exceeds it return
 *   WANVAE_ERR_WORKSPACE and enqueue nothing.  The call allocates nothing.
 *   The first call on a device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   All calls share the one array and it keeps the last call's contents;
 *   nothing in it needs to start at zero (every byte read is written earlier
 *   in the same call).  Calls that overlap on the GPU (other streams, other
 *   host threads) race on it: serialise them.
 * Errors: as wanvae_resblock_forward. */
wanvae_status wanvae_resblock_forward_static(const wanvae_resblock_params *p, const void *x,
                                             void *y, wanvae_dims d,
                                             const wanvae_resblock_cache *cache,
                                             wanvae_stream stream);

/* Synchronises `stream`, then reads and clears the library's device error
 * word for the current device and returns, in this order of precedence:
 *   WANVAE_ERR_UNDRAINED if a kernel gave up a bounded wait and afterwards
 *     also gave up waiting for its own in-flight TMA copies or MMAs (they may
 *     have completed into memory it no longer owned: do not reuse the context);
 *   WANVAE_ERR_CUDA if a kernel skipped an access its own checks refused (a
 *     misaligned TMA source) or if the stream reports an error;
 *   WANVAE_ERR_TIMEOUT if a kernel gave up a bounded wait and then drained
 *     cleanly (the context stays usable; the outputs of that call are not);
 *   WANVAE_OK otherwise.  Not for the hot path. */
wanvae_status wanvae_sync_status(wanvae_stream stream);

/* Upper bound, in nanoseconds, of every device-side wait in later launches
 * (default 1e9, i.e. one second).  0 makes every bounded wait give up at
 * once, before it looks at its barrier: a deterministic test hook for the
 * timeout path (the cleanup waits after a give-up keep their own bound).
 * Host-side setting, process-wide. */
void wanvae_set_wait_limit_ns(uint64_t ns);

/* Kernel-variant overrides for testing and tuning (process-wide, host-side;
 * no effect on results beyond the summation order of fp32 partial sums).
 * Each argument 0 or 1 forces a choice for later calls; -1 (or any other
 * value) restores the automatic, shape-driven choice:
 *   pair      : 1 = single-CTA conv kernel (cta_group::1) instead of CTA pairs
 *   halo      : 1 = halo tiles, 0 = per-tap im2col tiles (k = 3 convs)
 *   wide      : 1 = 16 x 16 halo patches where they apply, 0 = 16 x 8
 *   narrow    : 1 = the GEMM-plus-stencil kernel for c_out <= 3, 0 = the
 *               implicit GEMM for those layers too
 *   fuse_norm : 1 = the ResidualBlock's RMS_norm1 + SiLU fused into conv A's
 *               halo loads where the plan allows (halo tiles, c_in in one
 *               chunk of 16, 32, 48, 64, 96 or 128 channels; the values are
 *               bit for bit those of the separate pass, the time is longer);
 *               else (the default) a pass of its own
 * A forced choice that cannot run a given shape falls back to one that can. */
void wanvae_set_kernel_variant(int pair, int halo, int wide, int narrow, int fuse_norm);

/* Number of kernels this library has enqueued since load (host counter). */
uint64_t wanvae_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* WANVAE_H */
