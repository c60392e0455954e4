// api.cu -- the C ABI declared in include/wanvae.h: argument checks, the
// per-device error word, and the composition of the ResidualBlock
// ("Sharding of WAN 2.2 VAE", ResidualBlock listing: norm1, SiLU, conv A,
// norm2, SiLU, conv B, shortcut, residual add) out of the kernels.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "../../include/wanvae.h"
#include "kernels.h"

using namespace wanvae;

// Device error word: kernels OR error bits into it; wanvae_sync_status reads
// and clears it.
__device__ unsigned g_wanvae_err;

namespace {

std::atomic<uint64_t> g_wait_ns{1000000000ull};
std::atomic<uint64_t> g_launches{0};

struct DeviceState {
    bool ready;
    int num_sms;
    unsigned *err;
};
constexpr int kMaxDevices = 64;
DeviceState g_dev[kMaxDevices];
std::mutex g_dev_mu;

wanvae_status device_state(DeviceState &out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return WANVAE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceState &d = g_dev[dev];
    if (!d.ready) {
        int sms = 0;
        void *p = nullptr;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaGetSymbolAddress(&p, g_wanvae_err) != cudaSuccess)
            return WANVAE_ERR_CUDA;
        d.num_sms = sms;
        d.err = static_cast<unsigned *>(p);
        d.ready = true;
    }
    out = d;
    return WANVAE_OK;
}

wanvae_status make_ctx(LaunchCtx &ctx, wanvae_stream s) {
    DeviceState d;
    const wanvae_status st = device_state(d);
    if (st != WANVAE_OK) return st;
    ctx.stream = reinterpret_cast<cudaStream_t>(s);
    ctx.err = d.err;
    ctx.wait_ns = g_wait_ns.load();
    ctx.num_sms = d.num_sms;
    return WANVAE_OK;
}

wanvae_status from_cuda(cudaError_t e) { return e == cudaSuccess ? WANVAE_OK : WANVAE_ERR_CUDA; }

bool misaligned(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

bool dims_ok(const wanvae_dims &d) {
    if (d.B < 1 || d.T < 1 || d.H < 1 || d.W < 1) return false;
    if (d.H > (1 << 20) || d.W > (1 << 20) || d.T > (1 << 20) || d.B > (1 << 20)) return false;
    const int64_t hw = d.H * d.W;
    if (hw > INT32_MAX) return false;
    const int64_t vox = d.B * d.T * hw;
    return vox > 0 && vox < INT32_MAX;
}

int64_t voxels(const wanvae_dims &d) { return d.B * d.T * d.H * d.W; }

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

}  // namespace

extern "C" {

const char *wanvae_status_string(wanvae_status s) {
    switch (s) {
        case WANVAE_OK: return "ok";
        case WANVAE_ERR_INVALID_ARG: return "invalid argument";
        case WANVAE_ERR_UNSUPPORTED: return "unsupported size";
        case WANVAE_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case WANVAE_ERR_WORKSPACE: return "workspace missing or too small";
        case WANVAE_ERR_CUDA: return "CUDA error";
        case WANVAE_ERR_TIMEOUT: return "device-side wait timed out";
        case WANVAE_ERR_UNDRAINED:
            return "device-side wait timed out and in-flight copies were not drained "
                   "(do not reuse the CUDA context)";
    }
    return "unknown status";
}

int wanvae_version(void) { return 101; }

void wanvae_set_wait_limit_ns(uint64_t ns) { g_wait_ns.store(ns); }

uint64_t wanvae_launch_count(void) { return g_launches.load(); }

void wanvae_set_kernel_variant(int pair, int halo, int wide, int narrow, int fuse_norm) {
    set_kernel_variant(pair, halo, wide, narrow, fuse_norm);
}

wanvae_status wanvae_rmsnorm_silu(const void *x, void *y, const float *gamma, wanvae_dtype dt,
                                  int64_t n_voxels, int64_t C, float eps, wanvae_stream stream) {
    if (!x || !y || !gamma) return WANVAE_ERR_INVALID_ARG;
    if (dt != WANVAE_BF16 && dt != WANVAE_F32) return WANVAE_ERR_INVALID_ARG;
    if (n_voxels < 1 || n_voxels >= INT32_MAX || C < 16 || C % 16 || C > 4096)
        return WANVAE_ERR_INVALID_ARG;
    if (!(eps >= 0.f)) return WANVAE_ERR_INVALID_ARG;
    if (misaligned(x) || misaligned(y) || misaligned(gamma)) return WANVAE_ERR_MISALIGNED;
    const size_t bytes = (size_t)n_voxels * C * (dt == WANVAE_F32 ? 4 : 2);
    if (overlap(x, bytes, y, bytes)) return WANVAE_ERR_INVALID_ARG;
    LaunchCtx ctx;
    const wanvae_status st = make_ctx(ctx, stream);
    if (st != WANVAE_OK) return st;
    g_launches++;
    return from_cuda(launch_rmsnorm_silu(x, y, gamma, dt == WANVAE_F32, n_voxels, (int)C, eps, ctx));
}

wanvae_status wanvae_causal_conv3d(const void *x, const void *w, const float *bias, void *y,
                                   wanvae_dims d, int64_t c_in, int64_t c_out, int k, void *cache,
                                   wanvae_stream stream) {
    if (!x || !w || !y) return WANVAE_ERR_INVALID_ARG;
    if (k != 1 && k != 3) return WANVAE_ERR_INVALID_ARG;
    if (k == 1 && cache) return WANVAE_ERR_INVALID_ARG;
    if (!dims_ok(d) || c_in < 1 || c_out < 1) return WANVAE_ERR_INVALID_ARG;
    // c_out below 16 (a decoder's conv_out to RGB) is padded inside the kernel.
    if (c_in % 16 || (c_out % 16 && c_out > 15) || c_in > 512 || c_out > 512)
        return WANVAE_ERR_UNSUPPORTED;
    if (misaligned(x) || misaligned(w) || misaligned(y) || misaligned(bias) || misaligned(cache))
        return WANVAE_ERR_MISALIGNED;
    const int64_t M = voxels(d);
    const size_t xb = (size_t)M * c_in * 2, yb = (size_t)M * c_out * 2;
    const size_t cb = (size_t)d.B * 2 * d.H * d.W * c_in * 2;
    if (overlap(x, xb, y, yb)) return WANVAE_ERR_INVALID_ARG;
    if (cache && (overlap(cache, cb, y, yb) || overlap(cache, cb, x, xb)))
        return WANVAE_ERR_INVALID_ARG;

    ConvSpec s;
    memset(&s, 0, sizeof(s));
    s.in = x;
    s.cache = cache;
    s.w = w;
    s.bias = bias;
    s.out = y;
    s.B = (int)d.B;
    s.T = (int)d.T;
    s.H = (int)d.H;
    s.W = (int)d.W;
    s.c_in = (int)c_in;
    s.c_out = (int)c_out;
    s.k = k;
    s.epi = kEpiBias;
    if (conv3d_supported(s)) return WANVAE_ERR_UNSUPPORTED;

    LaunchCtx ctx;
    const wanvae_status st = make_ctx(ctx, stream);
    if (st != WANVAE_OK) return st;
    g_launches++;
    cudaError_t e = launch_conv3d(s, ctx);
    if (e == cudaSuccess && cache) {
        g_launches++;
        e = launch_cache_update(cache, x, s.B, s.T, (int64_t)d.H * d.W * c_in * 2, ctx);
    }
    return from_cuda(e);
}

size_t wanvae_upsample2d_workspace_size(int64_t c_in, int64_t c_out) {
    if (c_in < 1 || c_out < 1 || c_in > 4096 || c_out > 4096) return 0;
    return align256((size_t)4 * 4 * c_in * c_out * 2);  // 4 phases x 2 x 2 taps
}

wanvae_status wanvae_upsample2d_conv(const void *x, const void *w, const float *bias, void *y,
                                     wanvae_dims d, int64_t c_in, int64_t c_out,
                                     void *workspace, size_t ws_bytes, wanvae_stream stream) {
    if (!x || !w || !y || !workspace) return WANVAE_ERR_INVALID_ARG;
    if (!dims_ok(d) || c_in < 1 || c_out < 1) return WANVAE_ERR_INVALID_ARG;
    // one double-buffered TMEM accumulator pair per CTA: c_out <= 256
    if (c_in % 16 || c_out % 16 || c_in > 512 || c_out > 256) return WANVAE_ERR_UNSUPPORTED;
    if (misaligned(x) || misaligned(w) || misaligned(y) || misaligned(bias) ||
        misaligned(workspace))
        return WANVAE_ERR_MISALIGNED;
    const size_t need = wanvae_upsample2d_workspace_size(c_in, c_out);
    if (ws_bytes < need) return WANVAE_ERR_WORKSPACE;
    const int64_t M = voxels(d);
    const size_t xb = (size_t)M * c_in * 2, yb = (size_t)M * 4 * c_out * 2;
    if (overlap(x, xb, y, yb) || overlap(workspace, need, y, yb) ||
        overlap(workspace, need, x, xb))
        return WANVAE_ERR_INVALID_ARG;

    ConvSpec s;
    memset(&s, 0, sizeof(s));
    s.in = x;
    s.w = workspace;  // sub-pixel weights [4][c_out][2][2][c_in]
    s.bias = bias;
    s.out = y;
    s.B = (int)d.B;
    s.T = (int)d.T;
    s.H = (int)d.H;
    s.W = (int)d.W;
    s.c_in = (int)c_in;
    s.c_out = (int)c_out;
    s.k = 3;
    s.epi = kEpiBias;
    s.up2d = 1;
    if (conv3d_supported(s)) return WANVAE_ERR_UNSUPPORTED;

    LaunchCtx ctx;
    const wanvae_status st = make_ctx(ctx, stream);
    if (st != WANVAE_OK) return st;
    g_launches++;
    cudaError_t e = launch_expand_up2d_weights(w, workspace, (int)c_out, (int)c_in, ctx);
    if (e == cudaSuccess) {
        g_launches++;
        e = launch_conv3d(s, ctx);
    }
    return from_cuda(e);
}

size_t wanvae_time_upsample_workspace_size(int64_t c_in, int64_t c_out) {
    if (c_in < 1 || c_out < 1 || c_in > 4096 || c_out > 4096) return 0;
    return align256((size_t)2 * 2 * c_in * c_out * 2);  // 2 phases x 2 taps
}

wanvae_status wanvae_time_upsample_conv(const void *x, const void *w, const float *bias, void *y,
                                        wanvae_dims d, int64_t c_in, int64_t c_out,
                                        void *workspace, size_t ws_bytes, wanvae_stream stream) {
    if (!x || !w || !y || !workspace) return WANVAE_ERR_INVALID_ARG;
    if (!dims_ok(d) || c_in < 1 || c_out < 1) return WANVAE_ERR_INVALID_ARG;
    if (c_in % 16 || c_out % 16 || c_in > 512 || c_out > 512) return WANVAE_ERR_UNSUPPORTED;
    if (misaligned(x) || misaligned(w) || misaligned(y) || misaligned(bias) ||
        misaligned(workspace))
        return WANVAE_ERR_MISALIGNED;
    const size_t need = wanvae_time_upsample_workspace_size(c_in, c_out);
    if (ws_bytes < need) return WANVAE_ERR_WORKSPACE;
    const int64_t M = voxels(d);
    const size_t xb = (size_t)M * c_in * 2, yb = (size_t)M * 2 * c_out * 2;
    if (overlap(x, xb, y, yb) || overlap(workspace, need, y, yb) ||
        overlap(workspace, need, x, xb))
        return WANVAE_ERR_INVALID_ARG;

    ConvSpec s;
    memset(&s, 0, sizeof(s));
    s.in = x;
    s.w = workspace;  // phase weights [2][c_out][2][c_in]
    s.bias = bias;
    s.out = y;
    s.B = (int)d.B;
    s.T = (int)d.T;
    s.H = (int)d.H;
    s.W = (int)d.W;
    s.c_in = (int)c_in;
    s.c_out = (int)c_out;
    s.k = 3;
    s.epi = kEpiBias;
    s.up_t = 1;
    if (conv3d_supported(s)) return WANVAE_ERR_UNSUPPORTED;

    LaunchCtx ctx;
    const wanvae_status st = make_ctx(ctx, stream);
    if (st != WANVAE_OK) return st;
    g_launches++;
    cudaError_t e = launch_expand_time_up_weights(w, workspace, (int)c_out, (int)c_in, ctx);
    if (e == cudaSuccess) {
        g_launches++;
        e = launch_conv3d(s, ctx);
    }
    return from_cuda(e);
}

// upsample3d: the temporal half into a [B][2T][H][W][c_mid] slab of the
// workspace, then the spatial upsampler; the two weight sets after it.
size_t wanvae_upsample3d_workspace_size(wanvae_dims d, int64_t c_in, int64_t c_mid,
                                        int64_t c_out) {
    if (!dims_ok(d) || c_in < 1 || c_mid < 1 || c_out < 1 || c_in > 4096 || c_mid > 4096 ||
        c_out > 4096)
        return 0;
    return align256((size_t)voxels(d) * 2 * c_mid * 2) +
           wanvae_time_upsample_workspace_size(c_in, c_mid) +
           wanvae_upsample2d_workspace_size(c_mid, c_out);
}

wanvae_status wanvae_upsample3d(const void *x, const void *w_t, const float *b_t, const void *w_s,
                                const float *b_s, void *y, wanvae_dims d, int64_t c_in,
                                int64_t c_mid, int64_t c_out, void *workspace, size_t ws_bytes,
                                wanvae_stream stream) {
    if (!workspace) return WANVAE_ERR_INVALID_ARG;
    const size_t need = wanvae_upsample3d_workspace_size(d, c_in, c_mid, c_out);
    if (need == 0) return WANVAE_ERR_INVALID_ARG;
    if (ws_bytes < need) return WANVAE_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t mid = align256((size_t)voxels(d) * 2 * c_mid * 2);
    const size_t wt = wanvae_time_upsample_workspace_size(c_in, c_mid);
    wanvae_status st = wanvae_time_upsample_conv(x, w_t, b_t, ws, d, c_in, c_mid, ws + mid, wt,
                                                 stream);
    if (st != WANVAE_OK) return st;
    wanvae_dims d2 = d;
    d2.T = 2 * d.T;
    return wanvae_upsample2d_conv(ws, w_s, b_s, y, d2, c_mid, c_out, ws + mid + wt,
                                  ws_bytes - mid - wt, stream);
}

// Workspace of the attention block: the normed input, q, k, v and the
// attention output ([M][C] bf16 each) and V transposed ([B*T][C][ldn]).
size_t wanvae_frame_attention_workspace_size(wanvae_dims d, int64_t c) {
    if (!dims_ok(d) || c < 1 || c > 4096) return 0;
    const size_t M = (size_t)voxels(d), F = (size_t)(d.B * d.T);
    const size_t ldn = (size_t)frame_attention_ldn((int)(d.H * d.W));
    return 5 * align256(M * c * 2) + align256(F * c * ldn * 2);
}

wanvae_status wanvae_frame_attention(const void *x, const float *gamma, const void *wqkv,
                                     const float *bqkv, const void *wo, const float *bo, void *y,
                                     wanvae_dims d, int64_t c, float eps, void *workspace,
                                     size_t ws_bytes, wanvae_stream stream) {
    if (!x || !gamma || !wqkv || !wo || !y || !workspace) return WANVAE_ERR_INVALID_ARG;
    if (!dims_ok(d) || c < 1 || !(eps > 0.f)) return WANVAE_ERR_INVALID_ARG;
    if (c != 128 && c != 256 && c != 384) return WANVAE_ERR_UNSUPPORTED;
    if (d.H * d.W > (1 << 24)) return WANVAE_ERR_UNSUPPORTED;
    if (misaligned(x) || misaligned(gamma) || misaligned(wqkv) || misaligned(bqkv) ||
        misaligned(wo) || misaligned(bo) || misaligned(y) || misaligned(workspace))
        return WANVAE_ERR_MISALIGNED;
    const size_t need = wanvae_frame_attention_workspace_size(d, c);
    if (ws_bytes < need) return WANVAE_ERR_WORKSPACE;
    const int64_t M = voxels(d);
    const size_t xb = (size_t)M * c * 2;
    if (overlap(x, xb, y, xb) || overlap(workspace, need, x, xb) ||
        overlap(workspace, need, y, xb))
        return WANVAE_ERR_INVALID_ARG;
    const int F = (int)(d.B * d.T), N = (int)(d.H * d.W), C = (int)c;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const size_t slab = align256((size_t)M * c * 2);
    void *nx = ws, *q = ws + slab, *k = ws + 2 * slab, *v = ws + 3 * slab, *o = ws + 4 * slab;
    void *vt = ws + 5 * slab;

    // the four 1x1 projections on the conv kernel: q, k, v of the normed
    // input (bias), and the output projection of o with the input added
    auto spec = [&](const void *in, const void *w, const float *b, void *out, const void *res) {
        ConvSpec s;
        memset(&s, 0, sizeof(s));
        s.in = in;
        s.w = w;
        s.bias = b;
        s.out = out;
        s.resid = res;
        s.B = (int)d.B;
        s.T = (int)d.T;
        s.H = (int)d.H;
        s.W = (int)d.W;
        s.c_in = C;
        s.c_out = C;
        s.k = 1;
        s.epi = res ? kEpiResidual : kEpiBias;
        return s;
    };
    const __nv_bfloat16 *wq = static_cast<const __nv_bfloat16 *>(wqkv);
    const ConvSpec sq = spec(nx, wq, bqkv, q, nullptr);
    const ConvSpec sk = spec(nx, wq + (size_t)C * C, bqkv ? bqkv + C : nullptr, k, nullptr);
    const ConvSpec sv = spec(nx, wq + (size_t)2 * C * C, bqkv ? bqkv + 2 * C : nullptr, v, nullptr);
    const ConvSpec so = spec(o, wo, bo, y, x);
    if (conv3d_supported(sq) || conv3d_supported(so)) return WANVAE_ERR_UNSUPPORTED;

    LaunchCtx ctx;
    const wanvae_status st = make_ctx(ctx, stream);
    if (st != WANVAE_OK) return st;
    g_launches += 7;
    cudaError_t e = launch_rmsnorm(x, nx, gamma, M, C, eps, ctx);
    if (e == cudaSuccess) e = launch_conv3d(sq, ctx);
    if (e == cudaSuccess) e = launch_conv3d(sk, ctx);
    if (e == cudaSuccess) e = launch_conv3d(sv, ctx);
    if (e == cudaSuccess) e = launch_transpose_v(v, vt, F, N, C, ctx);
    if (e == cudaSuccess) e = launch_attention_core(q, k, vt, o, F, N, C, ctx);
    if (e == cudaSuccess) e = launch_conv3d(so, ctx);
    return from_cuda(e);
}

size_t wanvae_resblock_workspace_size(wanvae_dims d, int64_t c_in, int64_t c_out) {
    if (!dims_ok(d) || c_in < 1 || c_out < 1 || c_in > 4096 || c_out > 4096) return 0;
    const size_t M = (size_t)voxels(d);
    return align256(M * c_in * 2) + align256(M * c_out * 2);
}

// check_only: validate every argument and return before enqueuing anything.
static wanvae_status resblock_impl(const wanvae_resblock_params *p, const void *x, void *y,
                                   wanvae_dims d, const wanvae_resblock_cache *cache,
                                   void *workspace, size_t ws_bytes, void *const *events,
                                   wanvae_stream stream, bool check_only = false) {
    if (!p || !x || !y) return WANVAE_ERR_INVALID_ARG;
    if (!p->gamma1 || !p->gamma2 || !p->wA || !p->wB) return WANVAE_ERR_INVALID_ARG;
    if (!dims_ok(d) || p->c_in < 1 || p->c_out < 1) return WANVAE_ERR_INVALID_ARG;
    if (!(p->eps >= 0.f)) return WANVAE_ERR_INVALID_ARG;
    if (!p->wS && p->c_in != p->c_out) return WANVAE_ERR_INVALID_ARG;
    if (!p->wS && p->bS) return WANVAE_ERR_INVALID_ARG;
    if (cache && (!cache->convA_in || !cache->convB_in)) return WANVAE_ERR_INVALID_ARG;
    if (p->c_in % 16 || p->c_out % 16 || p->c_in > 512 || p->c_out > 512)
        return WANVAE_ERR_UNSUPPORTED;
    const void *ptrs[] = {x, y, p->gamma1, p->gamma2, p->wA, p->bA, p->wB, p->bB, p->wS, p->bS,
                          workspace, cache ? cache->convA_in : nullptr,
                          cache ? cache->convB_in : nullptr};
    for (const void *q : ptrs)
        if (misaligned(q)) return WANVAE_ERR_MISALIGNED;

    const int64_t M = voxels(d);
    const size_t xb = (size_t)M * p->c_in * 2, yb = (size_t)M * p->c_out * 2;
    const size_t need = wanvae_resblock_workspace_size(d, p->c_in, p->c_out);
    if (!workspace || ws_bytes < need) return WANVAE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return WANVAE_ERR_MISALIGNED;
    if (overlap(x, xb, y, yb) || overlap(workspace, need, x, xb) || overlap(workspace, need, y, yb))
        return WANVAE_ERR_INVALID_ARG;
    const size_t cab = (size_t)d.B * 2 * d.H * d.W * p->c_in * 2;
    const size_t cbb = (size_t)d.B * 2 * d.H * d.W * p->c_out * 2;
    if (cache) {
        const void *ca = cache->convA_in, *cbp = cache->convB_in;
        if (overlap(ca, cab, cbp, cbb) || overlap(ca, cab, x, xb) || overlap(ca, cab, y, yb) ||
            overlap(cbp, cbb, x, xb) || overlap(cbp, cbb, y, yb) ||
            overlap(ca, cab, workspace, need) || overlap(cbp, cbb, workspace, need))
            return WANVAE_ERR_INVALID_ARG;
    }

    uint8_t *ws = static_cast<uint8_t *>(workspace);
    void *a1 = ws;
    void *a2 = ws + align256((size_t)M * p->c_in * 2);

    ConvSpec sA;
    memset(&sA, 0, sizeof(sA));
    sA.in = a1;
    sA.cache = cache ? cache->convA_in : nullptr;
    sA.w = p->wA;
    sA.bias = p->bA;
    sA.gamma = p->gamma2;
    sA.eps = p->eps;
    sA.out = a2;
    sA.B = (int)d.B;
    sA.T = (int)d.T;
    sA.H = (int)d.H;
    sA.W = (int)d.W;
    sA.c_in = (int)p->c_in;
    sA.c_out = (int)p->c_out;
    sA.k = 3;
    sA.epi = kEpiNormSilu;

    ConvSpec sB = sA;
    sB.in = a2;
    sB.cache = cache ? cache->convB_in : nullptr;
    sB.w = p->wB;
    sB.bias = p->bB;
    sB.gamma = nullptr;
    sB.out = y;
    sB.c_in = (int)p->c_out;
    if (p->wS) {
        sB.epi = kEpiBias;
        sB.bias2 = p->bS;
        sB.sc_in = x;
        sB.sc_w = p->wS;
        sB.c_sc = (int)p->c_in;
    } else {
        sB.epi = kEpiResidual;
        sB.resid = x;
    }
    if (conv3d_supported(sA) || conv3d_supported(sB)) return WANVAE_ERR_UNSUPPORTED;
    // RMS_norm1 + SiLU fused into conv A's halo loads where its plan allows
    // ("Closing the gap", section 4: the norm and the activation in one pass;
    // here that pass is conv A's own input path), else a pass of its own.
    {
        ConvSpec sf = sA;
        sf.in = x;
        sf.norm_in = 1;
        sf.gamma_in = p->gamma1;
        if (conv3d_fuses_norm(sf)) sA = sf;
    }
    const bool fused = sA.norm_in != 0;
    if (check_only) return WANVAE_OK;

    LaunchCtx ctx;
    const wanvae_status st = make_ctx(ctx, stream);
    if (st != WANVAE_OK) return st;
    auto rec = [&](int i) -> cudaError_t {
        return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), ctx.stream)
                      : cudaSuccess;
    };
    const int64_t frA = d.H * d.W * p->c_in * 2, frB = d.H * d.W * p->c_out * 2;
    cudaError_t e = rec(0);
    if (e == cudaSuccess && !fused) {
        g_launches++;
        e = launch_rmsnorm_silu(x, a1, p->gamma1, false, M, (int)p->c_in, p->eps, ctx);
    }
    if (e == cudaSuccess) e = rec(1);
    if (e == cudaSuccess) {
        g_launches++;
        e = launch_conv3d(sA, ctx);
    }
    // The feat_cache updates: conv A's reads the input norm's output (fused:
    // recomputes it from x) and conv B never reads conv A's cache, so without
    // the fused norm both run in one launch after conv B, off the path between
    // the convs.
    if (e == cudaSuccess && cache && fused) {
        g_launches++;
        e = launch_cache_update_norm(cache->convA_in, x, p->gamma1, (int)d.B, (int)d.T,
                                     d.H * d.W, (int)p->c_in, p->eps, ctx);
    }
    if (e == cudaSuccess) e = rec(2);
    if (e == cudaSuccess) {
        g_launches++;
        e = launch_conv3d(sB, ctx);
    }
    if (e == cudaSuccess && cache) {
        g_launches++;
        e = fused ? launch_cache_update(cache->convB_in, a2, (int)d.B, (int)d.T, frB, ctx)
                  : launch_cache_update2(cache->convA_in, a1, frA, cache->convB_in, a2, frB,
                                         (int)d.B, (int)d.T, ctx);
    }
    if (e == cudaSuccess) e = rec(3);
    return from_cuda(e);
}

wanvae_status wanvae_resblock_forward(const wanvae_resblock_params *p, const void *x, void *y,
                                      wanvae_dims d, const wanvae_resblock_cache *cache,
                                      void *workspace, size_t ws_bytes, wanvae_stream stream) {
    return resblock_impl(p, x, y, d, cache, workspace, ws_bytes, nullptr, stream);
}

wanvae_status wanvae_resblock_forward_profiled(const wanvae_resblock_params *p, const void *x,
                                               void *y, wanvae_dims d,
                                               const wanvae_resblock_cache *cache,
                                               void *workspace, size_t ws_bytes,
                                               void *const *events, wanvae_stream stream) {
    if (!events || !events[0] || !events[1] || !events[2] || !events[3])
        return WANVAE_ERR_INVALID_ARG;
    return resblock_impl(p, x, y, d, cache, workspace, ws_bytes, events, stream);
}

// ---------------------------------------------------------------------------
// Whole-clip forward from host memory, chunked in T and pipelined over three
// streams.  Workspace: x chunks [2], y chunks [2], cache A, cache B, then the
// block workspace of one chunk.
namespace {
struct HostPlan {
    int64_t chunk;
    size_t xc, yc, ca, cb, blk, total;
};
bool host_plan(wanvae_dims d, int64_t c_in, int64_t c_out, int64_t chunk_T, HostPlan &hp) {
    if (!dims_ok(d) || c_in < 1 || c_out < 1 || c_in > 4096 || c_out > 4096 || chunk_T < 1)
        return false;
    hp.chunk = chunk_T < d.T ? chunk_T : d.T;
    const size_t fr = (size_t)d.B * hp.chunk * d.H * d.W;  // voxels of one chunk
    hp.xc = align256(fr * c_in * 2);
    hp.yc = align256(fr * c_out * 2);
    hp.ca = align256((size_t)d.B * 2 * d.H * d.W * c_in * 2);
    hp.cb = align256((size_t)d.B * 2 * d.H * d.W * c_out * 2);
    wanvae_dims dc = d;
    dc.T = hp.chunk;
    hp.blk = wanvae_resblock_workspace_size(dc, c_in, c_out);
    if (!hp.blk) return false;
    hp.total = 2 * hp.xc + 2 * hp.yc + hp.ca + hp.cb + hp.blk;
    return true;
}
}  // namespace

size_t wanvae_resblock_forward_host_workspace_size(wanvae_dims d, int64_t c_in, int64_t c_out,
                                                   int64_t chunk_T) {
    HostPlan hp;
    return host_plan(d, c_in, c_out, chunk_T, hp) ? hp.total : 0;
}

wanvae_status wanvae_resblock_forward_host(const wanvae_resblock_params *p, const void *x_host,
                                           void *y_host, wanvae_dims d, int64_t chunk_T,
                                           void *workspace, size_t ws_bytes,
                                           wanvae_stream compute, wanvae_stream copy_in,
                                           wanvae_stream copy_out) {
    if (!p || !x_host || !y_host) return WANVAE_ERR_INVALID_ARG;
    HostPlan hp;
    if (!host_plan(d, p->c_in, p->c_out, chunk_T, hp)) return WANVAE_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < hp.total) return WANVAE_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return WANVAE_ERR_MISALIGNED;
    const int64_t M = voxels(d);
    const size_t xbytes = (size_t)M * p->c_in * 2, ybytes = (size_t)M * p->c_out * 2;
    if (overlap(x_host, xbytes, y_host, ybytes)) return WANVAE_ERR_INVALID_ARG;
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    uint8_t *xb[2] = {ws, ws + hp.xc};
    uint8_t *yb[2] = {ws + 2 * hp.xc, ws + 2 * hp.xc + hp.yc};
    uint8_t *ca = ws + 2 * hp.xc + 2 * hp.yc;
    uint8_t *cb = ca + hp.ca;
    uint8_t *blk = cb + hp.cb;
    wanvae_resblock_cache cache{ca, cb};
    // Every argument the chunk calls will see, checked once before anything
    // is enqueued (the last chunk only differs in T).
    {
        wanvae_dims dc = d;
        dc.T = hp.chunk;
        const wanvae_status st =
            resblock_impl(p, xb[0], yb[0], dc, &cache, blk, hp.blk, nullptr, nullptr, true);
        if (st != WANVAE_OK) return st;
    }
    const cudaStream_t sc = reinterpret_cast<cudaStream_t>(compute);
    const cudaStream_t si = reinterpret_cast<cudaStream_t>(copy_in);
    const cudaStream_t so = reinterpret_cast<cudaStream_t>(copy_out);
    // x_ready[s]: chunk in slot s copied in; x_free[s]: its compute done;
    // y_ready[s]: its output written; y_free[s]: its output copied out.
    cudaEvent_t ev[8] = {};
    for (auto &e : ev)
        if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) {
            for (auto &f : ev)
                if (f) cudaEventDestroy(f);
            return WANVAE_ERR_CUDA;
        }
    cudaEvent_t *x_ready = ev, *x_free = ev + 2, *y_ready = ev + 4, *y_free = ev + 6;
    cudaError_t e = cudaMemsetAsync(ca, 0, hp.ca, sc);  // a new clip: empty caches
    if (e == cudaSuccess) e = cudaMemsetAsync(cb, 0, hp.cb, sc);
    const size_t fx = (size_t)d.H * d.W * p->c_in * 2, fy = (size_t)d.H * d.W * p->c_out * 2;
    wanvae_status st = WANVAE_OK;
    int64_t i = 0;
    for (int64_t t0 = 0; e == cudaSuccess && st == WANVAE_OK && t0 < d.T; t0 += hp.chunk, ++i) {
        const int s = (int)(i & 1);
        const int64_t n = d.T - t0 < hp.chunk ? d.T - t0 : hp.chunk;
        // copy in: the slot is free once the compute of chunk i-2 is done
        if (i >= 2) e = cudaStreamWaitEvent(si, x_free[s], 0);
        for (int64_t b = 0; e == cudaSuccess && b < d.B; ++b)
            e = cudaMemcpyAsync(xb[s] + (size_t)b * n * fx,
                                static_cast<const uint8_t *>(x_host) + ((size_t)b * d.T + t0) * fx,
                                (size_t)n * fx, cudaMemcpyHostToDevice, si);
        if (e == cudaSuccess) e = cudaEventRecord(x_ready[s], si);
        // compute: after its input landed and the y slot was copied out
        if (e == cudaSuccess) e = cudaStreamWaitEvent(sc, x_ready[s], 0);
        if (e == cudaSuccess && i >= 2) e = cudaStreamWaitEvent(sc, y_free[s], 0);
        if (e != cudaSuccess) break;
        wanvae_dims dc = d;
        dc.T = n;
        st = resblock_impl(p, xb[s], yb[s], dc, &cache, blk, hp.blk, nullptr, compute, false);
        if (st != WANVAE_OK) break;
        e = cudaEventRecord(x_free[s], sc);
        if (e == cudaSuccess) e = cudaEventRecord(y_ready[s], sc);
        // copy out
        if (e == cudaSuccess) e = cudaStreamWaitEvent(so, y_ready[s], 0);
        for (int64_t b = 0; e == cudaSuccess && b < d.B; ++b)
            e = cudaMemcpyAsync(static_cast<uint8_t *>(y_host) + ((size_t)b * d.T + t0) * fy,
                                yb[s] + (size_t)b * n * fy, (size_t)n * fy,
                                cudaMemcpyDeviceToHost, so);
        if (e == cudaSuccess) e = cudaEventRecord(y_free[s], so);
    }
    for (auto &f : ev) cudaEventDestroy(f);  // released once the work above completes
    if (st != WANVAE_OK) return st;
    return from_cuda(e);
}

wanvae_status wanvae_sync_status(wanvae_stream stream) {
    DeviceState d;
    const wanvae_status st = device_state(d);
    if (st != WANVAE_OK) return st;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return WANVAE_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_wanvae_err, sizeof(v)) != cudaSuccess) return WANVAE_ERR_CUDA;
    if (v) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_wanvae_err, &zero, sizeof(zero)) != cudaSuccess)
            return WANVAE_ERR_CUDA;
        // bit 0: a bounded device wait gave up; bit 2: so did a later wait for
        // the kernel's own in-flight work; bit 1: a kernel skipped an access
        // its own checks refused
        if (v & 4u) return WANVAE_ERR_UNDRAINED;
        return v == 1u ? WANVAE_ERR_TIMEOUT : WANVAE_ERR_CUDA;
    }
    return WANVAE_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free ResidualBlock forward.
//
// Some callers cannot call cudaMalloc at the point where they run the block:
// a plugin of an inference runtime that is handed only its input and output
// buffers, or a real-time frame-by-frame decode loop where an allocation
// would synchronise the device or is forbidden after start-up.  For them the
// workspace (the bf16 conv inputs a1 and a2) lives in this file-scope device
// array instead of a caller buffer.  Every GPU that loads the library holds
// it until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_wanvae_static_ws[WANVAE_STATIC_WORKSPACE_BYTES];

namespace {
std::mutex g_static_mu;
void *g_static_ws_ptr[kMaxDevices];  // device address of the array, per device

// Host code must not pass the array's name to a kernel (on the host it is a
// stand-in symbol, not a device address); look the device address up once
// per device, with that device current.
wanvae_status static_workspace(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return WANVAE_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ws_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_wanvae_static_ws) != cudaSuccess || !p)
            return WANVAE_ERR_CUDA;
        g_static_ws_ptr[dev] = p;
    }
    *out = g_static_ws_ptr[dev];
    return WANVAE_OK;
}
}  // namespace

extern "C" wanvae_status wanvae_resblock_forward_static(const wanvae_resblock_params *p,
                                                        const void *x, void *y, wanvae_dims d,
                                                        const wanvae_resblock_cache *cache,
                                                        wanvae_stream stream) {
    if (!p) return WANVAE_ERR_INVALID_ARG;
    const size_t need = wanvae_resblock_workspace_size(d, p->c_in, p->c_out);
    if (need == 0) return WANVAE_ERR_INVALID_ARG;
    if (need > (size_t)WANVAE_STATIC_WORKSPACE_BYTES) return WANVAE_ERR_WORKSPACE;
    void *ws = nullptr;
    const wanvae_status st = static_workspace(&ws);
    if (st != WANVAE_OK) return st;
    return resblock_impl(p, x, y, d, cache, ws, (size_t)WANVAE_STATIC_WORKSPACE_BYTES, nullptr,
                         stream);
}
