/*
 * wanvae_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, fp64 CPU oracle of the Wan 2.2 VAE decoder ResidualBlock
 * forward pass.  Only the tests, the package's smoke check and the bench's
 * CPU-baseline leg may load it; the product path never does.  It shares no
 * code, header, table or helper with the CUDA library.
 *
 * What it computes, and where the pages define it:
 *
 *  - "Sharding of WAN 2.2 VAE", section "Channel sharding (in Megatron
 *    style)": the ResidualBlock is residual(x) + shortcut(x) where residual =
 *    RMS_norm(in) -> SiLU -> CausalConv3d(in,out,3) -> RMS_norm(out) -> SiLU ->
 *    CausalConv3d(out,out,3) and shortcut = CausalConv3d(in,out,1), or Identity
 *    when in_dim == out_dim (op-sequence figure of the same page).  The
 *    shortcut acts on the raw input.
 *  - "Closing the gap: Wan 2.2 14B VAE decoder", section 4 "RMSNorm not
 *    fused": RMS_norm is the channel-wise chain |x| -> square -> sum over
 *    channels -> sqrt -> clamp(eps) -> divide -> times sqrt(D)*gamma.
 *  - Same page, section 2: the causal temporal pad is folded into the halo
 *    exchange, i.e. the 3x3x3 conv pads two leading frames in T (zeros, or the
 *    cached frames) and one element on each side of H and W.
 *  - "Sharding of WAN 2.2 VAE", section "Why depth sharding is not
 *    beneficial": frame-by-frame decode carries a feat_cache holding the last
 *    frames of each CausalConv3d's input.
 *  - Same page, decoder tree: the up blocks end in an upsample2d or an
 *    upsample3d resample whose second module is a conv; "Closing the gap",
 *    section 3, names 3x1x1 conv kernels in the graph.  Nothing else about
 *    them is on the pages, so the plain reading of "upsample + conv" is taken:
 *    upsample2d = nearest 2x in H and W, then a 3x3 conv (zero pad 1, bias);
 *    the temporal half of upsample3d = nearest 2x in T, then a causal 3x1x1
 *    conv (two zero frames before the first, bias).
 *  - "Closing the gap", section 5: the mid-block attention is a spatial
 *    self-attention within each frame (sequence = the H x W grid, batch =
 *    B x T).  Read plainly: RMS_norm, 1x1 q/k/v projections, one head of
 *    softmax(q k^T / sqrt(C)) v, a 1x1 output projection, plus the input.
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes): eps = 1e-12 clamps the L2 norm (F.normalize's default); no norm
 * bias; D is the normalised channel count; kt = 2 is the current frame and
 * kt = 0 is t-2; pads are zeros; the cache holds the two previous frames of
 * each conv's INPUT (post norm+SiLU), zero before frame 0; every conv has a
 * bias.  All arithmetic is IEEE fp64 in the order written below; nothing is
 * rounded to bf16.  Build with -ffp-contract=off so x86 and Arm agree.
 *
 * Layouts: every activation is NDHWC, i.e. [B][T][H][W][C], C fastest.
 * Conv weights are [C_out][kT][kH][kW][C_in]; k = 3 or 1.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define API __attribute__((visibility("default")))

/* ------------------------------------------------------------------ */
/* RMS_norm over channels (+ optional SiLU) of ONE voxel.              */
/* "Closing the gap", section 4: abs -> pow 2 -> sum(channel) -> sqrt  */
/* -> clamp(eps) -> div -> * (sqrt(D) * gamma).  SiLU(z) = z*sigmoid(z)*/
/* = z / (1 + exp(-z)) ("Sharding of WAN 2.2 VAE", block structure).   */
/* ------------------------------------------------------------------ */
static void norm_silu_voxel(const double *x, const double *gamma, int64_t C,
                            double eps, int apply_silu, double *out)
{
    double ss = 0.0;
    for (int64_t c = 0; c < C; ++c) {
        double a = fabs(x[c]);
        ss += a * a;
    }
    double nrm = sqrt(ss);
    if (nrm < eps) nrm = eps; /* clamp(min = eps) on the L2 norm */
    double sqrt_d = sqrt((double)C);
    for (int64_t c = 0; c < C; ++c) {
        double z = x[c] / nrm * (sqrt_d * gamma[c]);
        out[c] = apply_silu ? z / (1.0 + exp(-z)) : z;
    }
}

API void oracle_rms_norm_silu(const double *x, const double *gamma, int64_t n,
                              int64_t C, double eps, int apply_silu, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < n; ++v)
        norm_silu_voxel(x + v * C, gamma, C, eps, apply_silu, out + v * C);
}

/* ------------------------------------------------------------------ */
/* A "field" is the input of one conv for ONE batch element: a block   */
/* of voxels [nT][nH][nW][C] whose first voxel sits at (t0,y0,x0),     */
/* inside a frame of H x W.  Frames t < 0 come from the feat_cache     */
/* ([2][H][W][C], cache frame t+2) or are zero when there is no cache. */
/* field_at returns NULL for every zero (padding) position.            */
/* ------------------------------------------------------------------ */
typedef struct {
    const double *data;
    const unsigned char *valid; /* optional per-voxel mask (window mode) */
    int64_t nT, nH, nW, t0, y0, x0;
    int64_t H, W, C;
    const double *cache;
} field;

static const double *field_at(const field *f, int64_t t, int64_t y, int64_t x)
{
    if (y < 0 || y >= f->H || x < 0 || x >= f->W) return NULL; /* H/W zero pad */
    if (t < 0) {                                               /* causal pad */
        if (f->cache == NULL || t < -2) return NULL;
        return f->cache + (((t + 2) * f->H + y) * f->W + x) * f->C;
    }
    int64_t it = t - f->t0, iy = y - f->y0, ix = x - f->x0;
    if (it < 0 || it >= f->nT || iy < 0 || iy >= f->nH || ix < 0 || ix >= f->nW)
        return NULL; /* outside the clip (t >= T): never read by a causal conv */
    int64_t idx = (it * f->nH + iy) * f->nW + ix;
    if (f->valid && !f->valid[idx]) return NULL;
    return f->data + idx * f->C;
}

/* Weights [Co][taps][Ci] re-indexed to [taps][Ci][Co] so that the     */
/* per-output sums below run over o in the innermost loop; each        */
/* out[o] still receives its terms in (tap, c) order.                  */
static double *transpose_weights(const double *w, int64_t Co, int64_t taps, int64_t Ci)
{
    double *wt = (double *)malloc(sizeof(double) * (size_t)(Co * taps * Ci));
    if (!wt) return NULL;
    for (int64_t o = 0; o < Co; ++o)
        for (int64_t p = 0; p < taps; ++p)
            for (int64_t c = 0; c < Ci; ++c)
                wt[(p * Ci + c) * Co + o] = w[(o * taps + p) * Ci + c];
    return wt;
}

/* CausalConv3d at one output voxel (t,y,x):                           */
/*   out[o] = bias[o] + sum_{kt,kh,kw} sum_c W[o,kt,kh,kw,c] *          */
/*            in(t + kt - (k-1), y + kh - (k-1)/2, x + kw - (k-1)/2, c) */
/* "Sharding of WAN 2.2 VAE": weight [C_out, C_in, kD, kH, kW] (stored  */
/* here channels-last); "Closing the gap" section 2: causal T pad.     */
static void conv_voxel(const field *in, const double *wt, const double *bias,
                       int64_t Ci, int64_t Co, int k, int64_t t, int64_t y,
                       int64_t x, double *acc)
{
    for (int64_t o = 0; o < Co; ++o) acc[o] = bias ? bias[o] : 0.0;
    int64_t half = (k - 1) / 2;
    for (int kt = 0; kt < k; ++kt)
        for (int kh = 0; kh < k; ++kh)
            for (int kw = 0; kw < k; ++kw) {
                const double *a = field_at(in, t + kt - (k - 1), y + kh - half, x + kw - half);
                if (a == NULL) continue; /* zero padding contributes nothing */
                const double *wp = wt + (int64_t)((kt * k + kh) * k + kw) * Ci * Co;
                for (int64_t c = 0; c < Ci; ++c) {
                    double av = a[c];
                    const double *wc = wp + c * Co;
                    for (int64_t o = 0; o < Co; ++o) acc[o] += wc[o] * av;
                }
            }
}

static field full_field(const double *in, const double *cache, int64_t b,
                        int64_t T, int64_t H, int64_t W, int64_t C)
{
    field f;
    f.data = in + b * T * H * W * C;
    f.valid = NULL;
    f.nT = T; f.nH = H; f.nW = W;
    f.t0 = 0; f.y0 = 0; f.x0 = 0;
    f.H = H; f.W = W; f.C = C;
    f.cache = cache ? cache + b * 2 * H * W * C : NULL;
    return f;
}

/* Whole-tensor CausalConv3d, k in {1, 3}.  cache: [B][2][H][W][Ci] or  */
/* NULL (zeros).  Returns 0 on success, -1 on bad arguments / no memory.*/
API int oracle_causal_conv3d(const double *in, const double *w, const double *bias,
                             const double *cache, int64_t B, int64_t T, int64_t H,
                             int64_t W, int64_t Ci, int64_t Co, int k, double *out)
{
    if (k != 1 && k != 3) return -1;
    int64_t taps = (int64_t)k * k * k;
    double *wt = transpose_weights(w, Co, taps, Ci);
    if (!wt) return -1;
    int64_t nvox = B * T * H * W;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t v = 0; v < nvox; ++v) {
        int64_t x = v % W, y = (v / W) % H, t = (v / (W * H)) % T, b = v / (W * H * T);
        field f = full_field(in, cache, b, T, H, W, Ci);
        conv_voxel(&f, wt, bias, Ci, Co, k, t, y, x, out + v * Co);
    }
    free(wt);
    return 0;
}

/* feat_cache update: the new cache is the last two frames of           */
/* concat(old cache (zeros when NULL), in) along T, per batch element.  */
/* ("Sharding of WAN 2.2 VAE", streaming decode: the cache holds the    */
/* last frames of each CausalConv3d's input.)                           */
API void oracle_cache_next(const double *cache, const double *in, int64_t B,
                           int64_t T, int64_t H, int64_t W, int64_t C, double *cache_out)
{
    int64_t fr = H * W * C;
    for (int64_t b = 0; b < B; ++b)
        for (int64_t j = 0; j < 2; ++j) {
            int64_t src_t = T - 2 + j; /* index into concat(cache, in) minus 2 */
            double *dst = cache_out + (b * 2 + j) * fr;
            if (src_t >= 0) {
                memcpy(dst, in + (b * T + src_t) * fr, sizeof(double) * (size_t)fr);
            } else if (cache) {
                memcpy(dst, cache + (b * 2 + (src_t + 2)) * fr, sizeof(double) * (size_t)fr);
            } else {
                memset(dst, 0, sizeof(double) * (size_t)fr);
            }
        }
}

/* Parameters of one ResidualBlock (all fp64, layouts as above).        */
typedef struct {
    int64_t c_in, c_out;
    double eps;
    const double *gamma1, *gamma2; /* [c_in], [c_out] */
    const double *wA, *bA;         /* [c_out][3][3][3][c_in], [c_out] */
    const double *wB, *bB;         /* [c_out][3][3][3][c_out], [c_out] */
    const double *wS, *bS;         /* [c_out][c_in], [c_out]; wS NULL = Identity */
} oracle_params;

/* ResidualBlock forward over a whole clip (full-T when both caches are */
/* NULL; one streaming call otherwise).  cacheA [B][2][H][W][c_in] and  */
/* cacheB [B][2][H][W][c_out] are read, then replaced by their next     */
/* contents.  y: [B][T][H][W][c_out].  Returns 0, or -1 on bad args.    */
API int oracle_resblock_forward(const double *x, const oracle_params *p, int64_t B,
                                int64_t T, int64_t H, int64_t W, double *cacheA,
                                double *cacheB, double *y)
{
    int64_t Ci = p->c_in, Co = p->c_out, nvox = B * T * H * W;
    if ((cacheA == NULL) != (cacheB == NULL)) return -1;
    if (p->wS == NULL && Ci != Co) return -1;
    double *a1 = (double *)malloc(sizeof(double) * (size_t)(nvox * Ci));
    double *h = (double *)malloc(sizeof(double) * (size_t)(nvox * Co));
    double *a2 = (double *)malloc(sizeof(double) * (size_t)(nvox * Co));
    double *r = (double *)malloc(sizeof(double) * (size_t)(nvox * Co));
    int rc = -1;
    if (!a1 || !h || !a2 || !r) goto done;

    /* residual branch: norm1 -> SiLU -> conv A -> norm2 -> SiLU -> conv B */
    oracle_rms_norm_silu(x, p->gamma1, nvox, Ci, p->eps, 1, a1);
    if (oracle_causal_conv3d(a1, p->wA, p->bA, cacheA, B, T, H, W, Ci, Co, 3, h)) goto done;
    oracle_rms_norm_silu(h, p->gamma2, nvox, Co, p->eps, 1, a2);
    if (oracle_causal_conv3d(a2, p->wB, p->bB, cacheB, B, T, H, W, Co, Co, 3, r)) goto done;

    /* shortcut on the raw input, then the residual add */
    if (p->wS) {
        if (oracle_causal_conv3d(x, p->wS, p->bS, NULL, B, T, H, W, Ci, Co, 1, y)) goto done;
        for (int64_t i = 0; i < nvox * Co; ++i) y[i] = r[i] + y[i];
    } else {
        for (int64_t i = 0; i < nvox * Co; ++i) y[i] = r[i] + x[i];
    }

    if (cacheA) {
        size_t nA = (size_t)(B * 2 * H * W * Ci), nB = (size_t)(B * 2 * H * W * Co);
        double *ca = (double *)malloc(sizeof(double) * nA);
        double *cb = (double *)malloc(sizeof(double) * nB);
        if (!ca || !cb) { free(ca); free(cb); goto done; }
        oracle_cache_next(cacheA, a1, B, T, H, W, Ci, ca);
        oracle_cache_next(cacheB, a2, B, T, H, W, Co, cb);
        memcpy(cacheA, ca, sizeof(double) * nA);
        memcpy(cacheB, cb, sizeof(double) * nB);
        free(ca); free(cb);
    }
    rc = 0;
done:
    free(a1); free(h); free(a2); free(r);
    return rc;
}

/* ResidualBlock output at sampled voxels, each recomputed from its     */
/* receptive field (conv B needs a2 on the 3x3x3 causal neighbourhood,  */
/* each of those needs a1 on its own 3x3x3 neighbourhood, so x on       */
/* t-4..t, y-2..y+2, x-2..x+2).  Same arithmetic, in the same order, as */
/* oracle_resblock_forward, so the two agree bit for bit.               */
/*   xwins[i]: x of point i's batch element on frames [t0, t0+nT), rows */
/*         [y0, y0+nH), columns [x0, x0+nW) (win[6*i..6*i+5] = t0, y0,  */
/*         x0, nT, nH, nW), channels c_in; it must cover the point's    */
/*         receptive field clipped to the clip.  cacheA/cacheB: the     */
/*         point's batch element's caches ([2][H][W][C]) as they were   */
/*         at the start of the call, or NULL for full-T (one cache pair */
/*         for all points).  pts: npts (t, y, x) triples, relative to   */
/*         the call's first frame.  out: [npts][c_out].                 */
API int oracle_resblock_points(const double *const *xwins, const int64_t *win, int64_t H,
                               int64_t W, const oracle_params *p, const double *cacheA,
                               const double *cacheB, int64_t npts, const int64_t *pts,
                               double *out)
{
    int64_t Ci = p->c_in, Co = p->c_out;
    if ((cacheA == NULL) != (cacheB == NULL)) return -1;
    if (p->wS == NULL && Ci != Co) return -1;
    double *wtA = transpose_weights(p->wA, Co, 27, Ci);
    double *wtB = transpose_weights(p->wB, Co, 27, Co);
    double *wtS = p->wS ? transpose_weights(p->wS, Co, 1, Ci) : NULL;
    int bad = 0;
    if (!wtA || !wtB || (p->wS && !wtS)) { bad = 1; goto out_free; }

#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int64_t i = 0; i < npts; ++i) {
        int64_t t = pts[3 * i], y = pts[3 * i + 1], x = pts[3 * i + 2];
        const int64_t *wi = win + 6 * i;
        field fx = {xwins[i], NULL, wi[3], wi[4], wi[5], wi[0], wi[1], wi[2], H, W, Ci, NULL};
        /* a1 on the 5x5x5 window t-4..t, y-2..y+2, x-2..x+2 (frames >= 0) */
        double *a1 = (double *)malloc(sizeof(double) * 125 * (size_t)Ci);
        unsigned char va1[125];
        double *a2 = (double *)malloc(sizeof(double) * 27 * (size_t)Co);
        unsigned char va2[27];
        double *hv = (double *)malloc(sizeof(double) * (size_t)Co);
        double *sv = (double *)malloc(sizeof(double) * (size_t)Co);
        if (!a1 || !a2 || !hv || !sv) { bad = 1; free(a1); free(a2); free(hv); free(sv); continue; }
        for (int64_t j = 0; j < 125; ++j) {
            int64_t tt = t - 4 + j / 25, yy = y - 2 + (j / 5) % 5, xx = x - 2 + j % 5;
            const double *src = (tt >= 0) ? field_at(&fx, tt, yy, xx) : NULL;
            va1[j] = src != NULL;
            if (src) norm_silu_voxel(src, p->gamma1, Ci, p->eps, 1, a1 + j * Ci);
            else if (tt >= 0 && yy >= 0 && yy < H && xx >= 0 && xx < W) bad = 1; /* window too small */
        }
        field fa1 = {a1, va1, 5, 5, 5, t - 4, y - 2, x - 2, H, W, Ci, cacheA};
        /* a2 on the 3x3x3 window t-2..t, y-1..y+1, x-1..x+1 (frames >= 0) */
        for (int64_t j = 0; j < 27; ++j) {
            int64_t tt = t - 2 + j / 9, yy = y - 1 + (j / 3) % 3, xx = x - 1 + j % 3;
            va2[j] = tt >= 0 && yy >= 0 && yy < H && xx >= 0 && xx < W;
            if (!va2[j]) continue;
            conv_voxel(&fa1, wtA, p->bA, Ci, Co, 3, tt, yy, xx, hv);
            norm_silu_voxel(hv, p->gamma2, Co, p->eps, 1, a2 + j * Co);
        }
        field fa2 = {a2, va2, 3, 3, 3, t - 2, y - 1, x - 1, H, W, Co, cacheB};
        double *yo = out + i * Co;
        conv_voxel(&fa2, wtB, p->bB, Co, Co, 3, t, y, x, yo);
        const double *xv = field_at(&fx, t, y, x);
        if (!xv) { bad = 1; }
        else if (wtS) {
            conv_voxel(&fx, wtS, p->bS, Ci, Co, 1, t, y, x, sv);
            for (int64_t o = 0; o < Co; ++o) yo[o] = yo[o] + sv[o];
        } else {
            for (int64_t o = 0; o < Co; ++o) yo[o] = yo[o] + xv[o];
        }
        free(a1); free(a2); free(hv); free(sv);
    }
out_free:
    free(wtA); free(wtB); free(wtS);
    return bad ? -1 : 0;
}

/* ------------------------------------------------------------------ */
/* Spatial upsampling of the decoder's up blocks ("Sharding of WAN 2.2 */
/* VAE", decoder tree: WanUpBlock(..., upsample2d); section "Further   */
/* sharding consideration: WanResample": resample[1] carries the conv  */
/* weight).  The pages give no more; the plainest reading taken: each  */
/* frame is upsampled 2x in H and W by nearest neighbour (every pixel  */
/* becomes a 2x2 block), then a 3x3 conv with one pixel of zero pad on */
/* the upsampled grid and a bias.                                      */
/*   in  [B][T][H][W][Ci], w [Co][3][3][Ci], bias [Co]                  */
/*   out [B][T][2H][2W][Co]                                             */
/* ------------------------------------------------------------------ */
API int oracle_upsample2d_conv(const double *in, const double *w, const double *bias,
                               int64_t B, int64_t T, int64_t H, int64_t W, int64_t Ci,
                               int64_t Co, double *out)
{
    if (B < 1 || T < 1 || H < 1 || W < 1 || Ci < 1 || Co < 1) return -1;
    const int64_t H2 = 2 * H, W2 = 2 * W;
    const int64_t nvox = B * T * H2 * W2;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t v = 0; v < nvox; ++v) {
        const int64_t X = v % W2, Y = (v / W2) % H2, bt = v / (W2 * H2);
        double *o = out + v * Co;
        for (int64_t oc = 0; oc < Co; ++oc) {
            double acc = bias ? bias[oc] : 0.0;
            for (int kh = 0; kh < 3; ++kh) {
                const int64_t yy = Y + kh - 1;          /* row of the upsampled grid */
                if (yy < 0 || yy >= H2) continue;       /* zero pad */
                for (int kw = 0; kw < 3; ++kw) {
                    const int64_t xx = X + kw - 1;
                    if (xx < 0 || xx >= W2) continue;
                    /* nearest neighbour: upsampled (yy, xx) is input (yy/2, xx/2) */
                    const double *src = in + ((bt * H + yy / 2) * W + xx / 2) * Ci;
                    const double *wr = w + ((oc * 3 + kh) * 3 + kw) * Ci;
                    for (int64_t c = 0; c < Ci; ++c) acc += wr[c] * src[c];
                }
            }
            o[oc] = acc;
        }
    }
    return 0;
}

/* Temporal half of the decoder's upsample3d ("Sharding of WAN 2.2 VAE", decoder
 * tree: WanUpBlock(..., upsample3d); the graph's 3x1x1 conv kernels, "Closing the
 * gap", conv3d blocking).  The pages give no more, so the plain reading of
 * "upsample + conv": every frame is repeated twice in T (nearest neighbour),
 * then a causal conv with a 3x1x1 kernel -- two zero frames before the first,
 * like every CausalConv3d of the decoder -- and a bias, C_in -> C_out.  This
 * reading is unconfirmed: a 3x1x1 conv to twice the channels whose halves
 * become two output frames would also fit the pages' few words.
 *   in [B][T][H][W][Ci], w [Co][3][Ci] (tap 2 reads the current upsampled
 *   frame, tap 0 the one two before it), bias [Co] or NULL,
 *   out [B][2T][H][W][Co]. */
API int oracle_time_upsample_conv(const double *in, const double *w, const double *bias,
                                  int64_t B, int64_t T, int64_t H, int64_t W, int64_t Ci,
                                  int64_t Co, double *out)
{
    if (B < 1 || T < 1 || H < 1 || W < 1 || Ci < 1 || Co < 1) return -1;
    const int64_t T2 = 2 * T, HW = H * W;
    const int64_t nvox = B * T2 * HW;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t v = 0; v < nvox; ++v) {
        const int64_t pix = v % HW, s = (v / HW) % T2, b = v / (HW * T2);
        double *o = out + v * Co;
        for (int64_t oc = 0; oc < Co; ++oc) {
            double acc = bias ? bias[oc] : 0.0;
            for (int kt = 0; kt < 3; ++kt) {
                const int64_t u = s + kt - 2;   /* frame of the upsampled sequence */
                if (u < 0) continue;            /* causal zero pad */
                /* nearest neighbour: upsampled frame u is input frame u / 2 */
                const double *src = in + ((b * T + u / 2) * HW + pix) * Ci;
                const double *wr = w + (oc * 3 + kt) * Ci;
                for (int64_t c = 0; c < Ci; ++c) acc += wr[c] * src[c];
            }
            o[oc] = acc;
        }
    }
    return 0;
}

/* The decoder's mid-block attention ("Closing the gap: Wan 2.2 14B VAE
 * decoder", section 5: the decoder's one attention block is a spatial
 * self-attention in which, within a frame, every position attends to every
 * other; the sequence is the H x W grid and each (batch, frame) is an
 * independent problem).  The pages give no more, so the plain reading:
 * RMS_norm over channels (the block's norm, without SiLU), 1x1 projections to
 * q, k and v, one head, softmax(q k^T / sqrt(C)) v over the frame's
 * positions, a 1x1 output projection, and the block's input added back.
 *   in [B][T][H][W][C]; gamma [C]; wqkv [3C][C] (rows q, then k, then v);
 *   bqkv [3C]; wo [C][C]; bo [C]; out [B][T][H][W][C] (not aliasing in). */
API int oracle_frame_attention(const double *in, const double *gamma, const double *wqkv,
                               const double *bqkv, const double *wo, const double *bo,
                               int64_t B, int64_t T, int64_t H, int64_t W, int64_t C,
                               double eps, double *out)
{
    if (B < 1 || T < 1 || H < 1 || W < 1 || C < 1) return -1;
    const int64_t n = H * W;
    double *nx = (double *)malloc((size_t)n * C * sizeof(double));
    double *qkv = (double *)malloc((size_t)n * 3 * C * sizeof(double));
    if (!nx || !qkv) {
        free(nx);
        free(qkv);
        return -1;
    }
    const double scale = 1.0 / sqrt((double)C);
    int rc = 0;
    for (int64_t f = 0; f < B * T; ++f) {
        const double *x = in + f * n * C;
        double *y = out + f * n * C;
        oracle_rms_norm_silu(x, gamma, n, C, eps, 0, nx);
        /* q, k, v of every position: qkv[i][r] = b[r] + sum_c w[r][c] nx[i][c] */
#pragma omp parallel for schedule(static)
        for (int64_t i = 0; i < n; ++i)
            for (int64_t r = 0; r < 3 * C; ++r) {
                double acc = bqkv[r];
                for (int64_t c = 0; c < C; ++c) acc += wqkv[r * C + c] * nx[i * C + c];
                qkv[i * 3 * C + r] = acc;
            }
#pragma omp parallel
        {
            double *p = (double *)malloc((size_t)n * sizeof(double));
            double *o = (double *)malloc((size_t)C * sizeof(double));
            if (!p || !o) {
#pragma omp atomic write
                rc = -1;
            }
#pragma omp for schedule(dynamic, 16)
            for (int64_t i = 0; i < n; ++i) {
                if (!p || !o) continue;
                const double *q = qkv + i * 3 * C;
                /* scores against every key of the frame, softmax over them */
                double m = -INFINITY;
                for (int64_t j = 0; j < n; ++j) {
                    const double *k = qkv + j * 3 * C + C;
                    double s = 0.0;
                    for (int64_t c = 0; c < C; ++c) s += q[c] * k[c];
                    p[j] = s * scale;
                    if (p[j] > m) m = p[j];
                }
                double z = 0.0;
                for (int64_t j = 0; j < n; ++j) {
                    p[j] = exp(p[j] - m);
                    z += p[j];
                }
                for (int64_t c = 0; c < C; ++c) o[c] = 0.0;
                for (int64_t j = 0; j < n; ++j) {
                    const double *v = qkv + j * 3 * C + 2 * C;
                    const double a = p[j] / z;
                    for (int64_t c = 0; c < C; ++c) o[c] += a * v[c];
                }
                /* output projection, bias, residual */
                for (int64_t oc = 0; oc < C; ++oc) {
                    double acc = bo[oc];
                    for (int64_t c = 0; c < C; ++c) acc += wo[oc * C + c] * o[c];
                    y[i * C + oc] = x[i * C + oc] + acc;
                }
            }
            free(p);
            free(o);
        }
        if (rc) break;
    }
    free(nx);
    free(qkv);
    return rc;
}

/* Threads the oracle's OpenMP loops will use (1 when built without it). */
API int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
