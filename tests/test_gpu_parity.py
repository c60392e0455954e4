"""GPU parity: every kernel, called through the C ABI, against the fp64 oracle
on the same seeded inputs.  Bar: max|err| <= 2e-2 and relative L2 <= 1e-2
(bf16 in / fp32 accumulate); fp32-mode norm: relative L2 <= 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from _util import compare, sample_points, to_f64
from video_vae_causal_gb300 import synth

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(params=["pair-im2col", "pair-halo", "pair-wide", "single-im2col", "single-halo",
                        "single-wide"])
def variant(request, cuda_lib):
    """Run a conv test on every kernel variant: CTA pair or single CTA, and
    per-tap im2col A loads, halo tiles (16 x 8 patches, one halo load per
    temporal tap feeding the nine spatial taps) or wide halo tiles (16 x 16
    patches, two accumulators per CTA; layers with c_out <= 128 and no
    shortcut, others fall back to 16 x 8)."""
    pair, mode = request.param.split("-")
    cuda_lib.set_kernel_variant(pair=1 if pair == "single" else -1,
                                halo=0 if mode == "im2col" else 1,
                                wide=1 if mode == "wide" else 0)
    yield request.param
    cuda_lib.set_kernel_variant()


def dev(d):
    return {k: v.to(DEV) for k, v in d.items()}


# ------------------------------------------------------------------ norm
@pytest.mark.parametrize("C,n", [(16, 33), (32, 1000), (48, 517), (96, 4099), (192, 2001),
                                 (384, 6241), (4096, 37)])
def test_rmsnorm_silu_bf16(cuda_lib, C, n):
    x = synth.make_tensor((n, C), seed=C + n)
    g = synth.make_tensor((C,), seed=7, dtype=torch.float32, kind="uniform", lo=0.5, hi=1.5)
    y = cuda_lib.rmsnorm_silu(x.to(DEV), g.to(DEV))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.rms_norm_silu(x, g), what=f"norm bf16 C={C}")


@pytest.mark.parametrize("C,n", [(32, 1000), (96, 777), (384, 3001)])
def test_rmsnorm_silu_f32(cuda_lib, C, n):
    x = synth.make_tensor((n, C), seed=C, dtype=torch.float32)
    g = synth.make_tensor((C,), seed=8, dtype=torch.float32, kind="uniform", lo=0.5, hi=1.5)
    y = cuda_lib.rmsnorm_silu(x.to(DEV), g.to(DEV))
    cuda_lib.sync_status()
    ref = oracle.rms_norm_silu(x, g)
    got = to_f64(y)
    rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
    assert rel <= 1e-3, rel
    assert np.max(np.abs(got - ref) / np.maximum(np.abs(ref), 1e-3)) < 1e-3


def test_rmsnorm_zero_voxels_give_zero(cuda_lib):
    x = torch.zeros((64, 32), dtype=torch.bfloat16, device=DEV)
    x[1::2] = 1.0
    g = torch.ones(32, device=DEV)
    y = cuda_lib.rmsnorm_silu(x, g)
    cuda_lib.sync_status()
    assert torch.all(y[0::2] == 0)


# ------------------------------------------------------------------ conv
CONV_CASES = [
    # (B, T, H, W, c_in, c_out): several tiles per frame and a ragged tail
    (1, 3, 12, 20, 64, 64),
    (2, 2, 9, 15, 32, 48),
    (1, 4, 5, 7, 96, 96),
    (1, 2, 16, 16, 384, 384),
    (1, 3, 11, 13, 64, 192),
    (1, 2, 10, 10, 16, 16),
    (1, 1, 3, 200, 128, 96),    # 5 tiles: a CTA pair's second slot is empty
    (1, 4, 5, 7, 64, 32),       # 1 tile per frame: pairs straddle frames t=0|1, 2|3
    (1, 3, 32, 16, 96, 96),     # whole 16x8 and 16x16 patches (the halo modes' own choice)
    (2, 2, 16, 24, 64, 192),
    (1, 2, 32, 40, 64, 64),     # 16x16 patches with a ragged last patch column
    (2, 3, 17, 33, 96, 96),     # ragged in H and W, several patches, two clips
    (1, 3, 12, 20, 16, 384),    # a decoder's conv_in (16 -> 384)
]


def conv_inputs(B, T, H, W, ci, co, k, seed):
    x = synth.make_tensor((B, T, H, W, ci), seed=seed)
    bound = 1.0 / np.sqrt(k * k * k * ci)
    w = synth.make_tensor((co, k, k, k, ci), seed=seed + 1, kind="uniform", lo=-bound, hi=bound)
    b = synth.make_tensor((co,), seed=seed + 2, dtype=torch.float32, kind="uniform", lo=-.1, hi=.1)
    return x, w, b


@pytest.mark.parametrize("case", CONV_CASES)
def test_conv3d_k3_full_clip(cuda_lib, case, variant):
    B, T, H, W, ci, co = case
    x, w, b = conv_inputs(B, T, H, W, ci, co, 3, seed=sum(case))
    y = cuda_lib.causal_conv3d(x.to(DEV), w.to(DEV), b.to(DEV))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.causal_conv3d(x, w, b), what=f"conv3 {case}")


# Narrow outputs (c_out < 16): a decoder's conv_out to RGB and odd widths; N is
# padded inside the kernel and the weight rows past c_out read as zeros.
NARROW_CASES = [
    (1, 3, 12, 20, 96, 3),      # conv_out 96 -> 3, ragged tiles
    (2, 2, 9, 15, 32, 1),
    (1, 3, 32, 32, 64, 13),     # whole 16x16 patches (wide halo tiles)
    (1, 2, 16, 24, 128, 8),
    (2, 4, 17, 33, 48, 4),      # 16-channel weight sub-tiles, ragged patches, two clips
    (1, 2, 16, 16, 16, 2),
]


@pytest.fixture(params=["stencil", "gemm"])
def narrow_path(request, cuda_lib, variant):
    """Layers with c_out <= 3 and k=3 run as one GEMM over all taps plus a
    stencil sum unless the narrow variant is switched off, which sends them to
    the implicit GEMM (on the conv variant the `variant` fixture chose)."""
    pair, mode = variant.split("-")
    cuda_lib.set_kernel_variant(pair=1 if pair == "single" else -1,
                                halo=0 if mode == "im2col" else 1,
                                wide=1 if mode == "wide" else 0,
                                narrow=1 if request.param == "stencil" else 0)
    yield request.param
    cuda_lib.set_kernel_variant()


@pytest.mark.parametrize("case", NARROW_CASES)
def test_conv3d_k3_narrow_output(cuda_lib, case, variant, narrow_path):
    B, T, H, W, ci, co = case
    x, w, b = conv_inputs(B, T, H, W, ci, co, 3, seed=70 + sum(case))
    y = cuda_lib.causal_conv3d(x.to(DEV), w.to(DEV), b.to(DEV))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.causal_conv3d(x, w, b), what=f"conv3 narrow {case}")


def test_conv3d_narrow_with_cache_and_k1(cuda_lib, variant, narrow_path):
    B, T, H, W, ci, co = 1, 2, 9, 14, 64, 3
    x, w, b = conv_inputs(B, T, H, W, ci, co, 3, seed=80)
    cache = synth.make_tensor((B, 2, H, W, ci), seed=81)
    cache_d = cache.to(DEV)
    y = cuda_lib.causal_conv3d(x.to(DEV), w.to(DEV), b.to(DEV), cache=cache_d)
    x1, w1, b1 = conv_inputs(1, 2, 7, 9, 16, 5, 1, seed=82)
    y1 = cuda_lib.causal_conv3d(x1.to(DEV), w1.to(DEV), b1.to(DEV))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.causal_conv3d(x, w, b, cache=cache), what="conv3 narrow cache")
    assert np.array_equal(to_f64(cache_d), oracle.cache_next(cache, x))
    compare(to_f64(y1), oracle.causal_conv3d(x1, w1, b1), what="conv1 narrow")


@pytest.mark.parametrize("case", [(1, 3, 12, 20, 64, 64), (2, 2, 9, 15, 32, 48),
                                  (1, 2, 7, 9, 384, 192)])
def test_conv3d_k1(cuda_lib, case, variant):
    B, T, H, W, ci, co = case
    x, w, b = conv_inputs(B, T, H, W, ci, co, 1, seed=5 + sum(case))
    y = cuda_lib.causal_conv3d(x.to(DEV), w.to(DEV), b.to(DEV))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.causal_conv3d(x, w, b), what=f"conv1 {case}")


@pytest.mark.parametrize("T", [1, 2, 3])
def test_conv3d_with_cache_reads_and_updates_cache(cuda_lib, T, variant):
    B, H, W, ci, co = 2, 9, 14, 64, 32
    x, w, b = conv_inputs(B, T, H, W, ci, co, 3, seed=40 + T)
    cache = synth.make_tensor((B, 2, H, W, ci), seed=50 + T)
    cache_d = cache.to(DEV)
    y = cuda_lib.causal_conv3d(x.to(DEV), w.to(DEV), b.to(DEV), cache=cache_d)
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.causal_conv3d(x, w, b, cache=cache), what=f"conv3 cache T={T}")
    assert np.array_equal(to_f64(cache_d), oracle.cache_next(cache, x))


def test_conv3d_no_bias_and_output_guard_bands(cuda_lib):
    B, T, H, W, ci, co = 1, 2, 9, 11, 32, 32
    x, w, _ = conv_inputs(B, T, H, W, ci, co, 3, seed=60)
    n = B * T * H * W * co
    guard = 4096
    buf = torch.full((n + 2 * guard,), 12345.0, dtype=torch.bfloat16, device=DEV)
    y = buf[guard:guard + n].view(B, T, H, W, co)
    cuda_lib.causal_conv3d(x.to(DEV), w.to(DEV), None, y=y)
    cuda_lib.sync_status()
    assert torch.all(buf[:guard] == 12345.0) and torch.all(buf[guard + n:] == 12345.0)
    compare(to_f64(y), oracle.causal_conv3d(x, w, np.zeros(co)), what="conv no bias")


# ------------------------------------------------------------------ upsampler
UP_CASES = [
    # (B, T, H, W, c_in, c_out) at the low resolution; output is 2H x 2W
    (1, 2, 5, 7, 32, 16),       # ragged tiles
    (2, 1, 8, 12, 64, 32),
    (1, 3, 16, 16, 96, 48),
    (1, 1, 9, 13, 192, 96),     # the decoder's 192 -> 96 channels
]


@pytest.mark.parametrize("case", UP_CASES)
def test_upsample2d_conv(cuda_lib, case, variant):
    B, T, H, W, ci, co = case
    x = synth.make_tensor((B, T, H, W, ci), seed=100 + sum(case))
    bound = 1.0 / np.sqrt(9 * ci)
    w = synth.make_tensor((co, 3, 3, ci), seed=101 + sum(case), kind="uniform", lo=-bound,
                          hi=bound)
    b = synth.make_tensor((co,), seed=102, dtype=torch.float32, kind="uniform", lo=-.1, hi=.1)
    y = cuda_lib.upsample2d_conv(x.to(DEV), w.to(DEV), b.to(DEV))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.upsample2d_conv(x, w, b), what=f"upsample2d {case}")


# --------------------------------------------------------- temporal upsampler
TIME_UP_CASES = [
    # (B, T, H, W, c_in, c_out); output is 2T frames
    (1, 1, 5, 7, 32, 16),       # one frame: both phases read the causal zero frame
    (2, 3, 6, 9, 64, 32),       # two clips: frame t - 1 never crosses into the other
    (1, 4, 8, 16, 96, 48),
    (1, 2, 9, 13, 384, 384),    # the first up block's 384 channels (one accumulator)
]


@pytest.mark.parametrize("case", TIME_UP_CASES)
def test_time_upsample_conv(cuda_lib, case, variant):
    B, T, H, W, ci, co = case
    x = synth.make_tensor((B, T, H, W, ci), seed=200 + sum(case))
    bound = 1.0 / np.sqrt(3 * ci)
    w = synth.make_tensor((co, 3, ci), seed=201 + sum(case), kind="uniform", lo=-bound,
                          hi=bound)
    b = synth.make_tensor((co,), seed=202, dtype=torch.float32, kind="uniform", lo=-.1, hi=.1)
    y = cuda_lib.time_upsample_conv(x.to(DEV), w.to(DEV), b.to(DEV))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.time_upsample_conv(x, w, b), what=f"time upsample {case}")


def test_upsample3d(cuda_lib):
    """The composite (time then space) against the oracle's upsample3d."""
    B, T, H, W, ci, cm, co = 1, 2, 6, 9, 64, 64, 32
    x = synth.make_tensor((B, T, H, W, ci), seed=400)
    bt_ = 1.0 / np.sqrt(3 * ci)
    w_t = synth.make_tensor((cm, 3, ci), seed=401, kind="uniform", lo=-bt_, hi=bt_)
    b_t = synth.make_tensor((cm,), seed=402, dtype=torch.float32, kind="uniform", lo=-.1, hi=.1)
    bs_ = 1.0 / np.sqrt(9 * cm)
    w_s = synth.make_tensor((co, 3, 3, cm), seed=403, kind="uniform", lo=-bs_, hi=bs_)
    b_s = synth.make_tensor((co,), seed=404, dtype=torch.float32, kind="uniform", lo=-.1, hi=.1)
    y = cuda_lib.upsample3d(x.to(DEV), w_t.to(DEV), b_t.to(DEV), w_s.to(DEV), b_s.to(DEV))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.upsample3d(x, w_t, b_t, w_s, b_s), what="upsample3d")
# ------------------------------------------------------- mid-block attention
ATTN_CASES = [
    # (B, T, H, W, C): N = H*W positions per frame
    (1, 2, 4, 8, 128),          # one partial key block, one query tile
    (2, 1, 12, 16, 256),        # two clips, N = 192: a ragged second block
    (1, 2, 10, 13, 384),        # N = 130: two query tiles, the second of 2 rows
    (1, 1, 20, 30, 384),        # N = 600: five key blocks
]


@pytest.mark.parametrize("case", ATTN_CASES)
def test_frame_attention(cuda_lib, case):
    B, T, H, W, C = case
    s = sum(case)
    x = synth.make_tensor((B, T, H, W, C), seed=300 + s)
    g = synth.make_tensor((C,), seed=301, dtype=torch.float32, kind="uniform", lo=0.5, hi=1.5)
    bw = 1.0 / np.sqrt(C)
    wqkv = synth.make_tensor((3 * C, C), seed=302 + s, kind="uniform", lo=-bw, hi=bw)
    bqkv = synth.make_tensor((3 * C,), seed=303, dtype=torch.float32, kind="uniform",
                             lo=-.1, hi=.1)
    wo = synth.make_tensor((C, C), seed=304 + s, kind="uniform", lo=-bw, hi=bw)
    bo = synth.make_tensor((C,), seed=305, dtype=torch.float32, kind="uniform", lo=-.1, hi=.1)
    y = cuda_lib.frame_attention(x.to(DEV), g.to(DEV), wqkv.to(DEV), bqkv.to(DEV), wo.to(DEV),
                                 bo.to(DEV))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.frame_attention(x, g, wqkv, bqkv, wo, bo),
            what=f"attention {case}")


def _attn_inputs(B, T, H, W, C, seed):
    x = synth.make_tensor((B, T, H, W, C), seed=seed)
    g = synth.make_tensor((C,), seed=seed + 1, dtype=torch.float32, kind="uniform", lo=0.5,
                          hi=1.5)
    bw = 1.0 / np.sqrt(C)
    wqkv = synth.make_tensor((3 * C, C), seed=seed + 2, kind="uniform", lo=-bw, hi=bw)
    bqkv = synth.make_tensor((3 * C,), seed=seed + 3, dtype=torch.float32, kind="uniform",
                             lo=-.1, hi=.1)
    wo = synth.make_tensor((C, C), seed=seed + 4, kind="uniform", lo=-bw, hi=bw)
    bo = synth.make_tensor((C,), seed=seed + 5, dtype=torch.float32, kind="uniform", lo=-.1,
                           hi=.1)
    return x, g, wqkv, bqkv, wo, bo


def test_frame_attention_uniform_when_q_k_vanish(cuda_lib):
    """Zero q and k projections: every score is 0, so each query's output is
    the mean of v over its frame (closed form: x + bo + Wo mean(v)), across
    several key blocks and a ragged last one."""
    x, g, wqkv, bqkv, wo, bo = _attn_inputs(1, 2, 12, 25, 128, seed=310)
    C = 128
    wqkv[:2 * C] = 0
    bqkv[:2 * C] = 0
    y = cuda_lib.frame_attention(x.to(DEV), g.to(DEV), wqkv.to(DEV), bqkv.to(DEV), wo.to(DEV),
                                 bo.to(DEV))
    cuda_lib.sync_status()
    ref = oracle.frame_attention(x, g, wqkv, bqkv, wo, bo)
    compare(to_f64(y), ref, what="attention uniform")
    # the closed form itself, per frame
    xf = to_f64(x).reshape(2, -1, C)
    n = xf / np.maximum(np.linalg.norm(xf, axis=2, keepdims=True), 1e-12) * np.sqrt(C) * \
        to_f64(g)
    v = n @ to_f64(wqkv[2 * C:]).T + to_f64(bqkv[2 * C:])
    closed = xf + to_f64(bo) + v.mean(axis=1, keepdims=True) @ to_f64(wo).T
    compare(to_f64(y).reshape(2, -1, C), closed, what="attention uniform closed form")


def test_frame_attention_single_position(cuda_lib):
    """One position per frame: its only key gets all the weight, so
    y = x + bo + Wo v (a 1 x 1 frame: one ragged query tile and key block)."""
    x, g, wqkv, bqkv, wo, bo = _attn_inputs(2, 3, 1, 1, 256, seed=320)
    y = cuda_lib.frame_attention(x.to(DEV), g.to(DEV), wqkv.to(DEV), bqkv.to(DEV), wo.to(DEV),
                                 bo.to(DEV))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.frame_attention(x, g, wqkv, bqkv, wo, bo),
            what="attention one position")


# ------------------------------------------------------------------ block
BLOCK_CASES = [
    # (B, T, H, W, c_in, c_out)
    (1, 3, 16, 16, 32, 32),     # the 'tiny' workload
    (1, 5, 20, 24, 64, 64),
    (2, 3, 10, 13, 64, 32),     # channel-reducing, 1x1x1 shortcut
    (1, 3, 10, 12, 384, 384),
    (1, 2, 8, 8, 384, 192),
    (1, 4, 9, 11, 96, 96),
    (1, 1, 1, 1, 32, 32),       # one voxel: every spatial/temporal tap but one is padding
    (1, 3, 9, 11, 64, 64),      # odd tile count, pairs straddle frames
]


def block_inputs(case, seed):
    B, T, H, W, ci, co = case
    return synth.make_resblock_inputs((B, T, H, W), ci, co, seed=seed)


@pytest.mark.parametrize("case", BLOCK_CASES)
def test_resblock_fullT(cuda_lib, case, variant):
    x, p = block_inputs(case, seed=0)
    y = cuda_lib.resblock_forward(x.to(DEV), dev(p))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.resblock_forward(x, oracle.Params.from_dict(p)),
            what=f"block {case}")


def test_resblock_with_shortcut_and_equal_channels(cuda_lib):
    x, p = synth.make_resblock_inputs((1, 3, 9, 10), 64, 64, seed=3, shortcut=True)
    y = cuda_lib.resblock_forward(x.to(DEV), dev(p))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.resblock_forward(x, oracle.Params.from_dict(p)), what="block wS")


@pytest.mark.parametrize("case,chunks", [((1, 6, 12, 14, 64, 64), [1] * 6),
                                         ((2, 5, 9, 10, 64, 32), [2, 2, 1]),
                                         ((1, 4, 8, 8, 384, 384), [1, 3])])
def test_resblock_streaming_equals_fullT(cuda_lib, case, chunks, variant):
    B, T, H, W, ci, co = case
    x, p = block_inputs(case, seed=11)
    xd, pd = x.to(DEV), dev(p)
    full = cuda_lib.resblock_forward(xd, pd)
    cA = torch.zeros((B, 2, H, W, ci), dtype=torch.bfloat16, device=DEV)
    cB = torch.zeros((B, 2, H, W, co), dtype=torch.bfloat16, device=DEV)
    outs, t0 = [], 0
    for n in chunks:
        outs.append(cuda_lib.resblock_forward(xd[:, t0:t0 + n].contiguous(), pd, cache=(cA, cB)))
        t0 += n
    stream = torch.cat(outs, dim=1)
    cuda_lib.sync_status()
    # Same rounding points and accumulation order in both modes: bit-exact.
    assert torch.equal(stream, full)
    compare(to_f64(stream), oracle.resblock_forward(x, oracle.Params.from_dict(p)),
            what=f"stream {case}")


def test_resblock_deterministic(cuda_lib):
    x, p = block_inputs((1, 4, 16, 20, 64, 64), seed=12)
    xd, pd = x.to(DEV), dev(p)
    y1 = cuda_lib.resblock_forward(xd, pd)
    y2 = cuda_lib.resblock_forward(xd, pd)
    cuda_lib.sync_status()
    assert torch.equal(y1, y2)


def test_resblock_causal_on_gpu(cuda_lib):
    case = (1, 5, 8, 12, 64, 64)
    x, p = block_inputs(case, seed=13)
    pd = dev(p)
    y = cuda_lib.resblock_forward(x.to(DEV), pd)
    x2 = x.clone()
    x2[:, 3:] = synth.make_tensor(x2[:, 3:].shape, seed=99)
    y2 = cuda_lib.resblock_forward(x2.to(DEV), pd)
    cuda_lib.sync_status()
    assert torch.equal(y[:, :3], y2[:, :3])


# ------------------------------------------------------------------ norm1 fused into conv A
FUSE_CASES = [
    # (B, T, H, W, c): one chunk holds all c channels, halo tiles
    (1, 2, 16, 16, 32),         # the smallest: 32-channel planes, one 16 x 16 patch
    (1, 4, 32, 32, 96),         # the full-resolution block's 96 channels
    (2, 3, 17, 24, 64),         # 64-channel swizzled rows, ragged patches, two clips
    (1, 3, 16, 24, 48),         # three 16-channel sub-tiles
    (1, 2, 16, 16, 128),        # two 64-channel regions
]


@pytest.mark.parametrize("case", FUSE_CASES)
@pytest.mark.parametrize("mode", ["pair-wide", "pair-halo", "single-halo"])
def test_fused_norm_equals_separate_pass(cuda_lib, case, mode):
    """RMS_norm1 + SiLU applied in conv A's halo loads gives the block output
    of the separate norm pass bit for bit (same arithmetic), full-T and frame
    by frame over the feat_cache, and matches the oracle."""
    B, T, H, W, C = case
    pair, tiles = mode.split("-")
    x, p = synth.make_resblock_inputs((B, T, H, W), C, C, seed=31)
    xd, pd = x.to(DEV), dev(p)
    outs = {}
    try:
        for fuse in (0, 1):
            cuda_lib.set_kernel_variant(pair=1 if pair == "single" else -1, halo=1,
                                        wide=1 if tiles == "wide" else 0, fuse_norm=fuse)
            full = cuda_lib.resblock_forward(xd, pd)
            cA = torch.zeros((B, 2, H, W, C), dtype=torch.bfloat16, device=DEV)
            cB = torch.zeros((B, 2, H, W, C), dtype=torch.bfloat16, device=DEV)
            frames = [cuda_lib.resblock_forward(xd[:, t:t + 1].contiguous(), pd, cache=(cA, cB))
                      for t in range(T)]
            cuda_lib.sync_status()
            outs[fuse] = (full, torch.cat(frames, dim=1), cA.clone())
    finally:
        cuda_lib.set_kernel_variant()
    ref = oracle.resblock_forward(x, oracle.Params.from_dict(p))
    compare(to_f64(outs[1][0]), ref, what=f"fused {case} {mode}")
    compare(to_f64(outs[0][0]), ref, what=f"separate {case} {mode}")
    d = (outs[1][0].float() - outs[0][0].float()).abs().max().item()
    assert torch.equal(outs[1][0], outs[0][0]), f"fused full-T differs from the separate pass by {d}"
    assert torch.equal(outs[1][1], outs[1][0]), "fused streaming differs from fused full-T"
    assert torch.equal(outs[1][2], outs[0][2]), "fused feat_cache differs"


# ------------------------------------------------------------------ host buffers, pipelined
@pytest.mark.parametrize("case,chunk", [((1, 7, 16, 24, 64, 64), 3),     # ragged last chunk
                                        ((2, 5, 9, 10, 64, 32), 2),      # two clips, 1x1x1 shortcut
                                        ((1, 4, 16, 16, 96, 96), 1),     # frame by frame
                                        ((1, 3, 10, 12, 384, 384), 8)])  # one chunk
def test_resblock_forward_host_equals_fullT(cuda_lib, case, chunk):
    """The clip in host memory, chunked in T over the feat_cache and pipelined
    over three streams, gives the full-T result bit for bit."""
    B, T, H, W, ci, co = case
    x, p = block_inputs(case, seed=17)
    pd = dev(p)
    full = cuda_lib.resblock_forward(x.to(DEV), pd)
    x_host = x.pin_memory()
    y_host = torch.full((B, T, H, W, co), 7.0, dtype=torch.bfloat16).pin_memory()
    n = cuda_lib.resblock_forward_host_workspace_size((B, T, H, W), ci, co, chunk)
    ws = torch.empty(n, dtype=torch.uint8, device=DEV)
    streams = (torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream())
    cuda_lib.resblock_forward_host(x_host, pd, y_host, chunk, ws, streams)
    streams[2].synchronize()
    cuda_lib.sync_status()
    assert torch.equal(y_host, full.cpu())


# ------------------------------------------------------------------ closed form at x = 0
@pytest.mark.parametrize("ci,co", [(96, 96), (384, 384), (64, 32)])
def test_resblock_zero_input_closed_form(cuda_lib, ci, co):
    """x = 0 and bA = 0: a1 = 0, h = 0, so conv A's fused RMS_norm2 divides a
    zero vector by the eps clamp (a2 = 0) and y = bB (+ bS) exactly.  With bA
    drawn as usual, h = bA at every voxel and y follows the oracle (pinned by
    the closed form on the CPU)."""
    B, T, H, W = 1, 4, 16, 24
    _, p = synth.make_resblock_inputs((B, T, H, W), ci, co, seed=21)
    x = torch.zeros((B, T, H, W, ci), dtype=torch.bfloat16)
    y = cuda_lib.resblock_forward(x.to(DEV), dev(p))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.resblock_forward(x, oracle.Params.from_dict(p)), what="x=0")
    p0 = dict(p, bA=torch.zeros_like(p["bA"]))
    y0 = cuda_lib.resblock_forward(x.to(DEV), dev(p0))
    cuda_lib.sync_status()
    expect = p["bB"] + (p["bS"] if "bS" in p else 0)
    assert torch.equal(y0.cpu(), expect.to(torch.bfloat16).expand(B, T, H, W, co))


# ------------------------------------------------------------------ full sizes, whole tensor
def test_latent_fullT_whole_tensor(cuda_lib):
    """Every output element of the latent-resolution block [1,21,60,104,384]
    against the oracle's full-T run (about 20 s of oracle time)."""
    dims, ci, co, _ = synth.WORKLOADS["latent_fullT"]
    x, p = synth.make_resblock_inputs(dims, ci, co, seed=0)
    y = cuda_lib.resblock_forward(x.to(DEV), dev(p))
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.resblock_forward(x, oracle.Params.from_dict(p)),
            what="latent_fullT whole")


def test_streaming_720p_whole_tensor(cuda_lib):
    """The streaming workload's 21 calls of [1,1,90,160,384] with feat_cache:
    bit-exact against the full-T run, whose every element is compared with
    the oracle's full-T run (about 45 s of oracle time)."""
    dims, ci, co, calls = synth.WORKLOADS["stream_720p"]
    B, T, H, W = dims
    x, p = synth.make_resblock_inputs(dims, ci, co, seed=0)
    xd, pd = x.to(DEV), dev(p)
    cA = torch.zeros((B, 2, H, W, ci), dtype=torch.bfloat16, device=DEV)
    cB = torch.zeros((B, 2, H, W, co), dtype=torch.bfloat16, device=DEV)
    ws = cuda_lib.make_workspace((B, 1, H, W), ci, co)
    y = torch.cat([cuda_lib.resblock_forward(xd[:, t:t + 1].contiguous(), pd, cache=(cA, cB),
                                             workspace=ws) for t in range(calls)], dim=1)
    full = cuda_lib.resblock_forward(xd, pd)
    cuda_lib.sync_status()
    assert torch.equal(y, full)
    compare(to_f64(full), oracle.resblock_forward(x, oracle.Params.from_dict(p)),
            what="stream_720p whole")


HALO_IM2COL_SAME = [
    # (c_in = c_out, B, T, H, W): frames whose 16 x 8 patches are ragged, so
    # that one-frame calls pick halo tiles and longer calls im2col tiles
    (384, 1, 2, 20, 24),
    (192, 1, 2, 18, 40),
    (96, 2, 1, 20, 16),
]


@pytest.mark.parametrize("c,B,T,H,W", HALO_IM2COL_SAME)
def test_halo_and_im2col_tiles_give_the_same_bits(cuda_lib, c, B, T, H, W):
    """im2col tiles walk each temporal tap chunk by chunk, the nine spatial taps
    within a chunk, which is the halo tiles' order: with the same channel
    chunks both tilings add the same products in the same order, so the block
    gives the same bits either way.  This is what lets a frame-by-frame call
    take halo tiles on a ragged frame while the whole clip takes im2col ones
    (and stay bit-exact with it)."""
    dims = (B, T, H, W)
    x, p = synth.make_resblock_inputs(dims, c, c, seed=11, device=DEV)
    outs = []
    try:
        for halo in (1, 0):
            cuda_lib.set_kernel_variant(halo=halo, wide=0)
            outs.append(cuda_lib.resblock_forward(x, p))
            cuda_lib.sync_status()
    finally:
        cuda_lib.set_kernel_variant()
    assert torch.equal(outs[0], outs[1])


STREAM_RAGGED = [
    # (c, B, T, H, W): frames whose 16 x 8 patches are ragged, decoded frame by
    # frame (halo tiles, two producers) and whole (im2col tiles)
    (384, 2, 4, 20, 24),
    (96, 2, 3, 18, 40),
]


@pytest.mark.parametrize("c,B,T,H,W", STREAM_RAGGED)
def test_streaming_ragged_frames_bit_exact(cuda_lib, c, B, T, H, W):
    """Frame-by-frame decode of a batch of two on ragged frames, where each
    one-frame call takes halo tiles and the whole clip im2col tiles: the same
    bits, frame by frame and in the caches, and the oracle's values."""
    dims = (B, T, H, W)
    x, p = synth.make_resblock_inputs(dims, c, c, seed=23)
    xd, pd = x.to(DEV), dev(p)
    cA = torch.zeros((B, 2, H, W, c), dtype=torch.bfloat16, device=DEV)
    cB = torch.zeros((B, 2, H, W, c), dtype=torch.bfloat16, device=DEV)
    ws = cuda_lib.make_workspace((B, 1, H, W), c, c)
    y = torch.cat([cuda_lib.resblock_forward(xd[:, t:t + 1].contiguous(), pd, cache=(cA, cB),
                                             workspace=ws) for t in range(T)], dim=1)
    full = cuda_lib.resblock_forward(xd, pd)
    cuda_lib.sync_status()
    assert torch.equal(y, full)
    compare(to_f64(full), oracle.resblock_forward(x, oracle.Params.from_dict(p)),
            what="streaming ragged")


# ------------------------------------------------------------------ full sizes, sampled
FULL = [
    ("latent_fullT", 48),
    ("reduce_384_192", 24),
    ("fullres_96", 48),
]


@pytest.mark.parametrize("name,nrand", FULL)
def test_full_size_sampled(cuda_lib, name, nrand):
    dims, ci, co, _ = synth.WORKLOADS[name]
    B, T, H, W = dims
    x, p = synth.make_resblock_inputs(dims, ci, co, seed=0, device=DEV)
    y = cuda_lib.resblock_forward(x, p)
    cuda_lib.sync_status()
    pts = sample_points(T, H, W, nrand, seed=1)
    op = oracle.Params.from_dict(p)
    ref = oracle.resblock_points(x, op, pts)
    idx = torch.tensor(pts, device=DEV)
    got = y[0, idx[:, 0], idx[:, 1], idx[:, 2]]
    compare(to_f64(got), ref, what=name)
    assert torch.isfinite(y).all()


def test_streaming_720p_21_calls_sampled(cuda_lib):
    dims, ci, co, calls = synth.WORKLOADS["stream_720p"]
    B, T, H, W = dims
    x, p = synth.make_resblock_inputs(dims, ci, co, seed=0, device=DEV)
    cA = torch.zeros((B, 2, H, W, ci), dtype=torch.bfloat16, device=DEV)
    cB = torch.zeros((B, 2, H, W, co), dtype=torch.bfloat16, device=DEV)
    ws = cuda_lib.make_workspace((B, 1, H, W), ci, co)
    outs = [cuda_lib.resblock_forward(x[:, t:t + 1].contiguous(), p, cache=(cA, cB), workspace=ws)
            for t in range(calls)]
    y = torch.cat(outs, dim=1)
    full = cuda_lib.resblock_forward(x, p)
    cuda_lib.sync_status()
    assert torch.equal(y, full)  # output must equal full-T
    pts = sample_points(T, H, W, 24, seed=2)
    ref = oracle.resblock_points(x, oracle.Params.from_dict(p), pts)
    idx = torch.tensor(pts, device=DEV)
    compare(to_f64(y[0, idx[:, 0], idx[:, 1], idx[:, 2]]), ref, what="stream 720p")


# ------------------------------------------------------------------ failure path
def test_bounded_wait_timeout_reports_and_context_survives(cuda_lib):
    """A zero wait bound makes every bounded wait of the conv give up at once:
    the kernel drains its in-flight copies, frees TMEM, returns, and the host
    reads WANVAE_ERR_TIMEOUT.  The context must stay usable."""
    B, T, H, W, ci, co = 1, 2, 16, 16, 64, 64
    x, w, b = conv_inputs(B, T, H, W, ci, co, 3, seed=70)
    xd, wd, bd = x.to(DEV), w.to(DEV), b.to(DEV)
    cuda_lib.sync_status()
    try:
        cuda_lib.set_wait_limit_ns(0)
        cuda_lib.causal_conv3d(xd, wd, bd)
        with pytest.raises(cuda_lib.WanvaeError) as ei:
            cuda_lib.sync_status()
        assert ei.value.status == cuda_lib.ERR_TIMEOUT
    finally:
        cuda_lib.set_wait_limit_ns(10 ** 9)
    y = cuda_lib.causal_conv3d(xd, wd, bd)
    cuda_lib.sync_status()
    compare(to_f64(y), oracle.causal_conv3d(x, w, b), what="after timeout")
