"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test ties one part of the oracle to a library routine, a closed form, an
invariant the pages' definitions imply, or brute force, so that a dropped
term, a wrong sign or index, or a transposed operand fails at least one:

  I1  1x1x1 conv == matmul (numpy), non-square so a transposed weight fails.
  I2  delta kernels: identity, T/H/W shifts with zero borders, cache frames,
      channel permutation (pins tap order, causal pad, o/c indexing).
  I3  causality of the whole block.
  I4  full-T == frame-by-frame with feat_cache (chunks 1, 2, 5, save/resume).
  I5  whole block vs torch.nn.functional (conv3d, normalize, silu) in fp64.
  I6  norm invariants and the eps clamp in closed form.
  I7  closed form of the block at x = 0.
  +   sampled-point oracle == whole-tensor oracle, bit for bit.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from video_vae_causal_gb300 import synth


def rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def torch_resblock(x, p, eps=1e-12):
    """The block written with torch.nn.functional in fp64 (NCDHW inside)."""
    xt = torch.from_numpy(x).permute(0, 4, 1, 2, 3)

    def norm(v, g):
        g = torch.from_numpy(g).view(1, -1, 1, 1, 1)
        return F.normalize(v, p=2, dim=1, eps=eps) * math.sqrt(v.shape[1]) * g

    def conv3(v, w, b):
        v = F.pad(v, (1, 1, 1, 1, 2, 0))  # W: 1|1, H: 1|1, T: 2 leading frames
        return F.conv3d(v, torch.from_numpy(w).permute(0, 4, 1, 2, 3), torch.from_numpy(b))

    a1 = F.silu(norm(xt, p.gamma1))
    h = conv3(a1, p.wA, p.bA)
    a2 = F.silu(norm(h, p.gamma2))
    r = conv3(a2, p.wB, p.bB)
    if p.wS is None:
        s = xt
    else:
        s = F.conv3d(xt, torch.from_numpy(p.wS).permute(0, 4, 1, 2, 3), torch.from_numpy(p.bS))
    return (r + s).permute(0, 2, 3, 4, 1).numpy()


def make_params(ci, co, seed, shortcut=None):
    g = torch.Generator().manual_seed(seed)
    return oracle.Params.from_dict(synth.make_params(ci, co, g, shortcut=shortcut))


# ---------------------------------------------------------------- I1
def test_I1_pointwise_conv_is_matmul():
    x = rand((2, 3, 4, 5, 6), 1)
    w = rand((5, 1, 1, 1, 6), 2)
    b = rand((5,), 3)
    got = oracle.causal_conv3d(x, w, b)
    ref = x.reshape(-1, 6) @ w.reshape(5, 6).T + b
    np.testing.assert_allclose(got.reshape(-1, 5), ref, rtol=1e-13, atol=1e-13)


# ---------------------------------------------------------------- I2
def delta_w(C, kt, kh, kw, perm=None):
    w = np.zeros((C, 3, 3, 3, C))
    for o in range(C):
        w[o, kt, kh, kw, o if perm is None else perm[o]] = 1.0
    return w


def test_I2_delta_identity_exact():
    a = rand((1, 4, 5, 6, 3), 4)
    got = oracle.causal_conv3d(a, delta_w(3, 2, 1, 1), np.zeros(3))
    assert np.array_equal(got, a)


@pytest.mark.parametrize("kt", [0, 1])
def test_I2_delta_time_shift_causal(kt):
    a = rand((2, 5, 3, 4, 2), 5)
    got = oracle.causal_conv3d(a, delta_w(2, kt, 1, 1), np.zeros(2))
    shift = 2 - kt
    assert np.array_equal(got[:, shift:], a[:, :5 - shift])
    assert np.all(got[:, :shift] == 0)


@pytest.mark.parametrize("kh,kw", [(0, 1), (2, 1), (1, 0), (1, 2), (0, 0), (2, 2)])
def test_I2_delta_spatial_shift_zero_border(kh, kw):
    a = rand((1, 2, 5, 6, 2), 6)
    got = oracle.causal_conv3d(a, delta_w(2, 2, kh, kw), np.zeros(2))
    dy, dx = kh - 1, kw - 1
    ref = np.zeros_like(a)
    H, W = 5, 6
    for y in range(H):
        for x in range(W):
            if 0 <= y + dy < H and 0 <= x + dx < W:
                ref[:, :, y, x] = a[:, :, y + dy, x + dx]
    assert np.array_equal(got, ref)


def test_I2_delta_reads_cache_frames():
    a = rand((1, 3, 2, 3, 2), 7)
    cache = rand((1, 2, 2, 3, 2), 8)
    got = oracle.causal_conv3d(a, delta_w(2, 0, 1, 1), np.zeros(2), cache=cache)
    assert np.array_equal(got[:, 0], cache[:, 0])
    assert np.array_equal(got[:, 1], cache[:, 1])
    assert np.array_equal(got[:, 2], a[:, 0])


def test_I2_channel_permutation_pins_o_c_order():
    perm = [2, 0, 3, 1]
    a = rand((1, 2, 3, 3, 4), 9)
    got = oracle.causal_conv3d(a, delta_w(4, 2, 1, 1, perm), np.zeros(4))
    assert np.array_equal(got, a[..., perm])


# ---------------------------------------------------------------- I3
@pytest.mark.parametrize("ci,co", [(8, 8), (8, 16)])
def test_I3_block_is_causal(ci, co):
    p = make_params(ci, co, 10)
    x = rand((1, 6, 4, 5, ci), 11)
    y = oracle.resblock_forward(x, p)
    for t in range(5):
        x2 = x.copy()
        x2[:, t + 1:] += rand(x2[:, t + 1:].shape, 12 + t)
        y2 = oracle.resblock_forward(x2, p)
        assert np.array_equal(y2[:, :t + 1], y[:, :t + 1])
        assert not np.array_equal(y2[:, t + 1:], y[:, t + 1:])


# ---------------------------------------------------------------- I4
@pytest.mark.parametrize("chunks", [[1] * 7, [2, 2, 2, 1], [5, 2], [3, 1, 3]])
@pytest.mark.parametrize("ci,co", [(8, 8), (16, 8)])
def test_I4_fullT_equals_streaming(chunks, ci, co):
    p = make_params(ci, co, 20)
    x = rand((2, 7, 4, 5, ci), 21)
    full = oracle.resblock_forward(x, p)
    cA = cB = None
    outs, t0 = [], 0
    for n in chunks:
        y, cA, cB = oracle.resblock_forward(x[:, t0:t0 + n], p, cA, cB, streaming=True)
        outs.append(y)
        t0 += n
    assert np.array_equal(np.concatenate(outs, axis=1), full)


def test_I4_save_and_resume_cache():
    p = make_params(8, 8, 22)
    x = rand((1, 6, 3, 4, 8), 23)
    cA = cB = None
    ys = []
    for t in range(3):
        y, cA, cB = oracle.resblock_forward(x[:, t:t + 1], p, cA, cB, streaming=True)
        ys.append(y)
    saved = (cA.copy(), cB.copy())
    # an interruption: unrelated work through a fresh cache, then resume
    oracle.resblock_forward(rand((1, 2, 3, 4, 8), 24), p, None, np.zeros((1, 2, 3, 4, 8)))
    cA, cB = saved
    for t in range(3, 6):
        y, cA, cB = oracle.resblock_forward(x[:, t:t + 1], p, cA, cB, streaming=True)
        ys.append(y)
    assert np.array_equal(np.concatenate(ys, axis=1), oracle.resblock_forward(x, p))


def test_I4_cache_next_definition():
    c = rand((1, 2, 2, 2, 3), 25)
    x1 = rand((1, 1, 2, 2, 3), 26)
    n1 = oracle.cache_next(c, x1)
    assert np.array_equal(n1[:, 0], c[:, 1]) and np.array_equal(n1[:, 1], x1[:, 0])
    x3 = rand((1, 3, 2, 2, 3), 27)
    assert np.array_equal(oracle.cache_next(c, x3), x3[:, 1:])
    assert np.array_equal(oracle.cache_next(None, x1)[:, 0], np.zeros((1, 2, 2, 3)))


# ---------------------------------------------------------------- I5
@pytest.mark.parametrize("B,T,H,W,ci,co", [
    (1, 3, 4, 5, 4, 4), (2, 4, 3, 6, 8, 8), (1, 2, 5, 3, 8, 4), (2, 3, 4, 4, 4, 8),
    (1, 1, 1, 1, 8, 8), (1, 4, 6, 2, 2, 6),
])
def test_I5_block_matches_torch_functional(B, T, H, W, ci, co):
    p = make_params(ci, co, 30 + ci + co)
    x = rand((B, T, H, W, ci), 31)
    np.testing.assert_allclose(oracle.resblock_forward(x, p), torch_resblock(x, p),
                               rtol=1e-11, atol=1e-11)


def test_I5_conv_with_shortcut_param_but_equal_channels():
    # a 1x1x1 shortcut conv is also legal when c_in == c_out
    p = make_params(8, 8, 33, shortcut=True)
    x = rand((1, 3, 4, 4, 8), 34)
    np.testing.assert_allclose(oracle.resblock_forward(x, p), torch_resblock(x, p),
                               rtol=1e-11, atol=1e-11)


def test_I5_brute_force_tiny_workload():
    """The 'tiny' workload ([1,3,16,16,32], seed 0) end to end, every element."""
    dims, ci, co, _ = synth.WORKLOADS["tiny"]
    x, pd = synth.make_resblock_inputs(dims, ci, co, seed=0)
    p = oracle.Params.from_dict(pd)
    xd = x.double().numpy()
    np.testing.assert_allclose(oracle.resblock_forward(xd, p), torch_resblock(xd, p),
                               rtol=1e-11, atol=1e-11)


def test_I5_conv3_matches_torch():
    x = rand((2, 4, 5, 3, 6), 35)
    w = rand((7, 3, 3, 3, 6), 36)
    b = rand((7,), 37)
    ref = F.conv3d(F.pad(torch.from_numpy(x).permute(0, 4, 1, 2, 3), (1, 1, 1, 1, 2, 0)),
                   torch.from_numpy(w).permute(0, 4, 1, 2, 3), torch.from_numpy(b))
    np.testing.assert_allclose(oracle.causal_conv3d(x, w, b),
                               ref.permute(0, 2, 3, 4, 1).numpy(), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- I6
def test_I6_norm_invariants():
    C = 12
    x = rand((50, C), 40)
    g = np.random.default_rng(41).uniform(0.5, 1.5, C)
    n = oracle.rms_norm_silu(x, g, silu=False)
    np.testing.assert_allclose(np.sum((n / (math.sqrt(C) * g)) ** 2, axis=1), 1.0, rtol=1e-13)
    np.testing.assert_allclose(oracle.rms_norm_silu(3.7 * x, g, silu=False), n, rtol=1e-13)
    assert np.array_equal(oracle.rms_norm_silu(np.zeros((2, C)), g), np.zeros((2, C)))


def test_I6_norm_closed_form_and_eps_clamp():
    # x = (3, 4): |x| = 5, sqrt(D) = sqrt(2)
    g = np.array([1.0, 2.0])
    z = np.array([3 / 5 * math.sqrt(2) * 1.0, 4 / 5 * math.sqrt(2) * 2.0])
    np.testing.assert_allclose(oracle.rms_norm_silu(np.array([[3.0, 4.0]]), g, silu=False)[0],
                               z, rtol=1e-15)
    np.testing.assert_allclose(oracle.rms_norm_silu(np.array([[3.0, 4.0]]), g)[0],
                               z / (1 + np.exp(-z)), rtol=1e-15)
    # below eps the clamp divides by eps itself: 1e-13 * 2 / 1e-12 = 0.2
    tiny = np.full((1, 4), 1e-13)
    np.testing.assert_allclose(oracle.rms_norm_silu(tiny, np.ones(4), eps=1e-12, silu=False),
                               np.full((1, 4), 0.2), rtol=1e-12)


def test_I6_silu_sign_and_limits():
    v = np.array([[-30.0, 0.0, 30.0]])
    s = oracle.rms_norm_silu(v, np.ones(3), silu=True)
    zn = oracle.rms_norm_silu(v, np.ones(3), silu=False)
    assert s[0, 0] < 0 and abs(s[0, 0]) < 0.3 and s[0, 1] == 0
    np.testing.assert_allclose(s[0, 2], zn[0, 2] / (1 + math.exp(-zn[0, 2])), rtol=1e-15)


# ---------------------------------------------------------------- I7
@pytest.mark.parametrize("ci,co", [(6, 6), (6, 4)])
def test_I7_closed_form_at_zero_input(ci, co):
    p = make_params(ci, co, 50)
    B, T, H, W = 1, 4, 4, 5
    x = np.zeros((B, T, H, W, ci))
    y = oracle.resblock_forward(x, p)
    # a1 = 0, so h = bA at every voxel and a2 = silu(norm(bA)) is one vector
    nb = np.linalg.norm(p.bA)
    z = p.bA / nb * math.sqrt(co) * p.gamma2
    a2 = z / (1 + np.exp(-z))
    ref = np.zeros((B, T, H, W, co))
    for t in range(T):
        for yy in range(H):
            for xx in range(W):
                acc = p.bB.copy()
                for kt in range(3):
                    for kh in range(3):
                        for kw in range(3):
                            if t + kt - 2 >= 0 and 0 <= yy + kh - 1 < H and 0 <= xx + kw - 1 < W:
                                acc += p.wB[:, kt, kh, kw, :] @ a2
                ref[0, t, yy, xx] = acc + (0.0 if p.wS is None else p.bS)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- points
@pytest.mark.parametrize("ci,co", [(8, 8), (8, 4)])
def test_points_equal_full_forward_bitwise(ci, co):
    p = make_params(ci, co, 60)
    x = rand((2, 6, 5, 7, ci), 61)
    y = oracle.resblock_forward(x, p)
    rng = np.random.default_rng(62)
    for b in range(2):
        pts = [(t, yy, xx) for t in (0, 1, 5) for yy in (0, 2, 4) for xx in (0, 6)]
        pts += [tuple(rng.integers([0, 0, 0], [6, 5, 7])) for _ in range(6)]
        got = oracle.resblock_points(torch.from_numpy(x), p, pts, b=b)
        ref = np.stack([y[b, t, yy, xx] for t, yy, xx in pts])
        assert np.array_equal(got, ref)


def test_points_with_cache_equal_streaming_call():
    p = make_params(8, 8, 63)
    x = rand((1, 5, 4, 4, 8), 64)
    _, cA, cB = oracle.resblock_forward(x[:, :3], p, streaming=True)
    y, _, _ = oracle.resblock_forward(x[:, 3:], p, cA, cB)
    pts = [(t, yy, xx) for t in (0, 1) for yy in (0, 3) for xx in (0, 1, 3)]
    got = oracle.resblock_points(torch.from_numpy(x[:, 3:].copy()), p, pts, cA, cB)
    assert np.array_equal(got, np.stack([y[0, t, yy, xx] for t, yy, xx in pts]))


def test_bf16_widening_is_exact():
    t = synth.make_tensor((64,), seed=3)
    v = t.float().numpy().astype(np.float64)
    assert np.array_equal(oracle._f64(t), v)


# ---------------------------------------------------------------- upsample2d
# The decoder's spatial upsampler (nearest 2x in H and W, then a 3x3 conv with
# zero pad 1 and a bias) -- pinned against a library routine, a delta kernel
# and brute force on an explicitly upsampled array.
def test_U1_upsample2d_matches_torch_functional():
    x = rand((2, 3, 4, 5, 6), 90)
    w = rand((7, 3, 3, 6), 91)
    b = rand((7,), 92)
    y = oracle.upsample2d_conv(x, w, b)
    B, T, H, W, C = x.shape
    xt = torch.from_numpy(x).reshape(B * T, H, W, C).permute(0, 3, 1, 2)
    up = F.interpolate(xt, scale_factor=2, mode="nearest")
    ref = F.conv2d(up, torch.from_numpy(w).permute(0, 3, 1, 2), torch.from_numpy(b), padding=1)
    ref = ref.permute(0, 2, 3, 1).reshape(B, T, 2 * H, 2 * W, 7).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_U2_upsample2d_delta_is_nearest_upsampling():
    x = rand((1, 2, 3, 4, 5), 93)
    w = np.zeros((5, 3, 3, 5))
    w[:, 1, 1, :] = np.eye(5)
    y = oracle.upsample2d_conv(x, w, np.zeros(5))
    assert np.array_equal(y, x.repeat(2, axis=2).repeat(2, axis=3))


@pytest.mark.parametrize("kh,kw", [(0, 0), (2, 1), (1, 2)])
def test_U2_upsample2d_delta_shift_zero_border(kh, kw):
    x = rand((1, 1, 3, 3, 2), 94)
    w = np.zeros((2, 3, 3, 2))
    w[:, kh, kw, :] = np.eye(2)
    y = oracle.upsample2d_conv(x, w, np.zeros(2))
    up = x.repeat(2, axis=2).repeat(2, axis=3)
    ref = np.zeros_like(up)
    for Y in range(6):
        for X in range(6):
            yy, xx = Y + kh - 1, X + kw - 1
            if 0 <= yy < 6 and 0 <= xx < 6:
                ref[:, :, Y, X] = up[:, :, yy, xx]
    assert np.array_equal(y, ref)


def test_U3_upsample2d_brute_force_tiny():
    x = rand((1, 1, 2, 3, 2), 95)
    w = rand((3, 3, 3, 2), 96)
    b = rand((3,), 97)
    y = oracle.upsample2d_conv(x, w, b)
    up = np.zeros((4, 6, 2))
    for i in range(4):
        for j in range(6):
            up[i, j] = x[0, 0, i // 2, j // 2]
    for Y in range(4):
        for X in range(6):
            for o in range(3):
                acc = b[o]
                for kh in range(3):
                    for kw in range(3):
                        if 0 <= Y + kh - 1 < 4 and 0 <= X + kw - 1 < 6:
                            acc += float(np.dot(w[o, kh, kw], up[Y + kh - 1, X + kw - 1]))
                assert abs(y[0, 0, Y, X, o] - acc) < 1e-12


def test_U4_upsample2d_is_four_subpixel_2x2_convs():
    """The identity the GPU path computes by: output pixel (2i+a, 2j+b) reads the
    upsampled row 2i+a+kh-1, i.e. low-res row floor((a+kh-1)/2) + i, which is
    i+a-1 or i+a; so each phase (a, b) is a 2x2 conv of the low-res x at offsets
    (a+e-1, b+f-1), e, f in {0, 1}, whose taps sum the 3x3 taps landing there.
    Exact in fp64 up to summation order (the oracle itself is the definition)."""
    x = rand((2, 2, 5, 6, 4), 98)
    w = rand((3, 3, 3, 4), 99)
    b = rand((3,), 100)
    ref = oracle.upsample2d_conv(x, w, b)
    B, T, H, W, C = x.shape
    xp = np.zeros((B, T, H + 2, W + 2, C))
    xp[:, :, 1:-1, 1:-1] = x  # low-res zero pad 1
    y = np.zeros((B, T, 2 * H, 2 * W, 3))
    for a in range(2):
        for bb in range(2):
            w2 = np.zeros((3, 2, 2, C))
            for kh in range(3):
                for kw in range(3):
                    e = (a + kh - 1) // 2 - (a - 1)   # low-res row offset relative to a-1
                    f = (bb + kw - 1) // 2 - (bb - 1)
                    w2[:, e, f] += w[:, kh, kw]
            # every 3x3 tap lands on exactly one 2x2 tap of every phase
            np.testing.assert_allclose(w2.sum(axis=(1, 2)), w.sum(axis=(1, 2)), rtol=0, atol=1e-14)
            for e in range(2):
                for f in range(2):
                    # padded index of low-res row i + a + e - 1 is i + a + e
                    win = xp[:, :, a + e:a + e + H, bb + f:bb + f + W]
                    y[:, :, a::2, bb::2] += np.einsum("btijc,oc->btijo", win, w2[:, e, f])
            y[:, :, a::2, bb::2] += b
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------ upsample3d, temporal half
# Nearest 2x in T, then a causal 3x1x1 conv with bias -- pinned against a
# library routine, delta kernels, causality and brute force.
def _torch_time_upsample(x, w, b):
    xt = torch.from_numpy(x).permute(0, 4, 1, 2, 3)              # N C T H W
    up = xt.repeat_interleave(2, dim=2)
    up = F.pad(up, (0, 0, 0, 0, 2, 0))                            # two zero frames first
    wt = torch.from_numpy(w).permute(0, 2, 1)[..., None, None]    # Co Ci 3 1 1
    return F.conv3d(up, wt, torch.from_numpy(b)).permute(0, 2, 3, 4, 1).numpy()


def test_T1_time_upsample_matches_torch_functional():
    x = rand((2, 3, 2, 3, 5), 110)
    w = rand((4, 3, 5), 111)
    b = rand((4,), 112)
    y = oracle.time_upsample_conv(x, w, b)
    assert y.shape == (2, 6, 2, 3, 4)
    np.testing.assert_allclose(y, _torch_time_upsample(x, w, b), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("kt", [0, 1, 2])
def test_T2_time_upsample_delta_taps(kt):
    x = rand((1, 3, 2, 2, 3), 113)
    w = np.zeros((3, 3, 3))
    w[:, kt, :] = np.eye(3)
    y = oracle.time_upsample_conv(x, w, np.zeros(3))
    up = x.repeat(2, axis=1)          # frame s of the upsampled sequence is x[s // 2]
    shift = 2 - kt                    # tap kt reads upsampled frame s - shift
    ref = np.zeros_like(up)
    ref[:, shift:] = up[:, :up.shape[1] - shift]
    assert np.array_equal(y, ref)


def test_T3_time_upsample_is_causal():
    x = rand((1, 4, 2, 2, 3), 114)
    w = rand((2, 3, 3), 115)
    b = rand((2,), 116)
    y0 = oracle.time_upsample_conv(x, w, b)
    for t in range(4):
        x1 = x.copy()
        x1[:, t] += 1.0
        y1 = oracle.time_upsample_conv(x1, w, b)
        assert np.array_equal(y1[:, :2 * t], y0[:, :2 * t])       # nothing before 2t moves
        assert not np.array_equal(y1[:, 2 * t], y0[:, 2 * t])


def test_T4_time_upsample_brute_force_tiny():
    x = rand((1, 2, 1, 2, 2), 117)
    w = rand((2, 3, 2), 118)
    b = rand((2,), 119)
    y = oracle.time_upsample_conv(x, w, b)
    for s in range(4):
        for p in range(2):
            for o in range(2):
                acc = b[o]
                for kt in range(3):
                    u = s + kt - 2
                    if u >= 0:
                        acc += float(np.dot(w[o, kt], x[0, u // 2, 0, p]))
                assert abs(y[0, s, 0, p, o] - acc) < 1e-12


def test_T5_upsample3d_is_time_then_space():
    x = rand((1, 2, 2, 3, 4), 120)
    w_t, b_t = rand((4, 3, 4), 121), rand((4,), 122)
    w_s, b_s = rand((3, 3, 3, 4), 123), rand((3,), 124)
    y = oracle.upsample3d(x, w_t, b_t, w_s, b_s)
    assert y.shape == (1, 4, 4, 6, 3)
    mid = _torch_time_upsample(x, w_t, b_t)                     # [1, 4, 2, 3, 4]
    B, T2, H, W, C = mid.shape
    mt = torch.from_numpy(mid).reshape(B * T2, H, W, C).permute(0, 3, 1, 2)
    up = F.interpolate(mt, scale_factor=2, mode="nearest")
    ref = F.conv2d(up, torch.from_numpy(w_s).permute(0, 3, 1, 2), torch.from_numpy(b_s),
                   padding=1)
    ref = ref.permute(0, 2, 3, 1).reshape(B, T2, 2 * H, 2 * W, 3).numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_T6_time_upsample_is_two_frame_phases():
    """The identity the GPU path computes by: upsampled frame 2t+a+kt-2 is
    input frame t-1+((a+kt)//2) (or a causal zero), so output frame 2t+a is a
    2-tap conv of frames t-1 and t whose taps sum the 3 taps landing there."""
    x = rand((2, 3, 2, 3, 4), 125)
    w = rand((3, 3, 4), 126)
    b = rand((3,), 127)
    ref = oracle.time_upsample_conv(x, w, b)
    B, T, H, W, C = x.shape
    xp = np.concatenate([np.zeros((B, 1, H, W, C)), x], axis=1)   # frame -1 = zeros
    y = np.zeros((B, 2 * T, H, W, 3))
    for a in range(2):
        w2 = np.zeros((3, 2, C))
        for kt in range(3):
            w2[:, (a + kt) // 2] += w[:, kt]
        for e in range(2):
            # padded index of input frame t - 1 + e is t + e
            y[:, a::2] += np.einsum("bthwc,oc->bthwo", xp[:, e:e + T], w2[:, e])
        y[:, a::2] += b
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------- mid-block attention
# One head of softmax(q k^T / sqrt(C)) v over each frame's H*W positions,
# between an RMS_norm and a 1x1 output projection, plus the input.
def _attn_params(C, seed):
    g = rand((C,), seed) * 0.5 + 1.0
    return (g, rand((3 * C, C), seed + 1) / np.sqrt(C), rand((3 * C,), seed + 2) * 0.1,
            rand((C, C), seed + 3) / np.sqrt(C), rand((C,), seed + 4) * 0.1)


def _torch_attention(x, g, wqkv, bqkv, wo, bo, eps=1e-12):
    B, T, H, W, C = x.shape
    xt = torch.from_numpy(x).reshape(B * T, H * W, C)
    n = F.normalize(xt, dim=-1, eps=eps) * np.sqrt(C) * torch.from_numpy(g)
    qkv = n @ torch.from_numpy(wqkv).T + torch.from_numpy(bqkv)
    q, k, v = qkv[..., :C], qkv[..., C:2 * C], qkv[..., 2 * C:]
    o = F.scaled_dot_product_attention(q, k, v)            # scale 1 / sqrt(C)
    y = xt + o @ torch.from_numpy(wo).T + torch.from_numpy(bo)
    return y.reshape(B, T, H, W, C).numpy()


def test_A1_attention_matches_torch_sdpa():
    x = rand((2, 2, 3, 4, 8), 130)
    p = _attn_params(8, 131)
    np.testing.assert_allclose(oracle.frame_attention(x, *p), _torch_attention(x, *p),
                               rtol=1e-11, atol=1e-11)


def test_A2_attention_uniform_when_q_k_vanish():
    """Zero q and k weights and biases: every score is 0, attention is the mean
    of v over the frame, so out = x + bo + Wo mean_j(v_j)."""
    x = rand((1, 2, 2, 3, 6), 132)
    g, wqkv, bqkv, wo, bo = _attn_params(6, 133)
    wqkv[:12] = 0.0
    bqkv[:12] = 0.0
    y = oracle.frame_attention(x, g, wqkv, bqkv, wo, bo)
    C = 6
    for t in range(2):
        xf = x[0, t].reshape(-1, C)
        nrm = xf / np.maximum(np.linalg.norm(xf, axis=1, keepdims=True), 1e-12) * np.sqrt(C) * g
        v = nrm @ wqkv[12:].T + bqkv[12:]
        ref = xf + bo + wo @ v.mean(axis=0)
        np.testing.assert_allclose(y[0, t].reshape(-1, C), ref, rtol=1e-12, atol=1e-12)


def test_A3_attention_is_permutation_equivariant():
    x = rand((1, 1, 3, 5, 4), 134)
    p = _attn_params(4, 135)
    perm = np.random.default_rng(7).permutation(15)
    xp = x.reshape(1, 1, 15, 4)[:, :, perm].reshape(1, 1, 3, 5, 4)
    y = oracle.frame_attention(x, *p).reshape(1, 1, 15, 4)
    yp = oracle.frame_attention(xp, *p).reshape(1, 1, 15, 4)
    np.testing.assert_allclose(yp, y[:, :, perm], rtol=1e-12, atol=1e-12)


def test_A4_attention_single_position_is_v():
    """One position per frame: its only key gets weight 1, so out = x + bo + Wo v."""
    x = rand((1, 3, 1, 1, 5), 136)
    g, wqkv, bqkv, wo, bo = _attn_params(5, 137)
    y = oracle.frame_attention(x, g, wqkv, bqkv, wo, bo)
    for t in range(3):
        xv = x[0, t, 0, 0]
        nrm = xv / max(np.linalg.norm(xv), 1e-12) * np.sqrt(5) * g
        v = wqkv[10:] @ nrm + bqkv[10:]
        np.testing.assert_allclose(y[0, t, 0, 0], xv + bo + wo @ v, rtol=1e-12, atol=1e-12)


def test_A5_attention_frames_are_independent():
    x = rand((2, 3, 2, 2, 4), 138)
    p = _attn_params(4, 139)
    y0 = oracle.frame_attention(x, *p)
    x1 = x.copy()
    x1[1, 2] += 1.0
    y1 = oracle.frame_attention(x1, *p)
    changed = np.abs(y1 - y0).reshape(2, 3, -1).max(axis=2) > 0
    assert changed[1, 2] and changed.sum() == 1
