"""Seeded synthetic inputs for the ResidualBlock (shared by the CUDA path's
tests/bench and by the oracle's tests).  This module draws random numbers and
nothing else: it holds none of the block's arithmetic.

Recipe (the pages name no dataset; the workloads are synthetic):
  x ~ N(0, 1); RMS_norm gammas ~ U(0.5, 1.5); conv weights ~ U(+-1/sqrt(fan_in))
  (PyTorch's default Conv3d init, fan_in = 27*C_in for the 3x3x3 convs and C_in
  for the 1x1x1 shortcut); every bias ~ U(-0.1, 0.1).  Everything is drawn in
  fp32 from one torch.Generator seeded per workload, in the fixed order
  x, gamma1, wA, bA, gamma2, wB, bB, wS, bS; x and the weights are then rounded
  to bf16 (the stored type), gammas and biases stay fp32.
"""
import math

import torch

# Workloads: (name, (B, T, H, W), c_in, c_out, streaming calls)
WORKLOADS = {
    "tiny": ((1, 3, 16, 16), 32, 32, 0),
    "latent_fullT": ((1, 21, 60, 104), 384, 384, 0),
    "stream_720p": ((1, 21, 90, 160), 384, 384, 21),
    "reduce_384_192": ((1, 41, 240, 416), 384, 192, 0),
    "fullres_96": ((1, 81, 480, 832), 96, 96, 0),
}

# The decoder's boundary convs, as single CausalConv3d calls:
# (name, (B, T, H, W), c_in, c_out, k).  conv_in lifts the 16-channel latent
# to 384 channels, post_quant_conv is the pointwise 16 -> 16 before it, and
# conv_out maps the 96-channel full-resolution features to RGB.
CONV_WORKLOADS = {
    "conv_in_latent": ((1, 21, 60, 104), 16, 384, 3),
    "post_quant_latent": ((1, 21, 60, 104), 16, 16, 1),
    "conv_out_fullres": ((1, 81, 480, 832), 96, 3, 3),
}

# The decoder's spatial upsampler (nearest 2x in H and W, then a 3x3 conv),
# as in the last upsampling up block: (name, low-res (B, T, H, W), c_in, c_out).
UPSAMPLE_WORKLOADS = {
    "upsample2d_fullres": ((1, 81, 240, 416), 192, 96),
}

# The temporal half of the decoder's upsample3d (nearest 2x in T, then a causal
# 3x1x1 conv), as in the first up block: (name, (B, T, H, W), c_in, c_out).
TIME_UPSAMPLE_WORKLOADS = {
    "time_upsample_latent": ((1, 21, 60, 104), 384, 384),
}


def _uniform(g, shape, lo, hi, device):
    return torch.rand(shape, generator=g, device=device, dtype=torch.float32) * (hi - lo) + lo


def make_params(c_in, c_out, g, device="cpu", shortcut=None):
    """Draw gamma1, wA, bA, gamma2, wB, bB (and wS, bS when c_in != c_out or
    shortcut=True) from generator g, in that order."""
    if shortcut is None:
        shortcut = c_in != c_out
    p = {}
    p["gamma1"] = _uniform(g, (c_in,), 0.5, 1.5, device)
    ba = 1.0 / math.sqrt(27 * c_in)
    p["wA"] = _uniform(g, (c_out, 3, 3, 3, c_in), -ba, ba, device).to(torch.bfloat16)
    p["bA"] = _uniform(g, (c_out,), -0.1, 0.1, device)
    p["gamma2"] = _uniform(g, (c_out,), 0.5, 1.5, device)
    bb = 1.0 / math.sqrt(27 * c_out)
    p["wB"] = _uniform(g, (c_out, 3, 3, 3, c_out), -bb, bb, device).to(torch.bfloat16)
    p["bB"] = _uniform(g, (c_out,), -0.1, 0.1, device)
    if shortcut:
        bs = 1.0 / math.sqrt(c_in)
        p["wS"] = _uniform(g, (c_out, 1, 1, 1, c_in), -bs, bs, device).to(torch.bfloat16)
        p["bS"] = _uniform(g, (c_out,), -0.1, 0.1, device)
    return p


def make_resblock_inputs(dims, c_in, c_out, seed=0, device="cpu", shortcut=None):
    """x [B,T,H,W,c_in] bf16 plus the block parameters, all from one seed."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    B, T, H, W = dims
    x = torch.randn((B, T, H, W, c_in), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    return x, make_params(c_in, c_out, g, device=device, shortcut=shortcut)


def make_conv_inputs(dims, c_in, c_out, k, seed=0, device="cpu"):
    """x [B,T,H,W,c_in] bf16 ~ N(0,1), w [c_out,k,k,k,c_in] bf16 ~ U(+-1/sqrt(fan_in)),
    bias fp32 ~ U(-0.1, 0.1), drawn in that order from one seeded generator."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    B, T, H, W = dims
    x = torch.randn((B, T, H, W, c_in), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    bound = 1.0 / math.sqrt(k * k * k * c_in)
    w = _uniform(g, (c_out, k, k, k, c_in), -bound, bound, device).to(torch.bfloat16)
    b = _uniform(g, (c_out,), -0.1, 0.1, device)
    return x, w, b


def make_time_upsample_inputs(dims, c_in, c_out, seed=0, device="cpu"):
    """x [B,T,H,W,c_in] bf16 ~ N(0,1), w [c_out,3,c_in] bf16 ~ U(+-1/sqrt(3 c_in)),
    bias fp32 ~ U(-0.1, 0.1), drawn in that order from one seeded generator."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    B, T, H, W = dims
    x = torch.randn((B, T, H, W, c_in), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    bound = 1.0 / math.sqrt(3 * c_in)
    w = _uniform(g, (c_out, 3, c_in), -bound, bound, device).to(torch.bfloat16)
    b = _uniform(g, (c_out,), -0.1, 0.1, device)
    return x, w, b
# The mid-block attention at the latent size: (name, (B, T, H, W), C).
ATTENTION_WORKLOADS = {
    "mid_attention_latent": ((1, 21, 60, 104), 384),
}


def make_attention_inputs(dims, C, seed=0, device="cpu"):
    """x [B,T,H,W,C] bf16 ~ N(0,1), gamma fp32 ~ U(0.5,1.5), wqkv [3C,C] and
    wo [C,C] bf16 ~ U(+-1/sqrt(C)), biases fp32 ~ U(-0.1,0.1), drawn in the
    order x, gamma, wqkv, bqkv, wo, bo from one seeded generator."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    B, T, H, W = dims
    x = torch.randn((B, T, H, W, C), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    gamma = _uniform(g, (C,), 0.5, 1.5, device)
    bound = 1.0 / math.sqrt(C)
    wqkv = _uniform(g, (3 * C, C), -bound, bound, device).to(torch.bfloat16)
    bqkv = _uniform(g, (3 * C,), -0.1, 0.1, device)
    wo = _uniform(g, (C, C), -bound, bound, device).to(torch.bfloat16)
    bo = _uniform(g, (C,), -0.1, 0.1, device)
    return x, gamma, wqkv, bqkv, wo, bo


def make_upsample_inputs(dims, c_in, c_out, seed=0, device="cpu"):
    """x [B,T,H,W,c_in] bf16 ~ N(0,1), w [c_out,3,3,c_in] bf16 ~ U(+-1/sqrt(9 c_in)),
    bias fp32 ~ U(-0.1, 0.1), drawn in that order from one seeded generator."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    B, T, H, W = dims
    x = torch.randn((B, T, H, W, c_in), generator=g, device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    bound = 1.0 / math.sqrt(9 * c_in)
    w = _uniform(g, (c_out, 3, 3, c_in), -bound, bound, device).to(torch.bfloat16)
    b = _uniform(g, (c_out,), -0.1, 0.1, device)
    return x, w, b


def make_tensor(shape, seed=0, device="cpu", dtype=torch.bfloat16, kind="normal", lo=-1.0, hi=1.0):
    """One seeded tensor (normal or uniform[lo,hi)), drawn in fp32, cast to dtype."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    if kind == "normal":
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    else:
        t = _uniform(g, shape, lo, hi, device)
    return t.to(dtype)
