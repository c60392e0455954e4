"""fp64 CPU oracle of the Wan 2.2 VAE decoder ResidualBlock -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package.  The product path (the CUDA library and its
Python binding) never does, and this package imports nothing from it.

The arithmetic lives in ``wanvae_oracle.c`` (plain C, fp64, direct loops);
this module only marshals numpy float64 arrays into it.  See that file's
header for the passages of the source pages each function follows.
"""
import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


class OracleParams(ctypes.Structure):
    _fields_ = [
        ("c_in", ctypes.c_int64), ("c_out", ctypes.c_int64), ("eps", ctypes.c_double),
        ("gamma1", ctypes.c_void_p), ("gamma2", ctypes.c_void_p),
        ("wA", ctypes.c_void_p), ("bA", ctypes.c_void_p),
        ("wB", ctypes.c_void_p), ("bB", ctypes.c_void_p),
        ("wS", ctypes.c_void_p), ("bS", ctypes.c_void_p),
    ]


def lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        i64, vp, dbl, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double, ctypes.c_int
        L.oracle_rms_norm_silu.argtypes = [vp, vp, i64, i64, dbl, ci, vp]
        L.oracle_rms_norm_silu.restype = None
        L.oracle_causal_conv3d.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, ci, vp]
        L.oracle_causal_conv3d.restype = ci
        L.oracle_cache_next.argtypes = [vp, vp, i64, i64, i64, i64, i64, vp]
        L.oracle_cache_next.restype = None
        L.oracle_resblock_forward.argtypes = [vp, ctypes.POINTER(OracleParams), i64, i64, i64,
                                              i64, vp, vp, vp]
        L.oracle_resblock_forward.restype = ci
        L.oracle_resblock_points.argtypes = [vp, vp, i64, i64, ctypes.POINTER(OracleParams), vp,
                                             vp, i64, vp, vp]
        L.oracle_resblock_points.restype = ci
        L.oracle_upsample2d_conv.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp]
        L.oracle_upsample2d_conv.restype = ci
        L.oracle_time_upsample_conv.argtypes = [vp, vp, vp, i64, i64, i64, i64, i64, i64, vp]
        L.oracle_time_upsample_conv.restype = ci
        L.oracle_frame_attention.argtypes = [vp, vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, dbl,
                                             vp]
        L.oracle_frame_attention.restype = ci
        L.oracle_num_threads.argtypes = []
        L.oracle_num_threads.restype = ci
        _LIB = L
    return _LIB


def _f64(a):
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor -> exact widening to fp64
        a = a.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a):
    return None if a is None else a.ctypes.data


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def rms_norm_silu(x, gamma, eps=1e-12, silu=True):
    """RMS_norm over the last (channel) axis, then SiLU.  x: [..., C]."""
    x = _f64(x)
    g = _f64(gamma)
    C = x.shape[-1]
    out = np.empty_like(x)
    lib().oracle_rms_norm_silu(_ptr(x), _ptr(g), x.size // C, C, float(eps), int(silu), _ptr(out))
    return out


def causal_conv3d(x, w, bias, cache=None):
    """CausalConv3d over NDHWC x [B,T,H,W,Ci]; w [Co,k,k,k,Ci], k in {1,3}."""
    x, w, bias, cache = _f64(x), _f64(w), _f64(bias), _f64(cache)
    B, T, H, W, Ci = x.shape
    Co, k = w.shape[0], w.shape[1]
    out = np.empty((B, T, H, W, Co))
    rc = lib().oracle_causal_conv3d(_ptr(x), _ptr(w), _ptr(bias), _ptr(cache),
                                    B, T, H, W, Ci, Co, k, _ptr(out))
    if rc:
        raise ValueError("oracle_causal_conv3d rejected its arguments")
    return out


def upsample2d_conv(x, w, bias):
    """Nearest 2x upsampling in H and W, then a 3x3 conv (zero pad 1) with
    bias, per frame.  x [B,T,H,W,Ci], w [Co,3,3,Ci] -> [B,T,2H,2W,Co]."""
    x, w, bias = _f64(x), _f64(w), _f64(bias)
    B, T, H, W, Ci = x.shape
    Co = w.shape[0]
    out = np.empty((B, T, 2 * H, 2 * W, Co))
    rc = lib().oracle_upsample2d_conv(_ptr(x), _ptr(w), _ptr(bias), B, T, H, W, Ci, Co,
                                      _ptr(out))
    if rc:
        raise ValueError("oracle_upsample2d_conv rejected its arguments")
    return out


def time_upsample_conv(x, w, bias):
    """Temporal half of upsample3d: every frame repeated twice in T, then a
    causal 3x1x1 conv (two zero frames before the first) with bias.
    x [B,T,H,W,Ci], w [Co,3,Ci] (tap 2 = current frame) -> [B,2T,H,W,Co].

    An unconfirmed reading: the pages name the upsample3d block and 3x1x1
    conv kernels and nothing more.  A design whose 3x1x1 conv maps C to 2C
    channels and interleaves the two halves as two output frames is another
    reading the pages do not rule out; it is not what this function computes."""
    x, w, bias = _f64(x), _f64(w), _f64(bias)
    B, T, H, W, Ci = x.shape
    Co = w.shape[0]
    out = np.empty((B, 2 * T, H, W, Co))
    rc = lib().oracle_time_upsample_conv(_ptr(x), _ptr(w), _ptr(bias), B, T, H, W, Ci, Co,
                                         _ptr(out))
    if rc:
        raise ValueError("oracle_time_upsample_conv rejected its arguments")
    return out


def upsample3d(x, w_t, b_t, w_s, b_s):
    """The decoder's upsample3d as read from the pages: the temporal half
    (time_upsample_conv) and then the spatial upsampler (upsample2d_conv) on
    every frame of its output.  x [B,T,H,W,C] -> [B,2T,2H,2W,Co]."""
    return upsample2d_conv(time_upsample_conv(x, w_t, b_t), w_s, b_s)


def frame_attention(x, gamma, wqkv, bqkv, wo, bo, eps=1e-12):
    """The mid-block's spatial self-attention, per (batch, frame): RMS_norm,
    1x1 q/k/v projections, one head of softmax(q k^T / sqrt(C)) v over the
    frame's H*W positions, 1x1 output projection, plus the input.
    x [B,T,H,W,C], gamma [C], wqkv [3C,C], bqkv [3C], wo [C,C], bo [C]."""
    x, gamma, wqkv, bqkv, wo, bo = (_f64(a) for a in (x, gamma, wqkv, bqkv, wo, bo))
    B, T, H, W, C = x.shape
    out = np.empty_like(x)
    rc = lib().oracle_frame_attention(_ptr(x), _ptr(gamma), _ptr(wqkv), _ptr(bqkv), _ptr(wo),
                                      _ptr(bo), B, T, H, W, C, eps, _ptr(out))
    if rc:
        raise ValueError("oracle_frame_attention rejected its arguments")
    return out


def cache_next(cache, x):
    """Last two frames of concat(cache or zeros, x) along T."""
    x, cache = _f64(x), _f64(cache)
    B, T, H, W, C = x.shape
    out = np.empty((B, 2, H, W, C))
    lib().oracle_cache_next(_ptr(cache), _ptr(x), B, T, H, W, C, _ptr(out))
    return out


class Params:
    """ResidualBlock parameters widened to fp64 (kept alive for the C side)."""

    def __init__(self, gamma1, wA, bA, gamma2, wB, bB, wS=None, bS=None, eps=1e-12):
        self.gamma1, self.wA, self.bA = _f64(gamma1), _f64(wA), _f64(bA)
        self.gamma2, self.wB, self.bB = _f64(gamma2), _f64(wB), _f64(bB)
        self.wS, self.bS = _f64(wS), _f64(bS)
        self.c_out, self.c_in = self.wA.shape[0], self.wA.shape[-1]
        if self.wS is not None and self.bS is None:
            self.bS = np.zeros(self.c_out)
        self.eps = float(eps)

    @classmethod
    def from_dict(cls, d, eps=1e-12):
        return cls(d["gamma1"], d["wA"], d["bA"], d["gamma2"], d["wB"], d["bB"],
                   d.get("wS"), d.get("bS"), eps=eps)

    def c_struct(self):
        return OracleParams(self.c_in, self.c_out, self.eps,
                            _ptr(self.gamma1), _ptr(self.gamma2),
                            _ptr(self.wA), _ptr(self.bA), _ptr(self.wB), _ptr(self.bB),
                            _ptr(self.wS), _ptr(self.bS))


def resblock_forward(x, params: Params, cacheA=None, cacheB=None, streaming=None):
    """ResidualBlock forward.  Full-T unless streaming (default: a cache was
    given): then one streaming call whose caches [B,2,H,W,C] (None = zeros,
    i.e. before frame 0) are read, and (y, cacheA_next, cacheB_next) is
    returned."""
    x = _f64(x)
    B, T, H, W, Ci = x.shape
    y = np.empty((B, T, H, W, params.c_out))
    if streaming is None:
        streaming = cacheA is not None or cacheB is not None
    if streaming:
        cacheA = _f64(cacheA).copy() if cacheA is not None else np.zeros((B, 2, H, W, Ci))
        cacheB = (_f64(cacheB).copy() if cacheB is not None
                  else np.zeros((B, 2, H, W, params.c_out)))
    ps = params.c_struct()
    rc = lib().oracle_resblock_forward(_ptr(x), ctypes.byref(ps), B, T, H, W,
                                       _ptr(cacheA) if streaming else None,
                                       _ptr(cacheB) if streaming else None, _ptr(y))
    if rc:
        raise ValueError("oracle_resblock_forward rejected its arguments")
    return (y, cacheA, cacheB) if streaming else y


def resblock_points(x, params: Params, pts, cacheA=None, cacheB=None, b=0):
    """ResidualBlock output at sampled voxels pts [(t,y,x), ...] of batch b.

    x may be a torch tensor (CPU or CUDA, any float dtype) with the whole
    clip [B,T,H,W,Ci]; only each point's receptive field is widened to fp64.
    cacheA/cacheB: [B,2,H,W,C] caches at the start of the call, or None.
    Returns [npts, c_out] fp64.  Points run in parallel in the C oracle.
    """
    pts = np.asarray(pts, dtype=np.int64).reshape(-1, 3)
    B, T, H, W, Ci = x.shape
    out = np.empty((len(pts), params.c_out))
    ps = params.c_struct()
    cA = _f64(cacheA[b]) if cacheA is not None else None
    cB = _f64(cacheB[b]) if cacheB is not None else None
    wins, meta = [], np.empty((len(pts), 6), dtype=np.int64)
    for i, (t, yy, xx) in enumerate(pts):
        t0, y0, x0 = max(0, t - 4), max(0, yy - 2), max(0, xx - 2)
        t1, y1, x1 = t + 1, min(H, yy + 3), min(W, xx + 3)
        wins.append(_f64(x[b, t0:t1, y0:y1, x0:x1]))
        meta[i] = (t0, y0, x0, t1 - t0, y1 - y0, x1 - x0)
    ptrs = (ctypes.c_void_p * max(1, len(wins)))(*[w.ctypes.data for w in wins])
    rc = lib().oracle_resblock_points(ptrs, _ptr(meta), H, W, ctypes.byref(ps), _ptr(cA),
                                      _ptr(cB), len(pts), _ptr(pts), _ptr(out))
    if rc:
        raise ValueError("oracle_resblock_points rejected its arguments")
    return out
