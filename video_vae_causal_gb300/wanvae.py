"""Python binding of libwanvae.so (include/wanvae.h): argument marshalling only.

Every function here forwards to the C entry point of the same name; all the
work runs in the library's CUDA kernels.  torch is used for device memory
and streams.  There is no fallback: if the library is missing or a call
fails, an exception is raised.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwanvae.so")

(OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_MISALIGNED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT,
 ERR_UNDRAINED) = range(8)
BF16, F32 = 0, 1

# Every exported symbol of include/wanvae.h.
EXPORTS = (
    "wanvae_status_string", "wanvae_version", "wanvae_rmsnorm_silu", "wanvae_causal_conv3d",
    "wanvae_resblock_workspace_size", "wanvae_resblock_forward",
    "wanvae_resblock_forward_profiled", "wanvae_sync_status", "wanvae_set_wait_limit_ns",
    "wanvae_launch_count", "wanvae_resblock_forward_static", "wanvae_upsample2d_workspace_size",
    "wanvae_upsample2d_conv", "wanvae_set_kernel_variant", "wanvae_time_upsample_workspace_size",
    "wanvae_time_upsample_conv", "wanvae_upsample3d_workspace_size", "wanvae_upsample3d",
    "wanvae_frame_attention_workspace_size", "wanvae_frame_attention",
    "wanvae_resblock_forward_host_workspace_size", "wanvae_resblock_forward_host",
)

# Size of the library's own workspace used by resblock_forward_static.
STATIC_WORKSPACE_BYTES = 32 << 20


class WanvaeError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int64), ("T", ctypes.c_int64), ("H", ctypes.c_int64),
                ("W", ctypes.c_int64)]


class ResblockParams(ctypes.Structure):
    _fields_ = [
        ("c_in", ctypes.c_int64), ("c_out", ctypes.c_int64), ("eps", ctypes.c_float),
        ("gamma1", ctypes.c_void_p), ("gamma2", ctypes.c_void_p),
        ("wA", ctypes.c_void_p), ("bA", ctypes.c_void_p),
        ("wB", ctypes.c_void_p), ("bB", ctypes.c_void_p),
        ("wS", ctypes.c_void_p), ("bS", ctypes.c_void_p),
    ]


class ResblockCache(ctypes.Structure):
    _fields_ = [("convA_in", ctypes.c_void_p), ("convB_in", ctypes.c_void_p)]


_lib = None


def load(path=LIB_PATH):
    """Load the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with video_vae_causal_gb300.build")
    L = ctypes.CDLL(path)
    vp, i64, ci, st = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_int
    L.wanvae_status_string.argtypes = [st]
    L.wanvae_status_string.restype = ctypes.c_char_p
    L.wanvae_version.argtypes = []
    L.wanvae_version.restype = ci
    L.wanvae_rmsnorm_silu.argtypes = [vp, vp, vp, ci, i64, i64, ctypes.c_float, vp]
    L.wanvae_rmsnorm_silu.restype = st
    L.wanvae_causal_conv3d.argtypes = [vp, vp, vp, vp, Dims, i64, i64, ci, vp, vp]
    L.wanvae_causal_conv3d.restype = st
    L.wanvae_resblock_workspace_size.argtypes = [Dims, i64, i64]
    L.wanvae_resblock_workspace_size.restype = ctypes.c_size_t
    L.wanvae_resblock_forward.argtypes = [ctypes.POINTER(ResblockParams), vp, vp, Dims,
                                          ctypes.POINTER(ResblockCache), vp, ctypes.c_size_t, vp]
    L.wanvae_resblock_forward.restype = st
    L.wanvae_resblock_forward_profiled.argtypes = [
        ctypes.POINTER(ResblockParams), vp, vp, Dims, ctypes.POINTER(ResblockCache), vp,
        ctypes.c_size_t, ctypes.POINTER(vp), vp]
    L.wanvae_resblock_forward_profiled.restype = st
    L.wanvae_sync_status.argtypes = [vp]
    L.wanvae_sync_status.restype = st
    L.wanvae_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.wanvae_set_wait_limit_ns.restype = None
    L.wanvae_resblock_forward_host_workspace_size.argtypes = [Dims, i64, i64, i64]
    L.wanvae_resblock_forward_host_workspace_size.restype = ctypes.c_size_t
    L.wanvae_resblock_forward_host.argtypes = [ctypes.POINTER(ResblockParams), vp, vp, Dims, i64,
                                               vp, ctypes.c_size_t, vp, vp, vp]
    L.wanvae_resblock_forward_host.restype = st
    L.wanvae_set_kernel_variant.argtypes = [ci, ci, ci, ci, ci]
    L.wanvae_set_kernel_variant.restype = None
    L.wanvae_launch_count.argtypes = []
    L.wanvae_launch_count.restype = ctypes.c_uint64
    L.wanvae_resblock_forward_static.argtypes = [ctypes.POINTER(ResblockParams), vp, vp, Dims,
                                                 ctypes.POINTER(ResblockCache), vp]
    L.wanvae_resblock_forward_static.restype = st
    L.wanvae_upsample2d_workspace_size.argtypes = [i64, i64]
    L.wanvae_upsample2d_workspace_size.restype = ctypes.c_size_t
    L.wanvae_upsample2d_conv.argtypes = [vp, vp, vp, vp, Dims, i64, i64, vp, ctypes.c_size_t, vp]
    L.wanvae_upsample2d_conv.restype = st
    L.wanvae_time_upsample_workspace_size.argtypes = [i64, i64]
    L.wanvae_time_upsample_workspace_size.restype = ctypes.c_size_t
    L.wanvae_time_upsample_conv.argtypes = [vp, vp, vp, vp, Dims, i64, i64, vp, ctypes.c_size_t,
                                            vp]
    L.wanvae_time_upsample_conv.restype = st
    L.wanvae_upsample3d_workspace_size.argtypes = [Dims, i64, i64, i64]
    L.wanvae_upsample3d_workspace_size.restype = ctypes.c_size_t
    L.wanvae_upsample3d.argtypes = [vp, vp, vp, vp, vp, vp, Dims, i64, i64, i64, vp,
                                    ctypes.c_size_t, vp]
    L.wanvae_upsample3d.restype = st
    L.wanvae_frame_attention_workspace_size.argtypes = [Dims, i64]
    L.wanvae_frame_attention_workspace_size.restype = ctypes.c_size_t
    L.wanvae_frame_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, Dims, i64, ctypes.c_float, vp,
                                         ctypes.c_size_t, vp]
    L.wanvae_frame_attention.restype = st
    _lib = L
    return L


def status_string(status):
    return load().wanvae_status_string(int(status)).decode()


def _check(status, where):
    if status != OK:
        raise WanvaeError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dims(shape):
    B, T, H, W = shape[:4]
    return Dims(B, T, H, W)


def version():
    return int(load().wanvae_version())


def launch_count():
    return int(load().wanvae_launch_count())


def set_wait_limit_ns(ns):
    load().wanvae_set_wait_limit_ns(int(ns))


def set_kernel_variant(pair=-1, halo=-1, wide=-1, narrow=-1, fuse_norm=-1):
    """Force kernel variants for later calls (0 or 1 each; -1 = automatic)."""
    load().wanvae_set_kernel_variant(int(pair), int(halo), int(wide), int(narrow),
                                     int(fuse_norm))


def sync_status(stream=None):
    """Synchronise the stream; raise WanvaeError(ERR_TIMEOUT) if a kernel of
    the library gave up a bounded wait."""
    _check(load().wanvae_sync_status(_stream(stream)), "wanvae_sync_status")


def rmsnorm_silu(x, gamma, y=None, eps=1e-12, stream=None):
    """SiLU(RMS_norm(x)) over the last axis of x (bf16 or fp32, contiguous)."""
    dt = {torch.bfloat16: BF16, torch.float32: F32}[x.dtype]
    if y is None:
        y = torch.empty_like(x)
    C = x.shape[-1]
    st = load().wanvae_rmsnorm_silu(_ptr(x), _ptr(y), _ptr(gamma), dt, x.numel() // C, C,
                                    float(eps), _stream(stream))
    _check(st, "wanvae_rmsnorm_silu")
    return y


def causal_conv3d(x, w, bias=None, y=None, cache=None, stream=None):
    """CausalConv3d of NDHWC bf16 x [B,T,H,W,c_in] with w [c_out,k,k,k,c_in]."""
    c_out, k = w.shape[0], w.shape[1]
    if y is None:
        y = torch.empty(x.shape[:4] + (c_out,), dtype=torch.bfloat16, device=x.device)
    st = load().wanvae_causal_conv3d(_ptr(x), _ptr(w), _ptr(bias), _ptr(y), _dims(x.shape),
                                     x.shape[4], c_out, k, _ptr(cache), _stream(stream))
    _check(st, "wanvae_causal_conv3d")
    return y


def upsample2d_conv(x, w, bias=None, y=None, workspace=None, stream=None):
    """Nearest 2x upsampling in H and W, then a 3x3 conv with bias, per frame.
    x [B,T,H,W,c_in] bf16, w [c_out,3,3,c_in] bf16 -> y [B,T,2H,2W,c_out]."""
    B, T, H, W, c_in = x.shape
    c_out = w.shape[0]
    if y is None:
        y = torch.empty((B, T, 2 * H, 2 * W, c_out), dtype=torch.bfloat16, device=x.device)
    L = load()
    if workspace is None:
        n = int(L.wanvae_upsample2d_workspace_size(c_in, c_out))
        workspace = torch.empty(n, dtype=torch.uint8, device=x.device)
    st = L.wanvae_upsample2d_conv(_ptr(x), _ptr(w), _ptr(bias), _ptr(y), _dims(x.shape), c_in,
                                  c_out, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "wanvae_upsample2d_conv")
    return y


def time_upsample_conv(x, w, bias=None, y=None, workspace=None, stream=None):
    """Nearest 2x upsampling in T, then a causal 3x1x1 conv with bias (the
    temporal half of upsample3d).  x [B,T,H,W,c_in] bf16, w [c_out,3,c_in]
    bf16 -> y [B,2T,H,W,c_out]."""
    B, T, H, W, c_in = x.shape
    c_out = w.shape[0]
    if y is None:
        y = torch.empty((B, 2 * T, H, W, c_out), dtype=torch.bfloat16, device=x.device)
    L = load()
    if workspace is None:
        n = int(L.wanvae_time_upsample_workspace_size(c_in, c_out))
        workspace = torch.empty(n, dtype=torch.uint8, device=x.device)
    st = L.wanvae_time_upsample_conv(_ptr(x), _ptr(w), _ptr(bias), _ptr(y), _dims(x.shape), c_in,
                                     c_out, _ptr(workspace), workspace.numel(), _stream(stream))
    _check(st, "wanvae_time_upsample_conv")
    return y


def upsample3d(x, w_t, b_t, w_s, b_s, y=None, workspace=None, stream=None):
    """upsample3d: the temporal half (w_t [c_mid,3,c_in]) then the spatial
    upsampler (w_s [c_out,3,3,c_mid]).  x [B,T,H,W,c_in] -> [B,2T,2H,2W,c_out]."""
    B, T, H, W, c_in = x.shape
    c_mid, c_out = w_t.shape[0], w_s.shape[0]
    if y is None:
        y = torch.empty((B, 2 * T, 2 * H, 2 * W, c_out), dtype=torch.bfloat16, device=x.device)
    L = load()
    if workspace is None:
        n = int(L.wanvae_upsample3d_workspace_size(_dims(x.shape), c_in, c_mid, c_out))
        workspace = torch.empty(n, dtype=torch.uint8, device=x.device)
    st = L.wanvae_upsample3d(_ptr(x), _ptr(w_t), _ptr(b_t), _ptr(w_s), _ptr(b_s), _ptr(y),
                             _dims(x.shape), c_in, c_mid, c_out, _ptr(workspace),
                             workspace.numel(), _stream(stream))
    _check(st, "wanvae_upsample3d")
    return y


def frame_attention(x, gamma, wqkv, bqkv=None, wo=None, bo=None, y=None, workspace=None,
                    eps=1e-12, stream=None):
    """The mid-block attention: y = x + Wo softmax(q k^T / sqrt(C)) v + bo per
    frame, [q; k; v] = Wqkv RMS_norm(x) + bqkv.  x [B,T,H,W,C] bf16, gamma fp32
    [C], wqkv bf16 [3C,C], bqkv fp32 [3C], wo bf16 [C,C], bo fp32 [C]."""
    B, T, H, W, C = x.shape
    if y is None:
        y = torch.empty_like(x)
    L = load()
    if workspace is None:
        n = int(L.wanvae_frame_attention_workspace_size(_dims(x.shape), C))
        workspace = torch.empty(n, dtype=torch.uint8, device=x.device)
    st = L.wanvae_frame_attention(_ptr(x), _ptr(gamma), _ptr(wqkv), _ptr(bqkv), _ptr(wo),
                                  _ptr(bo), _ptr(y), _dims(x.shape), C, eps, _ptr(workspace),
                                  workspace.numel(), _stream(stream))
    _check(st, "wanvae_frame_attention")
    return y


def resblock_workspace_size(dims, c_in, c_out):
    return int(load().wanvae_resblock_workspace_size(_dims(dims), c_in, c_out))


def make_params(p, eps=1e-12):
    """ResblockParams from a dict of device tensors (gamma1, wA, bA, gamma2,
    wB, bB and optionally wS, bS).  Keep the dict alive while it is used."""
    c_out, c_in = p["wA"].shape[0], p["wA"].shape[-1]
    return ResblockParams(c_in, c_out, eps, p["gamma1"].data_ptr(), p["gamma2"].data_ptr(),
                          p["wA"].data_ptr(), p["bA"].data_ptr(), p["wB"].data_ptr(),
                          p["bB"].data_ptr(),
                          p["wS"].data_ptr() if p.get("wS") is not None else None,
                          p["bS"].data_ptr() if p.get("bS") is not None else None)


def make_workspace(dims, c_in, c_out, device="cuda"):
    n = resblock_workspace_size(dims, c_in, c_out)
    return torch.empty(n, dtype=torch.uint8, device=device)


def resblock_forward(x, params, y=None, cache=None, workspace=None, stream=None, events=None):
    """ResidualBlock forward of NDHWC bf16 x.

    params: a ResblockParams or a dict of device tensors.  cache: None for
    full-T, or a (convA_in, convB_in) pair of bf16 [B,2,H,W,C] tensors updated
    in place.  events: optional list of 4 torch.cuda.Event recorded around
    the kernels (see wanvae_resblock_forward_profiled)."""
    keep_alive = params  # the dict's tensors must outlive the allocations below
    if isinstance(params, dict):
        params = make_params(params)
    B, T, H, W, c_in = x.shape
    if y is None:
        y = torch.empty((B, T, H, W, params.c_out), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = make_workspace(x.shape, c_in, params.c_out, device=x.device)
    cs = None
    if cache is not None:
        cs = ctypes.byref(ResblockCache(cache[0].data_ptr(), cache[1].data_ptr()))
    L = load()
    if events is None:
        st = L.wanvae_resblock_forward(ctypes.byref(params), _ptr(x), _ptr(y), _dims(x.shape), cs,
                                       _ptr(workspace), workspace.numel(), _stream(stream))
    else:
        for e in events:
            if not e.cuda_event:  # torch creates the CUDA event lazily
                e.record()
        ev = (ctypes.c_void_p * 4)(*[e.cuda_event for e in events])
        st = L.wanvae_resblock_forward_profiled(ctypes.byref(params), _ptr(x), _ptr(y),
                                                _dims(x.shape), cs, _ptr(workspace),
                                                workspace.numel(), ev, _stream(stream))
    _check(st, "wanvae_resblock_forward")
    del keep_alive
    return y


def resblock_forward_host_workspace_size(dims, c_in, c_out, chunk_frames):
    return int(load().wanvae_resblock_forward_host_workspace_size(_dims(dims), c_in, c_out,
                                                                   chunk_frames))


def resblock_forward_host(x_host, params, y_host, chunk_frames, workspace, streams):
    """Whole-clip ResidualBlock forward of a clip in host memory (x_host, y_host:
    CPU bf16 tensors, pinned for the copies to overlap), as chunks of
    chunk_frames frames carried by the feat_cache and pipelined over
    streams = (compute, copy_in, copy_out).  Returns once enqueued; y_host is
    complete when streams[2] has drained."""
    keep_alive = params
    if isinstance(params, dict):
        params = make_params(params)
    sc, si, so = (ctypes.c_void_p(s.cuda_stream) for s in streams)
    st = load().wanvae_resblock_forward_host(ctypes.byref(params), _ptr(x_host), _ptr(y_host),
                                             _dims(x_host.shape), int(chunk_frames),
                                             _ptr(workspace), workspace.numel(), sc, si, so)
    _check(st, "wanvae_resblock_forward_host")
    del keep_alive
    return y_host


def resblock_forward_static(x, params, y, cache=None, stream=None):
    """resblock_forward with the library's own device workspace instead of a
    caller buffer, for callers that cannot allocate device memory where they
    run the block.  y must be given (nothing is allocated here either)."""
    keep_alive = params
    if isinstance(params, dict):
        params = make_params(params)
    cs = None
    if cache is not None:
        cs = ctypes.byref(ResblockCache(cache[0].data_ptr(), cache[1].data_ptr()))
    st = load().wanvae_resblock_forward_static(ctypes.byref(params), _ptr(x), _ptr(y),
                                               _dims(x.shape), cs, _stream(stream))
    _check(st, "wanvae_resblock_forward_static")
    del keep_alive
    return y
