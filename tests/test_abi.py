"""The C ABI library without a GPU: it loads, exports every symbol that
include/wanvae.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from video_vae_causal_gb300 import build as libbuild
from video_vae_causal_gb300 import wanvae

HEADER = os.path.join(ROOT, "include", "wanvae.h")


@pytest.fixture(scope="module")
def lib():
    libbuild.build()
    return wanvae.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wanvae_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_what_binding_lists():
    assert declared_functions() == sorted(wanvae.EXPORTS)


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(wanvae.LIB_PATH)
    for name in declared_functions():
        assert hasattr(raw, name), name


def test_only_c_abi_is_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", wanvae.LIB_PATH], capture_output=True,
                         text=True).stdout
    funcs = [l.split()[-1] for l in out.splitlines() if " T " in l]
    assert funcs and all(f.startswith("wanvae_") for f in funcs), funcs


def test_status_strings_and_version(lib):
    for s in range(8):
        assert wanvae.status_string(s)
    assert "context" in wanvae.status_string(wanvae.ERR_UNDRAINED)
    assert wanvae.status_string(99) == "unknown status"
    assert wanvae.version() == 101


def test_workspace_size(lib):
    n = wanvae.resblock_workspace_size((1, 21, 60, 104), 384, 384)
    M = 21 * 60 * 104
    assert n == 2 * ((M * 384 * 2 + 255) // 256 * 256)
    assert wanvae.resblock_workspace_size((1, 0, 4, 4), 32, 32) == 0
    assert wanvae.resblock_workspace_size((1, 2, 4, 4), 0, 32) == 0


def _dims(B, T, H, W):
    return wanvae.Dims(B, T, H, W)


A = 0x10000  # a 16-byte aligned fake device address (never dereferenced)


def test_norm_argument_errors(lib):
    L = lib
    f = L.wanvae_rmsnorm_silu
    assert f(None, A, A, 0, 10, 32, 1e-12, None) == wanvae.ERR_INVALID_ARG
    assert f(A, 0x90000, A, 0, 10, 24, 1e-12, None) == wanvae.ERR_INVALID_ARG  # C % 16
    assert f(A, 0x90000, A, 0, 0, 32, 1e-12, None) == wanvae.ERR_INVALID_ARG   # no voxels
    assert f(A, 0x90000, A, 7, 10, 32, 1e-12, None) == wanvae.ERR_INVALID_ARG  # bad dtype
    assert f(A, 0x90000, A, 0, 10, 32, -1.0, None) == wanvae.ERR_INVALID_ARG  # eps < 0
    assert f(A + 8, 0x90000, A, 0, 10, 32, 1e-12, None) == wanvae.ERR_MISALIGNED
    assert f(A, A + 64, A, 0, 10, 32, 1e-12, None) == wanvae.ERR_INVALID_ARG  # y aliases x


def test_conv_argument_errors(lib):
    f = lib.wanvae_causal_conv3d
    d = _dims(1, 2, 4, 4)
    Y = 0x900000
    assert f(A, A, None, Y, d, 32, 32, 2, None, None) == wanvae.ERR_INVALID_ARG  # k
    assert f(A, A, None, Y, d, 32, 32, 1, 0x200000, None) == wanvae.ERR_INVALID_ARG  # k=1 cache
    assert f(A, A, None, Y, _dims(1, 0, 4, 4), 32, 32, 3, None, None) == wanvae.ERR_INVALID_ARG
    assert f(A, A, None, Y, d, 40, 32, 3, None, None) == wanvae.ERR_UNSUPPORTED
    assert f(A, A, None, Y, d, 32, 1024, 3, None, None) == wanvae.ERR_UNSUPPORTED
    assert f(A, A, None, Y, d, 32, 17, 3, None, None) == wanvae.ERR_UNSUPPORTED  # 16 < c_out, % 16
    assert f(A, A, None, Y, d, 32, 0, 3, None, None) == wanvae.ERR_INVALID_ARG
    assert f(A, A + 4, None, Y, d, 32, 32, 3, None, None) == wanvae.ERR_MISALIGNED
    assert f(A, A, None, A + 16, d, 32, 32, 3, None, None) == wanvae.ERR_INVALID_ARG  # alias


def test_upsample_argument_errors(lib):
    f = lib.wanvae_upsample2d_conv
    d = _dims(1, 2, 4, 4)
    Y, WS = 0x900000, 0x2000000
    n = lib.wanvae_upsample2d_workspace_size(32, 16)
    assert n == 4 * 4 * 32 * 16 * 2  # 4 phases x 2 x 2 taps
    assert f(None, A, None, Y, d, 32, 16, WS, n, None) == wanvae.ERR_INVALID_ARG
    assert f(A, A, None, Y, d, 32, 16, None, n, None) == wanvae.ERR_INVALID_ARG
    assert f(A, A, None, Y, d, 32, 272, WS, 1 << 30, None) == wanvae.ERR_UNSUPPORTED
    assert f(A, A, None, Y, d, 40, 16, WS, n, None) == wanvae.ERR_UNSUPPORTED
    assert f(A, A, None, Y, d, 32, 16, WS, n - 2, None) == wanvae.ERR_WORKSPACE
    assert f(A, A + 4, None, Y, d, 32, 16, WS, n, None) == wanvae.ERR_MISALIGNED


def test_time_upsample_argument_errors(lib):
    f = lib.wanvae_time_upsample_conv
    d = _dims(1, 2, 4, 4)
    Y, WS = 0x900000, 0x2000000
    n = lib.wanvae_time_upsample_workspace_size(32, 16)
    assert n == 2 * 2 * 32 * 16 * 2  # 2 phases x 2 taps
    assert f(None, A, None, Y, d, 32, 16, WS, n, None) == wanvae.ERR_INVALID_ARG
    assert f(A, A, None, Y, d, 32, 16, None, n, None) == wanvae.ERR_INVALID_ARG
    assert f(A, A, None, Y, d, 32, 528, WS, 1 << 30, None) == wanvae.ERR_UNSUPPORTED
    assert f(A, A, None, Y, d, 40, 16, WS, n, None) == wanvae.ERR_UNSUPPORTED
    assert f(A, A, None, Y, d, 32, 16, WS, n - 2, None) == wanvae.ERR_WORKSPACE
    assert f(A, A + 4, None, Y, d, 32, 16, WS, n, None) == wanvae.ERR_MISALIGNED
def test_frame_attention_argument_errors(lib):
    f = lib.wanvae_frame_attention
    d = _dims(1, 2, 4, 4)
    Y, WS = 0x900000, 0x2000000
    n = lib.wanvae_frame_attention_workspace_size(d, 128)
    assert n > 0
    assert f(None, A, A, None, A, None, Y, d, 128, 1e-12, WS, n, None) == wanvae.ERR_INVALID_ARG
    assert f(A, A, A, None, A, None, Y, d, 128, 0.0, WS, n, None) == wanvae.ERR_INVALID_ARG
    assert f(A, A, A, None, A, None, Y, d, 192, 1e-12, WS, 1 << 30, None) == wanvae.ERR_UNSUPPORTED
    assert f(A, A, A, None, A, None, Y, d, 128, 1e-12, WS, n - 2, None) == wanvae.ERR_WORKSPACE
    assert f(A, A + 4, A, None, A, None, Y, d, 128, 1e-12, WS, n, None) == wanvae.ERR_MISALIGNED


def test_resblock_argument_errors(lib):
    f = lib.wanvae_resblock_forward
    d = _dims(1, 2, 4, 4)
    P = wanvae.ResblockParams(32, 32, 1e-12, A, A, A, A, A, A, None, None)
    X, Y, WS = 0x100000, 0x200000, 0x300000
    need = wanvae.resblock_workspace_size((1, 2, 4, 4), 32, 32)
    assert f(None, X, Y, d, None, WS, need, None) == wanvae.ERR_INVALID_ARG
    assert f(ctypes.byref(P), X, Y, d, None, None, need, None) == wanvae.ERR_WORKSPACE
    assert f(ctypes.byref(P), X, Y, d, None, WS, need - 1, None) == wanvae.ERR_WORKSPACE
    assert f(ctypes.byref(P), X, Y, d, None, WS + 16, need, None) == wanvae.ERR_MISALIGNED
    assert f(ctypes.byref(P), X, X + 32, d, None, WS, need, None) == wanvae.ERR_INVALID_ARG
    P2 = wanvae.ResblockParams(64, 32, 1e-12, A, A, A, A, A, A, None, None)  # no wS, c_in != c_out
    assert f(ctypes.byref(P2), X, Y, d, None, WS, need, None) == wanvae.ERR_INVALID_ARG
    P3 = wanvae.ResblockParams(32, 40, 1e-12, A, A, A, A, A, A, A, None)
    assert f(ctypes.byref(P3), X, Y, d, None, WS, 1 << 30, None) == wanvae.ERR_UNSUPPORTED
    c = wanvae.ResblockCache(0x400000, None)
    assert f(ctypes.byref(P), X, Y, d, ctypes.byref(c), WS, need, None) == wanvae.ERR_INVALID_ARG


def test_valid_call_without_gpu_reports_cuda_error(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    st = lib.wanvae_rmsnorm_silu(A, 0x900000, A, 0, 10, 32, 1e-12, None)
    assert st == wanvae.ERR_CUDA
