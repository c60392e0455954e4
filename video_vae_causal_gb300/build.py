"""Compile the CUDA library libwanvae.so in-tree for sm_103a.

nvcc only (no CMake): each .cu file is compiled in parallel, then linked into
``video_vae_causal_gb300/libwanvae.so`` with a version script that exports the
``wanvae_*`` C symbols and nothing else.
"""
import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libwanvae.so")
SOURCES = ["api.cu", "rmsnorm_silu.cu", "conv3d_tcgen05.cu", "conv3d_narrow.cu",
           "attn_tcgen05.cu", "conv3d_kernels_p1_n1.cu", "conv3d_kernels_p1_n2.cu",
           "conv3d_kernels_p2_n1.cu", "conv3d_kernels_p2_n2.cu", "conv3d_kernels_misc.cu",
           "conv3d_kernels_fuse.cu"]
DEPS = SOURCES + ["ptx.cuh", "kernels.h", "exports.map", "conv3d_tcgen05.cuh",
                  "conv3d_kernels.inc", "norm_act.cuh"]
HEADER = os.path.join(ROOT, "include", "wanvae.h")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
         "-I" + os.path.join(ROOT, "include")]


def nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libwanvae.so")
    return exe


def _stale():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    srcs = [os.path.join(CSRC, f) for f in DEPS] + [HEADER, __file__]
    return any(os.path.getmtime(s) > t for s in srcs)


def build(force=False, verbose=False, extra_flags=()):
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(" ".join(cmd))
            if r.stderr.strip():
                print(r.stderr)
        return obj

    # largest translation units first, all of them in parallel
    with cf.ThreadPoolExecutor(min(len(SOURCES), max(2, os.cpu_count() or 2))) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs,
           "-Xlinker", "--version-script=" + os.path.join(CSRC, "exports.map")]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    if verbose:
        print(" ".join(cmd))
    return LIB


if __name__ == "__main__":
    extra = [a for a in sys.argv[1:] if a.startswith("-X") or a.startswith("--")]
    print(build(force=True, verbose=True,
                extra_flags=[a for a in extra if a != "--force"]))
