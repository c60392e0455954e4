"""bench.py's host-side helpers on CPU: the kernel-source hash that decides
whether a committed ncu summary still describes the kernel, the lookup of its
traffic figure, and the end-to-end pipeline's chunking."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _write(d, name, text):
    with open(os.path.join(d, name), "w") as f:
        f.write(text)


def test_source_hash_ignores_comments_but_not_code(tmp_path):
    d = str(tmp_path)
    code = "// header\nint f(int x) {  // doubles\n    return 2 * x;\n}\n/* block\n comment */\n"
    _write(d, "k.cu", code)
    h0 = bench.conv_source_sha(("k.cu",), root=d)
    _write(d, "k.cu", "// another header\n\nint f(int x) {  // twice x\n    return 2 * x;\n}\n")
    assert bench.conv_source_sha(("k.cu",), root=d) == h0
    _write(d, "k.cu", "int f(int x) {\n    return 3 * x;\n}\n")
    assert bench.conv_source_sha(("k.cu",), root=d) != h0


def test_profiled_traffic_matches_the_committed_summaries():
    # every summary under profiles/ that carries a source hash was taken on
    # the kernel source as it stands, so bench.py reports its traffic
    for name in ("fullres_96", "latent_fullT", "stream_720p", "reduce_384_192",
                 "conv_in_latent", "upsample2d_fullres", "time_upsample_latent"):
        t = bench.profiled_traffic(name)
        assert isinstance(t, int) and t > 0, name
    t = bench.profiled_traffic("conv_out_fullres", "conv3d_narrow",
                               ("conv3d_narrow.cu", "ptx.cuh"))
    assert isinstance(t, int) and t > 0
    assert bench.profiled_traffic("no_such_workload") is None


def test_e2e_chunking():
    assert bench.e2e_chunk_frames(81, 480, 832, False) == 3   # the full-resolution clip
    assert bench.e2e_chunk_frames(21, 60, 104, False) == 3    # the latent clip
    assert bench.e2e_chunk_frames(21, 90, 160, True) == 1     # frame-by-frame decode
    assert bench.e2e_chunk_frames(1, 480, 832, False) == 1
