"""The allocation-free ResidualBlock entry point (wanvae_resblock_forward_static).

It serves callers that cannot allocate device memory where they run the
block: its workspace is the library's own fixed-size device array.  It runs
the same kernels on the same inputs as the regular entry point (caller
workspace), so its output must equal that entry point's bit for bit, call
after call (the array keeps the previous call's contents), and sizes beyond
the array are refused before anything is enqueued.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import pytest
import torch

from video_vae_causal_gb300 import synth

pytestmark = pytest.mark.gpu


def _run_both(lib, dims, ci, co, seed):
    x, p = synth.make_resblock_inputs(dims, ci, co, seed=seed, device="cuda")
    params = lib.make_params(p)
    y_ref = lib.resblock_forward(x, params)
    y_static = torch.empty_like(y_ref)
    lib.resblock_forward_static(x, params, y_static)
    lib.sync_status()
    return x, p, y_ref, y_static


@pytest.mark.parametrize("dims,ci,co", [((1, 3, 16, 16), 32, 32),
                                        ((1, 2, 9, 13), 64, 32),
                                        ((1, 1, 90, 160), 384, 384)])
def test_static_matches_caller_workspace_two_calls_in_a_row(cuda_lib, dims, ci, co):
    for seed in (1, 2):  # second call reuses the array the first one left behind
        _, _, y_ref, y_static = _run_both(cuda_lib, dims, ci, co, seed)
        assert torch.equal(y_static, y_ref), f"static vs workspace seed={seed}"
        assert torch.isfinite(y_static.float()).all()


def test_static_streaming_two_frames_matches(cuda_lib):
    dims, ci, co = (1, 2, 12, 20), 64, 64
    x, p = synth.make_resblock_inputs(dims, ci, co, seed=3, device="cuda")
    params = cuda_lib.make_params(p)
    B, T, H, W = dims
    caches = [tuple(torch.zeros((B, 2, H, W, c), dtype=torch.bfloat16, device="cuda")
                    for c in (ci, co)) for _ in range(2)]
    for t in range(T):
        xt = x[:, t:t + 1].contiguous()
        y_ref = cuda_lib.resblock_forward(xt, params, cache=caches[0])
        y_st = cuda_lib.resblock_forward_static(xt, params, torch.empty_like(y_ref),
                                                cache=caches[1])
        cuda_lib.sync_status()
        assert torch.equal(y_st, y_ref), f"static streaming t={t}"
    assert torch.equal(caches[0][0], caches[1][0]) and torch.equal(caches[0][1], caches[1][1])


def test_static_rejects_sizes_beyond_its_array(cuda_lib):
    dims, ci, co = (1, 21, 60, 104), 384, 384
    assert cuda_lib.resblock_workspace_size(dims, ci, co) > cuda_lib.STATIC_WORKSPACE_BYTES
    x = torch.zeros((1, 21, 60, 104, ci), dtype=torch.bfloat16, device="cuda")
    y = torch.full((1, 21, 60, 104, co), 7.0, dtype=torch.bfloat16, device="cuda")
    _, p = synth.make_resblock_inputs((1, 1, 1, 1), ci, co, seed=0, device="cuda")
    with pytest.raises(cuda_lib.WanvaeError) as ei:
        cuda_lib.resblock_forward_static(x, cuda_lib.make_params(p), y)
    assert ei.value.status == cuda_lib.ERR_WORKSPACE
    cuda_lib.sync_status()
    assert torch.all(y == 7.0)  # nothing was enqueued
