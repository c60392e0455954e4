"""Throughput of the Wan 2.2 VAE decoder ResidualBlock forward on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one full-T ResidualBlock forward (RMS_norm1+SiLU, conv A with
RMS_norm2+SiLU fused, conv B with the residual fused) over the full-resolution
clip x bf16 [1, 81, 480, 832, 96] (C_in = C_out = 96, identity shortcut: the
largest block configuration), inputs already resident in HBM.  The metric is
voxels/s (B*T*H*W / step time); the conv's TFLOP/s and its fraction of the
measured bf16 peak (burst, and sustained for this seconds-long region) are
reported in the `roofline` object.  --workload selects the other block
configurations and the decoder's boundary convs and upsampler.

Between timed steps L2 is flushed by writing a 256 MiB buffer (outside the
timed events).  Unless --steps is given, the timed region is sized to last
about 1.5 s, so that the clock sampler sees it many times.
Under torchrun each rank runs its own replica (the block needs no exchange at
one GPU per clip): weak scaling, value = all ranks' voxels / max rank time.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (the only reference this subject has).
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "fullres_96"
METRIC = "ResidualBlock voxels/s (conv TFLOP/s as fraction of bf16 peak in roofline)"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: per workload, ~0.5-1.5 s of GPU time)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--frames", type=int, default=None,
                    help="override the workload's T (smaller cases for profiling); the "
                         "JSON line's config records the dims actually run")
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["tiny", "latent_fullT", "stream_720p", "reduce_384_192",
                             "fullres_96", "conv_in_latent", "post_quant_latent",
                             "conv_out_fullres", "upsample2d_fullres", "time_upsample_latent",
                             "mid_attention_latent"],
                    help="fullres_96 (default) is the headline; the others are the remaining "
                         "workloads of the design notes (the conv_* / post_quant_* ones time "
                         "one CausalConv3d call: the decoder's boundary convs)")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": float(d["bf16_tflops"]), "hbm_gbs": float(d["hbm_gbs"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", 0)) or None,
                "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, source="fallback")


CONV_SOURCES = ("conv3d_tcgen05.cu", "conv3d_tcgen05.cuh", "ptx.cuh", "norm_act.cuh")


def conv_source_sha(files=CONV_SOURCES, root=None):
    """Hash of the kernel sources (in `root`, by default the package's csrc/)
    with comments and blank lines removed (no string literal in them holds a
    comment marker), so that an edited comment does not count as a changed
    kernel."""
    root = root or os.path.join(ROOT, "video_vae_causal_gb300", "csrc")
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(root, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        lines = [ln.rstrip() for ln in text.splitlines() if ln.strip()]
        h.update("\n".join(lines).encode())
    return h.hexdigest()[:16]


def profiled_traffic(name, kernel="conv3d_tcgen05", files=CONV_SOURCES):
    """DRAM bytes per launch of `kernel` in workload `name` from its committed
    ncu summary, if there is one taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{name}.md")
    try:
        kv = {}
        for line in open(path):
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                kv[k.strip()] = v.strip().strip("`")
        if kv.get("source_sha") == conv_source_sha(files):
            return int(kv["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


def max_over_ranks(value, ws, device=None):
    """Max of a per-rank float over all ranks of the default process group
    (identity at world size 1).  Timing only: no data-path collective."""
    if ws <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_throughput(units_per_rank, ws, steps, max_ms):
    """Whole-job units/s when every rank processed units_per_rank per step."""
    return ws * units_per_rank * steps / (max_ms / 1e3)


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples during the timed region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


WORKLOAD_TEXT = {
    "tiny": "tiny: ResidualBlock full-T over x bf16 [1,3,16,16,32], identity shortcut",
    "latent_fullT": "latent_fullT: ResidualBlock full-T over x bf16 [1,21,60,104,384], "
                    "C_in=C_out=384, identity shortcut",
    "stream_720p": "stream_720p: ResidualBlock frame by frame, 21 calls of x bf16 "
                   "[1,1,90,160,384] with a 2-frame feat_cache per conv, C=384",
    "reduce_384_192": "reduce_384_192: ResidualBlock full-T over x bf16 [1,41,240,416,384], "
                      "C_in=384 -> C_out=192, 1x1x1 conv shortcut",
    "fullres_96": "fullres_96: ResidualBlock full-T over x bf16 [1,81,480,832,96], C=96, "
                  "identity shortcut",
    "conv_in_latent": "conv_in_latent: CausalConv3d k=3 over x bf16 [1,21,60,104,16], "
                      "16 -> 384 (the decoder's conv_in), full clip",
    "post_quant_latent": "post_quant_latent: CausalConv3d k=1 over x bf16 [1,21,60,104,16], "
                         "16 -> 16 (the decoder's post_quant_conv)",
    "conv_out_fullres": "conv_out_fullres: CausalConv3d k=3 over x bf16 [1,81,480,832,96], "
                        "96 -> 3 (the decoder's conv_out to RGB), full clip",
    "upsample2d_fullres": "upsample2d_fullres: nearest 2x upsampling + 3x3 conv of x bf16 "
                          "[1,81,240,416,192] -> [1,81,480,832,96] (the last up block's "
                          "upsampler)",
    "time_upsample_latent": "time_upsample_latent: nearest 2x upsampling in T + causal 3x1x1 "
                            "conv of x bf16 [1,21,60,104,384] -> [1,42,60,104,384] (the "
                            "temporal half of the first up block's upsample3d)",
    "mid_attention_latent": "mid_attention_latent: the mid-block's per-frame spatial "
                            "self-attention over x bf16 [1,21,60,104,384] (6240 positions per "
                            "frame, one head of 384, 1x1 q/k/v/out projections, residual)",
}


def workload_config(name, B, T, H, W, ci, co, ws):
    return {"workload": WORKLOAD_TEXT[name],
            "B": B, "T": T, "H": H, "W": W, "c_in": ci, "c_out": co,
            "l2": "flushed between steps (256 MiB write outside the timed events)",
            "parallelism": f"replicas x{ws}"}


def cpu_baseline(x, params, H, W, budget_s=12.0):
    """The oracle, as it stands, on one streaming call of one frame over the
    first `rows` rows of the frame (random caches: every tap does work, like
    an interior frame of the clip), sized to roughly budget_s of CPU time."""
    import numpy as np
    import oracle
    C_in, C_out = params.c_in, params.c_out
    rng = np.random.default_rng(0)

    def run(rows):
        xs = x[:, 2:3, :rows].contiguous().cpu()
        cA = rng.standard_normal((1, 2, rows, W, C_in))
        cB = rng.standard_normal((1, 2, rows, W, C_out))
        t0 = time.perf_counter()
        oracle.resblock_forward(xs, params, cA, cB)
        return time.perf_counter() - t0

    t1 = run(1)
    rows = int(max(1, min(H, budget_s / max(t1, 1e-3))))
    dt = run(rows) if rows > 1 else t1
    vox = rows * W
    return {"value": vox / dt, "unit": "voxels/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"one streaming frame (T=1, feat_cache full of data) over {rows} of {H} rows "
                      f"x {W} columns, C={C_in}->{C_out}: {vox} voxels in {dt:.2f} s"}


def bench_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from video_vae_causal_gb300 import synth
    name = args.workload
    if (name in synth.CONV_WORKLOADS or name in synth.UPSAMPLE_WORKLOADS
            or name in synth.TIME_UPSAMPLE_WORKLOADS):
        return bench_reference_conv(args)
    if name in synth.ATTENTION_WORKLOADS:
        return bench_reference_attention(args)
    dims, ci, co, _ = synth.WORKLOADS[name]
    B, T, H, W = dims
    # The oracle only needs the few rows it runs on: draw the clip's first
    # frames with the same recipe (small workloads: the whole clip).
    x, p = synth.make_resblock_inputs((B, min(T, 3), H, W), ci, co, seed=0)
    params = oracle.Params.from_dict(p)
    steps = args.steps if args.steps else 10
    budget = max(1.0, 60.0 / max(1, steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(x, params, H, W, budget_s=budget)
    vals, samples = [], []
    for _ in range(steps):
        r = cpu_baseline(x, params, H, W, budget_s=budget)
        vals.append(r["value"])
        samples.append(r["sample"])
    v = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v,
        "unit": "voxels/s", "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(name, B, T, H, W, ci, co, 1),
        "cpu_baseline": {"value": v, "unit": "voxels/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": samples[-1]},
        "e2e": {"value": v, "unit": "voxels/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def bench_reference_conv(args):
    """The oracle's CausalConv3d, as it stands, on the host cores: each step
    one bounded sample (the clip's first frames over a band of rows)."""
    import oracle
    from video_vae_causal_gb300 import synth
    name = args.workload
    up = name in synth.UPSAMPLE_WORKLOADS
    upt = name in synth.TIME_UPSAMPLE_WORKLOADS
    if up:
        dims, ci, co = synth.UPSAMPLE_WORKLOADS[name]
        B, T, H, W = dims
        x, w, b = synth.make_upsample_inputs((B, min(T, 3), H, W), ci, co, seed=0)
        fn = oracle.upsample2d_conv
    elif upt:
        dims, ci, co = synth.TIME_UPSAMPLE_WORKLOADS[name]
        B, T, H, W = dims
        x, w, b = synth.make_time_upsample_inputs((B, min(T, 3), H, W), ci, co, seed=0)
        fn = oracle.time_upsample_conv
    else:
        dims, ci, co, k = synth.CONV_WORKLOADS[name]
        B, T, H, W = dims
        x, w, b = synth.make_conv_inputs((B, min(T, 3), H, W), ci, co, k, seed=0)
        fn = oracle.causal_conv3d
    per_row = 4 if up else (2 if upt else 1)  # output voxels per input voxel
    steps = args.steps if args.steps else 10
    budget = max(1.0, 60.0 / max(1, steps + args.warmup))
    t0 = time.perf_counter()
    fn(x[:, :, :1], w, b)
    rows = int(max(1, min(H, budget / max(time.perf_counter() - t0, 1e-3))))
    vals = []
    for i in range(args.warmup + steps):
        t0 = time.perf_counter()
        fn(x[:, :, :rows], w, b)
        if i >= args.warmup:
            vals.append(per_row * x.shape[0] * x.shape[1] * rows * W /
                        (time.perf_counter() - t0))
    v = statistics.median(vals)
    sample = f"the clip's first {x.shape[1]} frames over {rows} of {H} rows x {W} columns"
    print(json.dumps({
        "impl": "reference",
        "metric": metric_name(up, upt),
        "value": v, "unit": "voxels/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup, "ms_per_step": None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(name, B, T, H, W, ci, co, 1),
        "cpu_baseline": {"value": v, "unit": "voxels/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": "voxels/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


TIMED_REGION_S = 1.5  # default length of the timed region (clock samples every 100 ms)
MAX_STEPS = 4000


def e2e_chunk_frames(T, H, W, streaming):
    """Frames per chunk of the end-to-end host pipeline.  Large frames: the
    copies outweigh the block, and only the first chunk's copy-in and the last
    chunk's copy-out overlap nothing, so chunks of about 1/27 of the clip (3
    frames of 81: 818-857 M voxels/s against 587 M with 11-frame chunks, on one
    box).  Small frames: a chunk must still fill the GPU with tiles, so an
    eighth of the clip.  Frame-by-frame decode: one frame."""
    if streaming:
        return 1
    if H * W >= 65536:
        return max(1, -(-T // 27))
    return max(1, -(-T // 8))


def default_steps(args, step_ms):
    """--steps, else enough steps for about TIMED_REGION_S of timed work."""
    if args.steps:
        return args.steps
    return int(min(MAX_STEPS, max(10, -(-TIMED_REGION_S * 1e3 // max(step_ms, 1e-3)))))


def time_one(stream, fn):
    """Device time in ms of fn() on `stream` (CUDA events, synchronised)."""
    import torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    fn()
    b.record(stream)
    torch.cuda.synchronize()
    return a.elapsed_time(b)


def metric_name(up, upt):
    what = ("Upsampler output voxels/s" if up else
            "Temporal upsampler output voxels/s" if upt else "CausalConv3d voxels/s")
    return what + " (roofline: the bound its arithmetic intensity sets)"


def bench_reference_attention(args):
    """The oracle's attention, as it stands, on the host cores: each step one
    frame of the workload (all its queries against all its keys)."""
    import oracle
    from video_vae_causal_gb300 import synth
    name = args.workload
    dims, C = synth.ATTENTION_WORKLOADS[name]
    B, T, H, W = dims
    x, g, wqkv, bqkv, wo, bo = synth.make_attention_inputs((1, 1, H, W), C, seed=0)
    steps = args.steps if args.steps else 3
    vals = []
    for i in range(args.warmup + steps):
        t0 = time.perf_counter()
        oracle.frame_attention(x, g, wqkv, bqkv, wo, bo)
        if i >= args.warmup:
            vals.append(H * W / (time.perf_counter() - t0))
    v = statistics.median(vals)
    print(json.dumps({
        "impl": "reference", "metric": ATTN_METRIC, "value": v, "unit": "voxels/s",
        "n_gpus": args.gpus, "steps": steps, "warmup": args.warmup, "ms_per_step": None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(name, B, T, H, W, C, C, 1),
        "cpu_baseline": {"value": v, "unit": "voxels/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": f"one {H}x{W} frame per step"},
        "e2e": {"value": v, "unit": "voxels/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


ATTN_METRIC = "Attention block voxels/s (roofline: the attention core's TFLOP/s)"


def bench_attention(args):
    """One attention-block call per step: device time by CUDA events around
    the call, the core's FLOPs (4 N^2 C per frame) against the bf16 peak, end
    to end with host buffers, and the oracle on one frame."""
    import torch

    from video_vae_causal_gb300 import synth, wanvae

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    if ws > 1:
        raise RuntimeError("the attention workload runs on one GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    wanvae.load()
    name = args.workload
    dims, C = synth.ATTENTION_WORKLOADS[name]
    if args.frames:
        dims = (dims[0], args.frames) + tuple(dims[2:])
    B, T, H, W = dims
    N, F, M = H * W, B * T, B * T * H * W
    x, g, wqkv, bqkv, wo, bo = synth.make_attention_inputs(dims, C, seed=0)
    x_cpu = x
    x, g, wqkv, bqkv, wo, bo = (t.to(dev) for t in (x, g, wqkv, bqkv, wo, bo))
    y = torch.empty_like(x)
    nws = int(wanvae.load().wanvae_frame_attention_workspace_size(wanvae._dims(x.shape), C))
    wsb = torch.empty(nws, dtype=torch.uint8, device=dev)

    def call(xin):
        wanvae.frame_attention(xin, g, wqkv, bqkv, wo, bo, y=y, workspace=wsb)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        call(x)
    torch.cuda.synchronize(dev)
    K = default_steps(args, time_one(stream, lambda: call(x)))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    n0 = wanvae.launch_count()
    with ClockSampler(local) as clk:
        for e in evs:
            flush.zero_()
            e[0].record(stream)
            call(x)
            e[1].record(stream)
        torch.cuda.synchronize(dev)
    launches = wanvae.launch_count() - n0
    wanvae.sync_status()
    ms = sum(a.elapsed_time(z) for a, z in evs) / K
    value = M / (ms / 1e3)
    x_host = x_cpu.pin_memory()
    y_host = torch.empty(x.shape, dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    E = max(1, min(args.e2e_steps, K))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        x_dev.copy_(x_host, non_blocking=True)
        call(x_dev)
        y_host.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_value = M * E / (e0.elapsed_time(e1) / 1e3)
    peaks = load_peaks()
    flop_core = 4.0 * F * N * N * C                # Q K^T and P V
    flop_proj = 2.0 * 4 * M * C * C                # q, k, v and output projections
    tflops = (flop_core + flop_proj) / (ms / 1e3) / 1e12
    line = {
        "metric": ATTN_METRIC, "value": value, "unit": "voxels/s", "n_gpus": 1, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(name, B, T, H, W, C, C, 1),
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"],
                     "flop_per_launch": flop_core + flop_proj, "kernel": "whole block",
                     "traffic": None,
                     "peak_source": peaks["source"] + " bf16 burst"},
        "e2e": {"value": e2e_value, "unit": "voxels/s", "h2d_bytes_per_step": x.numel() * 2,
                "d2h_bytes_per_step": y.numel() * 2, "steps": E},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline:
        import oracle
        xs = x_cpu[:1, :1]
        t0 = time.perf_counter()
        oracle.frame_attention(xs, g.cpu(), wqkv.cpu(), bqkv.cpu(), wo.cpu(), bo.cpu())
        dt = time.perf_counter() - t0
        line["cpu_baseline"] = {"value": N / dt, "unit": "voxels/s",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": f"one {H}x{W} frame: {N} voxels in {dt:.2f} s"}
    print(json.dumps(line), flush=True)




def bench_conv(args):
    """One CausalConv3d call per step (the decoder's boundary convs): device
    time by CUDA events around the call, end to end with host buffers, the
    roofline of the conv against whichever of the tensor and HBM peaks its
    arithmetic intensity makes binding, and the oracle on a bounded sample."""
    import torch
    import torch.distributed as dist

    from video_vae_causal_gb300 import synth, wanvae

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    wanvae.load()
    name = args.workload
    up = name in synth.UPSAMPLE_WORKLOADS
    upt = name in synth.TIME_UPSAMPLE_WORKLOADS
    if up:
        dims, ci, co = synth.UPSAMPLE_WORKLOADS[name]
        k = 3
    elif upt:
        dims, ci, co = synth.TIME_UPSAMPLE_WORKLOADS[name]
        k = 3
    else:
        dims, ci, co, k = synth.CONV_WORKLOADS[name]
    if args.frames:
        dims = (dims[0], args.frames) + tuple(dims[2:])
    B, T, H, W = dims
    Ho, Wo = (2 * H, 2 * W) if up else (H, W)
    To = 2 * T if upt else T
    M = B * To * Ho * Wo                      # output voxels
    on_dev = M * max(ci, co) > (1 << 30)
    make = (synth.make_upsample_inputs if up else synth.make_time_upsample_inputs if upt else
            lambda d, a, c, seed, device: synth.make_conv_inputs(d, a, c, k, seed=seed,
                                                                 device=device))
    x, w, b = make(dims, ci, co, seed=0, device=dev if on_dev else "cpu")
    x_cpu = None if on_dev else x
    w_cpu, b_cpu = w.cpu(), b.cpu()
    x, w, b = x.to(dev), w.to(dev), b.to(dev)
    y = torch.empty((B, To, Ho, Wo, co), dtype=torch.bfloat16, device=dev)
    ws_up = None
    if up:
        n = int(wanvae.load().wanvae_upsample2d_workspace_size(ci, co))
        ws_up = torch.empty(n, dtype=torch.uint8, device=dev)
    elif upt:
        n = int(wanvae.load().wanvae_time_upsample_workspace_size(ci, co))
        ws_up = torch.empty(n, dtype=torch.uint8, device=dev)

    def call(xin):
        if up:
            wanvae.upsample2d_conv(xin, w, b, y=y, workspace=ws_up)
        elif upt:
            wanvae.time_upsample_conv(xin, w, b, y=y, workspace=ws_up)
        else:
            wanvae.causal_conv3d(xin, w, b, y=y)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        call(x)
    torch.cuda.synchronize(dev)
    K = default_steps(args, time_one(stream, lambda: call(x)))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    n0 = wanvae.launch_count()
    with ClockSampler(local) as clk:
        for e in evs:
            flush.zero_()
            e[0].record(stream)
            call(x)
            e[1].record(stream)
        torch.cuda.synchronize(dev)
    launches = wanvae.launch_count() - n0
    wanvae.sync_status()
    total_ms = max_over_ranks(sum(a.elapsed_time(z) for a, z in evs), ws, dev)
    ms = total_ms / K
    value = replica_throughput(M, ws, K, total_ms)

    if x_cpu is None:
        x_cpu = x.cpu()
    x_host = x_cpu.pin_memory()
    y_host = torch.empty((B, To, Ho, Wo, co), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    E = max(1, min(args.e2e_steps, K))
    for _ in range(2):
        x_dev.copy_(x_host, non_blocking=True)
        call(x_dev)
        y_host.copy_(y, non_blocking=True)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        x_dev.copy_(x_host, non_blocking=True)
        call(x_dev)
        y_host.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_value = replica_throughput(M, ws, E, max_over_ranks(e0.elapsed_time(e1), ws, dev))

    peaks = load_peaks()
    # useful work (a padded N is not counted).  The upsampler: the 2 x 2 sub-pixel
    # conv each output voxel reduces to exactly (the 3 x 3 conv of the upsampled
    # frame would count 9 taps instead of 4: reported beside it, not used).  The
    # temporal upsampler likewise: 2 taps per output voxel, not the 3 of the
    # 3x1x1 conv over the repeated frames.
    flop = 2.0 * (4 if up else 2 if upt else k ** 3) * ci * co * M
    nbytes = (ci * 2.0 * B * T * H * W + co * 2.0 * M + w.numel() * 2.0 + co * 4.0)  # x, y once
    tflops = flop / (ms / 1e3) / 1e12
    gbs = nbytes / (ms / 1e3) / 1e9
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    tensor = {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"],
              "unit": "TFLOP/s", "frac": tflops / peaks["bf16_tflops"], "flop_per_launch": flop}
    if up:
        tensor["flop_per_launch_3x3_on_upsampled"] = 2.0 * 9 * ci * co * M
    if upt:
        tensor["flop_per_launch_3x1x1_on_upsampled"] = 2.0 * 3 * ci * co * M
    hbm = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
           "frac": gbs / peaks["hbm_gbs"], "bytes_per_launch": nbytes}
    main, other = (tensor, hbm) if flop / nbytes >= ridge else (hbm, tensor)
    narrow = not up and not upt and ci >= 32 and ci % 32 == 0 and ci <= 128 and co <= 3 and k == 3
    kname = "conv3d_narrow" if narrow else "conv3d_tcgen05"
    traffic = None if args.frames else profiled_traffic(
        name, kname, ("conv3d_narrow.cu", "ptx.cuh") if narrow else CONV_SOURCES)
    main.update({"kernel": kname + "_kernel", "traffic": traffic,
                 "peak_source": peaks["source"] + (" bf16 burst" if main is tensor else " HBM copy"),
                 "arith_intensity_flop_per_byte": flop / nbytes, "ridge_flop_per_byte": ridge})
    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": metric_name(up, upt),
        "value": value, "unit": "voxels/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": workload_config(name, B, T, H, W, ci, co, ws),
        "roofline": main, "roofline_other": other,
        "e2e": {"value": e2e_value, "unit": "voxels/s", "h2d_bytes_per_step": x.numel() * 2,
                "d2h_bytes_per_step": y.numel() * 2, "steps": E},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
    }
    if not args.no_cpu_baseline and ws == 1:
        import oracle
        # The oracle on the first frames of the clip over as many rows as fit ~10 s.
        xs = x_cpu[:, :min(T, 3)]
        fn = (oracle.upsample2d_conv if up else oracle.time_upsample_conv if upt else
              oracle.causal_conv3d)
        t0 = time.perf_counter()
        fn(xs[:, :, :1], w_cpu, b_cpu)
        t1 = max(time.perf_counter() - t0, 1e-3)
        rows = int(max(1, min(H, 10.0 / t1)))
        t0 = time.perf_counter()
        fn(xs[:, :, :rows], w_cpu, b_cpu)
        dt = time.perf_counter() - t0
        vox = xs.shape[0] * xs.shape[1] * rows * W * (4 if up else 2 if upt else 1)  # output
        line["cpu_baseline"] = {"value": vox / dt, "unit": "voxels/s",
                                "cores": oracle.num_threads(), "kind": "oracle",
                                "sample": f"the clip's first {xs.shape[1]} frames over {rows} "
                                          f"of {H} rows x {W} columns: {vox} voxels in {dt:.2f} s"}
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def bench_ours(args):
    import torch
    import torch.distributed as dist

    from video_vae_causal_gb300 import synth, wanvae

    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise RuntimeError("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if ws > 1:
        dist.init_process_group("nccl", device_id=dev)
    wanvae.load()

    name = args.workload
    dims, ci, co, calls = synth.WORKLOADS[name]
    if args.frames:
        dims = (dims[0], args.frames) + tuple(dims[2:])
    B, T, H, W = dims
    M = B * T * H * W
    streaming = calls > 0
    # Small workloads are drawn on the CPU generator, the multi-GB ones on the
    # device generator (same recipe, different stream of numbers).
    on_dev = M * max(ci, co) > (1 << 30)
    x, p = synth.make_resblock_inputs(dims, ci, co, seed=0, device=dev if on_dev else "cpu")
    x_cpu = None if on_dev else x
    p_cpu = {k: v.cpu() for k, v in p.items()}
    x = x.to(dev)
    p = {k: v.to(dev) for k, v in p.items()}
    params = wanvae.make_params(p)
    y = torch.empty((B, T, H, W, co), dtype=torch.bfloat16, device=dev)
    call_dims = (B, 1, H, W) if streaming else dims
    wsp = wanvae.make_workspace(call_dims, ci, co, device=dev)
    caches = None
    if streaming:
        caches = (torch.zeros((B, 2, H, W, ci), dtype=torch.bfloat16, device=dev),
                  torch.zeros((B, 2, H, W, co), dtype=torch.bfloat16, device=dev))
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    ncalls = T if streaming else 1

    def forward(xin, events=None):
        """One step: the whole clip, full-T or frame by frame with feat_cache."""
        if not streaming:
            wanvae.resblock_forward(xin, params, y=y, workspace=wsp,
                                    events=events[0] if events else None)
            return
        for c in caches:
            c.zero_()  # a new clip starts with empty caches (before the first event)
        for t in range(T):
            wanvae.resblock_forward(xin[:, t:t + 1], params, y=y[:, t:t + 1], cache=caches,
                                    workspace=wsp, events=events[t] if events else None)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        forward(x)
    wanvae.sync_status()

    K = default_steps(args, time_one(stream, lambda: forward(x)))
    # The timed region: K steps of plain calls, a CUDA event pair around each
    # step (the L2 flush between steps stays outside the events).
    step_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    n0 = wanvae.launch_count()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for k in range(K):
            flush.zero_()
            step_ev[k][0].record(stream)
            forward(x)
            step_ev[k][1].record(stream)
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches = wanvae.launch_count() - n0
    wanvae.sync_status()
    step_ms = [a.elapsed_time(b) for a, b in step_ev]
    total_ms = max_over_ranks(sum(step_ms), ws, dev)
    ms_per_step = total_ms / K
    value = replica_throughput(M, ws, K, total_ms)

    # The kernels inside a step: a second timed pass of Kp steps through the
    # profiled call, which records CUDA events between its kernels (events
    # between the launches keep the next kernel from starting early, so this
    # pass is not the one the step time comes from).
    Kp = max(3, min(K, int(K * 0.25) + 1))
    evs = [[[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(ncalls)]
           for _ in range(Kp)]
    for step_e in evs:
        for e4 in step_e:
            for e in e4:
                e.record(stream)
    torch.cuda.synchronize(dev)
    for k in range(Kp):
        flush.zero_()
        forward(x, evs[k])
    torch.cuda.synchronize(dev)
    wanvae.sync_status()
    prof_step_ms = [e[0][0].elapsed_time(e[-1][3]) for e in evs]
    norm_ms = [sum(c[0].elapsed_time(c[1]) for c in e) for e in evs]
    convA_ms = [sum(c[1].elapsed_time(c[2]) for c in e) for e in evs]
    convB_ms = [sum(c[2].elapsed_time(c[3]) for c in e) for e in evs]

    # ---- end to end through the public API with host buffers: the clip in
    # pinned host memory, chunked in T over the feat_cache and pipelined over
    # three streams (copy in / compute / copy out); streaming workloads run
    # frame by frame, as in the timed loop above
    if x_cpu is None:
        x_cpu = x.cpu()
    x_host = x_cpu.pin_memory()
    y_host = torch.empty((B, T, H, W, co), dtype=torch.bfloat16).pin_memory()
    chunk = e2e_chunk_frames(T, H, W, streaming)
    hws = torch.empty(wanvae.resblock_forward_host_workspace_size(dims, ci, co, chunk),
                      dtype=torch.uint8, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    streams = (stream, s_in, s_out)
    E = max(1, min(args.e2e_steps, K))

    def e2e_step():
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        wanvae.resblock_forward_host(x_host, params, y_host, chunk, hws, streams)
        stream.wait_stream(s_out)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    e2e_value = replica_throughput(M, ws, E, e2e_ms)
    if not torch.equal(y_host, y.cpu()):
        raise RuntimeError("the host-buffer pipeline's output differs from the device run")

    # ---- roofline of the dominant kernel (the conv: two launches per call)
    peaks = load_peaks()
    flop_A = 2.0 * 27 * ci * co * M
    flop_B = 2.0 * 27 * co * co * M + (2.0 * ci * co * M if ci != co else 0.0)
    n_conv_launches = 2 * ncalls
    flop_conv = (flop_A + flop_B) / n_conv_launches          # per launch, averaged
    conv_ms = (sum(convA_ms) + sum(convB_ms)) / (Kp * n_conv_launches)
    achieved = flop_conv / (conv_ms / 1e3) / 1e12
    norm_gbs = (2.0 * ci * 2 * M) / (statistics.mean(norm_ms) / 1e3) / 1e9
    traffic = profiled_traffic(name) if not args.frames else None
    block_flop = flop_A + flop_B
    # Of a full clip's 27 T taps per voxel, frames 0 and 1 have 18 and 9 in the
    # causal pad: 27 of 27 T per pixel.  Streaming calls read the cache instead.
    nonpad = 1.0 if streaming else 1.0 - 1.0 / T

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC,
        "value": value, "unit": "voxels/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(name, B, T, H, W, ci, co, ws),
        "block_tflops": block_flop / (ms_per_step / 1e3) / 1e12,
        "kernels_ms": {"rmsnorm_silu": statistics.mean(norm_ms),
                       "conv3d_A_normsilu": statistics.mean(convA_ms),
                       "conv3d_B_residual": statistics.mean(convB_ms),
                       "profiled_step": statistics.mean(prof_step_ms),
                       "profiled_steps": Kp,
                       "note": "a second timed pass through wanvae_resblock_forward_profiled "
                               "(CUDA events between the kernels); the step time above "
                               "comes from plain calls"},
        "roofline": {"bound": "tensor", "kernel": "conv3d_tcgen05_kernel",
                     "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                     "peak_source": peaks["source"] + " bf16 burst",
                     "peak_sustained": peaks.get("bf16_tflops_sustained"),
                     "frac_of_sustained": (achieved / peaks["bf16_tflops_sustained"]
                                           if peaks.get("bf16_tflops_sustained") else None),
                     "flop_per_launch": flop_conv,
                     # the dense conv definition counts the causal-pad taps as work
                     # (frames t < 2 read zeros); the kernel skips most of them
                     "padded_taps_counted": True,
                     "nonpad_tap_fraction": nonpad,
                     "achieved_nonpad_taps": achieved * nonpad},
        "norm_roofline": {"bound": "hbm", "achieved": norm_gbs, "peak": peaks["hbm_gbs"],
                          "unit": "GB/s", "frac": norm_gbs / peaks["hbm_gbs"]},
        "e2e": {"value": e2e_value, "unit": "voxels/s", "h2d_bytes_per_step": x.numel() * 2,
                "d2h_bytes_per_step": y.numel() * 2, "steps": E,
                "call": "wanvae_resblock_forward_host (pinned host x and y; chunks of %d "
                        "frame(s) over the feat_cache, copy in / compute / copy out on three "
                        "streams)" % chunk},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "wall_s_timed": t_wall,
    }
    if streaming:
        line["per_call_ms"] = ms_per_step / ncalls
        line["kernels_ms_note"] = ("per step of %d calls; the conv intervals include each "
                                   "call's feat_cache update kernel" % ncalls)
    if not args.no_cpu_baseline and ws == 1:
        import oracle
        line["cpu_baseline"] = cpu_baseline(x_cpu, oracle.Params.from_dict(p_cpu), H, W)
    print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.impl == "reference":
        bench_reference(args)
    elif args.workload in ("conv_in_latent", "post_quant_latent", "conv_out_fullres",
                           "upsample2d_fullres", "time_upsample_latent"):
        bench_conv(args)
    elif args.workload == "mid_attention_latent":
        bench_attention(args)
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
