"""Throughput of the Wan 2.2 VAE decoder ResidualBlock forward on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step = one full-T ResidualBlock forward (RMS_norm1+SiLU, conv A with
RMS_norm2+SiLU fused, conv B with the residual fused) over the latent-res clip
x bf16 [1, 21, 60, 104, 384] (C_in = C_out = 384), inputs already resident in
HBM.  The metric is voxels/s (B*T*H*W / step time); the conv's TFLOP/s and its
fraction of the measured bf16 peak are reported in the `roofline` object.

Between timed steps L2 is flushed by writing a 256 MiB buffer (outside the
timed events; the inputs themselves are ~100 MB, below L2's 129 MB).
Under torchrun each rank runs its own replica (the block needs no exchange at
one GPU per clip): weak scaling, value = all ranks' voxels / max rank time.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload (the only reference this subject has).
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "latent_fullT"
METRIC = "ResidualBlock voxels/s (conv TFLOP/s as fraction of bf16 peak in roofline)"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=30)
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


def conv_source_sha():
    h = hashlib.sha256()
    for f in ("conv3d_tcgen05.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "video_vae_causal_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per conv launch from the committed ncu summary, if it was
    taken on the current conv source (else None)."""
    path = os.path.join(ROOT, "profiles", "conv3d_tcgen05_latent_fullT.md")
    try:
        kv = {}
        for line in open(path):
            if line.startswith("- ") and ":" in line:
                k, v = line[2:].split(":", 1)
                kv[k.strip()] = v.strip().strip("`")
        if kv.get("source_sha") == conv_source_sha():
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


def workload_config(B, T, H, W, ci, co, ws):
    return {"workload": "latent_fullT: ResidualBlock full-T over x bf16 [1,21,60,104,384], "
                        "C_in=C_out=384, identity shortcut",
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
        xs = x[:, 2:3, :rows].contiguous()
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
    import torch
    import oracle
    from video_vae_causal_gb300 import synth
    dims, ci, co, _ = synth.WORKLOADS[WORKLOAD]
    B, T, H, W = dims
    x, p = synth.make_resblock_inputs(dims, ci, co, seed=0)
    params = oracle.Params.from_dict(p)
    budget = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(x, params, H, W, budget_s=budget)
    vals, samples = [], []
    for _ in range(args.steps):
        r = cpu_baseline(x, params, H, W, budget_s=budget)
        vals.append(r["value"])
        samples.append(r["sample"])
    v = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": v,
        "unit": "voxels/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": workload_config(B, T, H, W, ci, co, 1),
        "cpu_baseline": {"value": v, "unit": "voxels/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": samples[-1]},
        "e2e": {"value": v, "unit": "voxels/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


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

    dims, ci, co, _ = synth.WORKLOADS[WORKLOAD]
    B, T, H, W = dims
    M = B * T * H * W
    x_cpu, p_cpu = synth.make_resblock_inputs(dims, ci, co, seed=0)
    x = x_cpu.to(dev)
    p = {k: v.to(dev) for k, v in p_cpu.items()}
    params = wanvae.make_params(p)
    y = torch.empty((B, T, H, W, co), dtype=torch.bfloat16, device=dev)
    wsp = wanvae.make_workspace(dims, ci, co, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(events=None):
        wanvae.resblock_forward(x, params, y=y, workspace=wsp, events=events)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    wanvae.sync_status()

    K = args.steps
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for e4 in evs:
        for e in e4:
            e.record(stream)
    torch.cuda.synchronize(dev)
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    n0 = wanvae.launch_count()
    with ClockSampler(local) as clk:
        t_wall = time.perf_counter()
        for k in range(K):
            flush.zero_()
            step(evs[k])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall
    if ws > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    launches = wanvae.launch_count() - n0
    wanvae.sync_status()

    step_ms = [e[0].elapsed_time(e[3]) for e in evs]
    norm_ms = [e[0].elapsed_time(e[1]) for e in evs]
    convA_ms = [e[1].elapsed_time(e[2]) for e in evs]
    convB_ms = [e[2].elapsed_time(e[3]) for e in evs]
    total_ms = max_over_ranks(sum(step_ms), ws, dev)
    ms_per_step = total_ms / K
    value = replica_throughput(M, ws, K, total_ms)

    # ---- end to end through the public API with host buffers
    x_host = x_cpu.pin_memory()
    y_host = torch.empty((B, T, H, W, co), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty_like(x)
    E = max(1, min(args.e2e_steps, K))
    for _ in range(2):
        x_dev.copy_(x_host, non_blocking=True)
        wanvae.resblock_forward(x_dev, params, y=y, workspace=wsp)
        y_host.copy_(y, non_blocking=True)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(E):
        x_dev.copy_(x_host, non_blocking=True)
        wanvae.resblock_forward(x_dev, params, y=y, workspace=wsp)
        y_host.copy_(y, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
    e2e_value = replica_throughput(M, ws, E, e2e_ms)

    # ---- roofline of the dominant kernel (the conv)
    peaks = load_peaks()
    flop_conv = 2.0 * 27 * ci * co * M  # conv A; conv B is 2*27*co*co*M (equal here)
    conv_ms = (sum(convA_ms) + sum(convB_ms)) / (2 * K)
    achieved = flop_conv / (conv_ms / 1e3) / 1e12
    norm_gbs = (2.0 * ci * 2 * M) / (statistics.mean(norm_ms) / 1e3) / 1e9
    traffic = profiled_traffic()
    block_flop = 2.0 * 27 * M * (ci * co + co * co) + (2.0 * ci * co * M if ci != co else 0.0)

    if rank != 0:
        if ws > 1:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC,
        "value": value, "unit": "voxels/s", "n_gpus": ws, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": workload_config(B, T, H, W, ci, co, ws),
        "block_tflops": block_flop / (ms_per_step / 1e3) / 1e12,
        "kernels_ms": {"rmsnorm_silu": statistics.mean(norm_ms),
                       "conv3d_A_normsilu": statistics.mean(convA_ms),
                       "conv3d_B_residual": statistics.mean(convB_ms)},
        "roofline": {"bound": "tensor", "kernel": "conv3d_tcgen05_kernel",
                     "achieved": achieved, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["bf16_tflops"], "traffic": traffic,
                     "peak_source": peaks["source"] + " bf16 burst",
                     "flop_per_launch": flop_conv},
        "norm_roofline": {"bound": "hbm", "achieved": norm_gbs, "peak": peaks["hbm_gbs"],
                          "unit": "GB/s", "frac": norm_gbs / peaks["hbm_gbs"]},
        "e2e": {"value": e2e_value, "unit": "voxels/s", "h2d_bytes_per_step": x.numel() * 2,
                "d2h_bytes_per_step": y.numel() * 2, "steps": E},
        "gpu_launches": int(launches),
        "clocks": clk.summary(),
        "wall_s_timed": t_wall,
    }
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
    else:
        bench_ours(args)


if __name__ == "__main__":
    main()
