"""Throughput of batched Gram Newton-Schulz on GB300.

Workload: one bucket of 24 fp32 matrices of 1024 x 4096 (MLP-like, alpha = 4),
entries N(0, 1) from a seed, orthogonalized in place per step (5 quintic steps,
restart after step 2). A step is one gns_orthogonalize_batched call over the
whole bucket. The input (384 MiB) is larger than the 129 MB L2, so nothing is
flushed between steps. Each step orthogonalizes the previous step's output
(same work, same shapes).

Prints one JSON line. `value` is matrices/s over all ranks (device-timed,
CUDA events); `e2e` is the same metric through the host-buffer C entry point
(pinned host -> device copy, compute, device -> host copy inside the timed
region); `roofline` is the dominant kernel (the tcgen05 GEMM) against the
measured dense fp16/bf16 peak; `cpu_baseline` is the fp64 oracle timed on
this host's cores on a bounded sample.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

G, R, C = 24, 1024, 4096
T_STEPS, RESTART = 5, 2
WORKLOAD = "mlp_bucket_24x1024x4096_fp32"
METRIC = "matrices/sec (batched Gram Newton-Schulz, bucket of 24 fp32 1024x4096)"
UNIT = "matrices/s"


def alg_flops_per_matrix(n, m, steps=T_STEPS):
    """(4T + 6 alpha - 6) n^3 with one restart: the work restarted Gram NS must do
    (Dion3 §4.1 plus the restart cost of §4.2)."""
    return 4 * steps * n ** 3 + 6 * m * n * n - 6 * n ** 3


def eff_flops_per_matrix(n, m, steps=T_STEPS):
    """Standard-NS FLOPs T (4 m n^2 + 2 n^3) (Dion3 §2.2)."""
    return steps * (4 * m * n * n + 2 * n ** 3)


def config_dict(world):
    return {"workload": WORKLOAD if G == 24 else f"mlp_bucket_{G}x1024x4096_fp32", "G_per_gpu": G, "R": R, "C": C, "ns_steps": T_STEPS, "restart_at": RESTART,
            "coeffs": "constant quintic (3.4445, -4.7750, 2.0315)", "storage": "fp16 operands, fp32 accumulate",
            "l2": "inputs larger than L2 (384 MiB fp32 bucket per GPU), no flush",
            "parallelism": f"independent buckets, one per GPU ({world} GPU)"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"tflops": float(p["bf16_tflops"]), "tflops_sustained": float(p["bf16_tflops_sustained"]),
                "hbm_gbs": float(p["hbm_gbs"]), "source": "measured"}
    except Exception:
        return {"tflops": 1900.0, "tflops_sustained": 1700.0, "hbm_gbs": 6800.0, "source": "fallback"}


def gemm_source_hash():
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "gemm.cuh", "ptx.cuh"):
        with open(os.path.join(ROOT, "newton_schulz_gram_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per GEMM launch from the committed ncu summary, if it was
    taken on the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", "gemm_tc_mlp_bucket_24x1024x4096.md")
    try:
        text = open(path).read()
    except OSError:
        return None
    src = gemm_source_hash()
    for line in text.splitlines():
        if line.startswith("traffic_bytes_per_launch:"):
            parts = dict(kv.split("=") for kv in line.split(":", 1)[1].split())
            if parts.get("source_hash") == src:
                return float(parts["bytes"])
    return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,utilization.gpu,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 8:
                self.rows.append(parts)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            if self.thread:
                self.thread.join(timeout=2)

    def summary(self):
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        loaded, reasons, maxes = [], set(), []
        for r in self.rows:
            try:
                sm, smax, util = float(r[0]), float(r[1]), float(r[3])
            except ValueError:
                continue
            maxes.append(smax)
            if util > 0:
                loaded.append(sm)
                for nm, v in zip(names, r[4:]):
                    if v.lower().startswith("active"):
                        reasons.add(nm)
        if not maxes:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(maxes),
                "reasons": sorted(reasons), "samples": len(self.rows), "samples_under_load": len(loaded)}


def smi_id(torch, dev):
    try:
        p = torch.cuda.get_device_properties(dev)
        return f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v for v in vis.split(",") if v.strip()]
        return ids[dev] if dev < len(ids) else str(dev)


def cpu_baseline(bucket, budget_s=15.0):
    """The fp64 oracle (restarted Gram NS) on this host, on matrices of the same
    bucket until the budget is spent."""
    import numpy as np
    from oracle import gram_ns
    done, t0 = 0, time.perf_counter()
    while done < len(bucket):
        gram_ns.orthogonalize(bucket[done].astype(np.float64), T_STEPS, None, RESTART)
        done += 1
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "sample": f"{done} of the {len(bucket)} {R}x{C} matrices of the bucket, fp64 numpy, {dt:.1f} s"}


def cpu_threads():
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        v = os.environ.get(var)
        if v and v.isdigit():
            return int(v)
    return os.cpu_count()


def rank_seed(rank):
    """Seed of a rank's bucket: every rank orthogonalizes its own independent
    bucket (the matrices of a bucket are independent problems), so ranks
    share no data and exchange nothing but timings."""
    return 2000 + rank


def max_over_ranks(value, dist, device):
    """The job's time is its slowest rank's: max of a per-rank scalar over all
    ranks (identity without a process group)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, seconds):
    """Units processed by all ranks per second of the slowest rank."""
    return units_per_rank * world / seconds


def make_bucket(seed):
    from inputs import generators as gen
    return gen.gaussian_bucket(G, R, C, seed)


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step orthogonalizes one matrix of
    the bucket in fp64 on the host cores (rank 0 only)."""
    if rank != 0:
        return
    bucket = make_bucket(rank_seed(0))
    import numpy as np
    from oracle import gram_ns
    for i in range(args.warmup):
        gram_ns.orthogonalize(bucket[i % G].astype(np.float64), T_STEPS, None, RESTART)
    t0 = time.perf_counter()
    for i in range(args.steps):
        gram_ns.orthogonalize(bucket[i % G].astype(np.float64), T_STEPS, None, RESTART)
    dt = time.perf_counter() - t0
    value = args.steps / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(world),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
                             "sample": f"one {R}x{C} matrix of the bucket per step, fp64 numpy"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="gns", choices=["gns", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--G", type=int, default=24, help="matrices per bucket (24 is the benchmark; smaller only for profiling)")
    args = ap.parse_args()
    global G
    G = args.G
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        return run_reference(args, rank, world)

    import torch
    import newton_schulz_gram_gb300 as gns

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    gns.load()

    bucket = make_bucket(rank_seed(rank))
    host = torch.from_numpy(bucket).pin_memory()
    x = host.to(dev, non_blocking=False)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()

    sampler = ClockSampler(smi_id(torch, local))
    sampler.start()
    for _ in range(args.warmup):
        gns.gns_orthogonalize_batched(x, T_STEPS, RESTART)
    if gns.gns_get_status() != 0:
        raise SystemExit("device status error during warm-up")

    # Timed region: K steps, CUDA events on the launching stream.
    barrier()
    launches0 = gns.gns_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        gns.gns_orthogonalize_batched(x, T_STEPS, RESTART)
    e1.record(stream)
    barrier()
    launches = gns.gns_launch_count() - launches0
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)

    # Same K steps again with per-launch events, for the per-kernel roofline.
    gns.gns_profile_enable(True)
    for _ in range(args.steps):
        gns.gns_orthogonalize_batched(x, T_STEPS, RESTART)
    torch.cuda.synchronize(dev)
    gns.gns_profile_enable(False)
    prof = gns.gns_profile_read()
    sampler.stop()
    status = gns.gns_get_status()
    if status != 0:
        raise SystemExit(f"device status {status} after the timed region")

    # End to end through the host-buffer entry point.
    e2e_steps = max(1, args.e2e_steps)
    hbuf = host.clone().pin_memory()
    gns.gns_orthogonalize_batched_host(hbuf, T_STEPS, RESTART)
    if dist is not None:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        gns.gns_orthogonalize_batched_host(hbuf, T_STEPS, RESTART)
    e2e_s = max_over_ranks(time.perf_counter() - t0, dist, dev)

    peaks = load_peaks()
    value = job_throughput(G * args.steps, world, ms / 1e3)
    per_step_s = ms / 1e3 / args.steps
    alg = G * alg_flops_per_matrix(R, C)
    eff = G * eff_flops_per_matrix(R, C)
    gemm_n, gemm_ms = prof["gemm_tc"]
    gemm_launches_per_step = gemm_n / args.steps
    achieved = (alg * args.steps) / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else None
    traffic = profiled_traffic()
    kernels = {k: {"launches": n, "total_ms": round(t, 4), "share": round(t / max(1e-9, sum(v[1] for v in prof.values())), 4)}
               for k, (n, t) in prof.items() if n}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded N(0,1))", "config": config_dict(world),
        "algorithmic_tflops": alg * world / per_step_s / 1e12,
        "effective_tflops": eff * world / per_step_s / 1e12,
        "pct_fp16_peak_algorithmic": 100.0 * alg / per_step_s / 1e12 / peaks["tflops"],
        "pct_fp16_peak_effective": 100.0 * eff / per_step_s / 1e12 / peaks["tflops"],
        "roofline": {"kernel": "gemm_tc (tcgen05 grouped GEMM, all phases)", "bound": "tensor",
                     "achieved": achieved, "peak": peaks["tflops"], "unit": "TFLOP/s",
                     "frac": (achieved / peaks["tflops"]) if achieved else None,
                     "peak_source": f"{peaks['source']} dense bf16 burst (fp16 rate taken equal)",
                     "launches_per_step": gemm_launches_per_step,
                     "avg_launch_ms": gemm_ms / max(1, gemm_n),
                     "algorithmic_flops_per_launch": alg / max(1e-9, gemm_launches_per_step),
                     "traffic": traffic},
        "kernels": kernels,
        "gpu_launches": launches,
        "clocks": sampler.summary(),
        "e2e": {"value": job_throughput(G * e2e_steps, world, e2e_s), "unit": UNIT, "h2d_bytes_per_step": G * R * C * 4,
                "d2h_bytes_per_step": G * R * C * 4},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(bucket, args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
