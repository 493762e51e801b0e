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


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemm_tc_mlp_bucket_24x1024x4096.traffic.txt")


def profiled_traffic():
    """DRAM bytes per GEMM launch of the 24-matrix bucket from the committed
    summary that --record-traffic wrote from an ncu capture, if that capture
    was taken on the current kernel source (else None)."""
    try:
        text = open(TRAFFIC_FILE).read()
    except OSError:
        return None
    kv = dict(tok.split("=", 1) for tok in text.split() if "=" in tok)
    if kv.get("source_hash") != gemm_source_hash():
        return None
    return float(kv["bytes_per_launch"])


def record_traffic(csv_path, matrices):
    """Reads an `ncu --csv --page raw` capture of gemm_tc launches (metrics
    dram__bytes_read.sum and dram__bytes_write.sum, bytes) and writes the
    traffic summary the bench reads: the mean per launch, scaled from the
    captured bucket of `matrices` matrices to the benchmark's 24 (the
    per-matrix traffic does not depend on the bucket size)."""
    import csv
    with open(csv_path) as f:
        rows = [r for r in csv.reader(line for line in f if not line.startswith("=="))]
    hdr = rows[0]
    ki, ri, wi = hdr.index("Kernel Name"), hdr.index("dram__bytes_read.sum"), hdr.index("dram__bytes_write.sum")
    units = rows[1]
    scale = {"byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    vals = []
    for r in rows[2:]:
        if "gemm_tc" in r[ki]:
            vals.append(float(r[ri].replace(",", "")) * scale[units[ri]] + float(r[wi].replace(",", "")) * scale[units[wi]])
    if not vals:
        raise SystemExit("no gemm_tc launch in the capture")
    per = sum(vals) / len(vals) * 24.0 / matrices
    with open(TRAFFIC_FILE, "w") as f:
        f.write(f"kernel=gemm_tc source_hash={gemm_source_hash()} launches_captured={len(vals)} "
                f"matrices_captured={matrices} bytes_per_captured_launch={sum(vals) / len(vals):.0f} "
                f"bytes_per_launch={per:.0f}\n")
    print(open(TRAFFIC_FILE).read().strip())


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
                                          "--format=csv,noheader,nounits", "-lms", "50"],
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


SEED = 2000


def rank_chunk(rank, world):
    """(start, count) of this rank's matrices: the job orthogonalizes one
    bucket of G x world matrices, split into contiguous per-rank chunks
    (newton_schulz_gram_gb300.partition; the matrices are independent, so
    ranks share no data and exchange nothing but timings). G per rank is
    fixed: weak scaling."""
    from newton_schulz_gram_gb300.partition import partition
    return partition(G * world, world, rank)


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


def make_bucket(rank=0, world=1):
    from inputs import generators as gen
    start, count = rank_chunk(rank, world)
    return gen.gaussian_bucket(count, R, C, SEED, first=start)


def run_reference(args, rank, world):
    """The oracle as the reference arm: each step orthogonalizes one matrix of
    the bucket in fp64 on the host cores (rank 0 only)."""
    if rank != 0:
        return
    bucket = make_bucket()
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


def median(v):
    return statistics.median(v) if v else None


def quantiles(v):
    """(min, p25, median, p75, max) of a list of numbers."""
    s = sorted(v)
    if not s:
        return None
    q = statistics.quantiles(s, n=4, method="inclusive") if len(s) > 1 else [s[0]] * 3
    return [s[0], q[0], q[1], q[2], s[-1]]


def time_calls(torch, stream, fn, calls, warmup=2, blocks=5):
    """Median ms per call over `blocks` blocks of `calls` calls each (CUDA
    events on the launching stream, synchronized on both sides)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    per_call = []
    for _ in range(blocks):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(calls):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        per_call.append(a.elapsed_time(b) / calls)
    return median(per_call), quantiles(per_call)


def bucket_line(gns, torch, stream, dev, name, G_, R_, C_, calls, peak):
    """Throughput of one bucket shape (inputs N(0, 1) drawn on the device: the
    work does not depend on the values)."""
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    x = torch.randn(G_, R_, C_, device=dev, generator=gen)
    l0 = gns.gns_launch_count()
    gns.gns_orthogonalize_batched(x, T_STEPS, RESTART)
    torch.cuda.synchronize()
    launches = gns.gns_launch_count() - l0
    ms, q = time_calls(torch, stream, lambda: gns.gns_orthogonalize_batched(x, T_STEPS, RESTART), calls)
    if gns.gns_get_status() != 0:
        raise SystemExit(f"device status error in {name}")
    n, m = min(R_, C_), max(R_, C_)
    alg = G_ * alg_flops_per_matrix(n, m)
    tf = alg / (ms / 1e3) / 1e12
    del x
    return {"workload": name, "G": G_, "R": R_, "C": C_, "ms_per_call": ms, "ms_quartiles": q,
            "matrices_per_s": G_ / (ms / 1e3), "algorithmic_tflops": tf, "frac_of_peak": tf / peak,
            "effective_tflops": G_ * eff_flops_per_matrix(n, m) / (ms / 1e3) / 1e12,
            "launches_per_call": launches}


def llama7b_line(gns, torch, stream, dev, peaks):
    """One Muon step over the 7B Llama-like stack (Dion3 Fig. 1 workload;
    W bf16 N(0, 0.02), G bf16 N(0, 1e-3), M fp32, drawn on the device), and
    the standalone update kernel's HBM rate."""
    from inputs import generators as gen_mod
    shapes = gen_mod.llama7b_shapes()
    g = torch.Generator(device=dev)
    g.manual_seed(5000)
    W, Gr, M = [], [], []
    for _, r, c in shapes:
        W.append((0.02 * torch.randn(r, c, device=dev, generator=g)).to(torch.bfloat16))
        Gr.append((1e-3 * torch.randn(r, c, device=dev, generator=g)).to(torch.bfloat16))
        M.append(1e-3 * torch.randn(r, c, device=dev, generator=g))
    params = sum(w.numel() for w in W)
    alg = 0
    for _, r, c in shapes:
        n, m = min(r, c), max(r, c)
        alg += 4 * T_STEPS * n ** 3 if n == m else alg_flops_per_matrix(n, m)
    step = [2]

    def one():
        gns.muon_step(W, Gr, M, lr=0.02, wd=0.01, mu=0.95, seed=0, step=step[0])
        step[0] += 1

    one()
    torch.cuda.synchronize()
    gns.gns_profile_enable(True)
    gns.gns_profile_read()
    ms, q = time_calls(torch, stream, one, calls=1, warmup=0, blocks=3)
    gns.gns_profile_enable(False)
    prof = gns.gns_profile_read()
    if gns.gns_get_status() != 0:
        raise SystemExit("device status error in the 7B step")
    nc_n, nc_ms = prof["norm_cast"]
    # Momentum + norm + cast over the 3 timed steps: M read and written (8 B),
    # G read (2 B), fp16 X written (2 B) per parameter.
    nc_step_ms = nc_ms / 3
    nc_gbs = 12.0 * params / (nc_step_ms / 1e3) / 1e9 if nc_ms > 0 else None
    del W, Gr, M
    torch.cuda.empty_cache()
    upd = update_rate(gns, torch, stream, dev, 30, peaks)
    return {"workload": "llama7b_muon_step (224 matrices, 6.98e9 params, buckets by shape)",
            "ms_per_step": ms, "ms_quartiles": q, "params": params, "algorithmic_tflops": alg / (ms / 1e3) / 1e12,
            "frac_of_peak": alg / (ms / 1e3) / 1e12 / peaks["tflops_sustained"],
            "peak_used": "sustained bf16 (a step of about 0.3 s)",
            "elementwise": {
                "norm_cast_momentum": {"ms_per_step": nc_step_ms, "launches_per_step": nc_n / 3, "gbs": nc_gbs,
                                       "bytes_per_element": 12, "frac_of_hbm": (nc_gbs / peaks["hbm_gbs"]) if nc_gbs else None},
                "muon_update_kernel": upd}}


def muon_bucket_line(gns, torch, stream, dev, G_, blocks):
    """muon_step over G_ parameters of R x C (the benchmark's matrix shape):
    bf16 W ~ N(0, 0.02), bf16 G ~ N(0, 1e-3), fp32 M, drawn on the device.
    One call is the momentum + norm + cast pass and the GEMM program with the
    update fused into its last product's epilogue."""
    g = torch.Generator(device=dev)
    g.manual_seed(5000)
    W = [(0.02 * torch.randn(R, C, device=dev, generator=g)).to(torch.bfloat16) for _ in range(G_)]
    Gr = [(1e-3 * torch.randn(R, C, device=dev, generator=g)).to(torch.bfloat16) for _ in range(G_)]
    M = [1e-3 * torch.randn(R, C, device=dev, generator=g) for _ in range(G_)]
    step = [2]

    def one():
        gns.muon_step(W, Gr, M, lr=0.02, wd=0.01, mu=0.95, seed=0, step=step[0])
        step[0] += 1

    one()
    torch.cuda.synchronize()
    gns.gns_profile_enable(True)
    gns.gns_profile_read()
    ms, q = time_calls(torch, stream, one, calls=1, warmup=2, blocks=blocks)
    gns.gns_profile_enable(False)
    prof = gns.gns_profile_read()
    if gns.gns_get_status() != 0:
        raise SystemExit("device status error in muon_step")
    calls = blocks + 2
    return {"workload": f"muon_step over {G_} x {R}x{C}", "ms_per_step": ms, "ms_quartiles": q,
            "kernels_ms_per_step": {k: t / calls for k, (n, t) in prof.items() if n}}


def update_rate(gns, torch, stream, dev, log2n, peaks, blocks=10):
    """The standalone update kernel (W <- SR_bf16(decay W - step O)) over
    2^log2n elements of a square matrix: W read and written, O read, 6 B per
    element; O ~ N(0, 1) in fp16 so every element takes the rounding path."""
    N = 1 << log2n
    side = 1 << (log2n // 2)
    w = (0.02 * torch.randn(side, N // side, device=dev)).to(torch.bfloat16)
    o = torch.randn(side, N // side, device=dev).to(torch.float16)
    ums, uq = time_calls(torch, stream, lambda: gns.gns_muon_update(w, o, 0.02, 0.01, 1.0, 0, 1), calls=1,
                         warmup=2, blocks=blocks)
    if gns.gns_get_status() != 0:
        raise SystemExit("device status error in the update kernel")
    del w, o
    torch.cuda.empty_cache()
    gbs = 6.0 * N / (ums / 1e3) / 1e9
    return {"elements": N, "ms": ums, "ms_quartiles": uq, "gbs": gbs, "bytes_per_element": 6,
            "frac_of_hbm": gbs / peaks["hbm_gbs"]}


def single_thread_oracle(budget_s=10.0):
    """The oracle on one host thread (BLAS threads pinned to 1 in a child
    process), over matrices of the benchmark bucket until the budget is spent."""
    code = ("import sys, time, numpy as np; sys.path.insert(0, %r); from inputs import generators as gen; "
            "from oracle import gram_ns; X = gen.gaussian_bucket(3, %d, %d, %d); t0 = time.perf_counter(); n = 0\n"
            "while n < 3:\n"
            "    gram_ns.orthogonalize(X[n].astype(np.float64), %d, None, %d); n += 1\n"
            "    if time.perf_counter() - t0 > %f: break\n"
            "print(n, time.perf_counter() - t0)") % (ROOT, R, C, SEED, T_STEPS, RESTART, budget_s)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                           timeout=budget_s * 6 + 60)
        n, dt = r.stdout.split()[-2:]
        n, dt = int(n), float(dt)
    except Exception as e:  # reported, not fatal
        return {"error": str(e)[:200]}
    return {"value": n / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} {R}x{C} matrices of the bucket, fp64 numpy, one thread, {dt:.1f} s"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gns", choices=["gns", "reference"])
    ap.add_argument("--min-timed-s", type=float, default=1.5,
                    help="repeat the timed block of K steps (at least 5 times) until this much time is timed")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads' table")
    ap.add_argument("--G", type=int, default=24, help="matrices per bucket (24 is the benchmark; smaller only for profiling)")
    ap.add_argument("--record-traffic", metavar="CSV",
                    help="write the GEMM traffic summary from an ncu --csv --page raw capture and exit")
    ap.add_argument("--traffic-matrices", type=int, default=12, help="matrices in the captured launch")
    ap.add_argument("--only-update", type=int, metavar="LOG2N",
                    help="time only the standalone Muon update kernel on 2^LOG2N elements, print its rate and exit")
    ap.add_argument("--only-muon", type=int, metavar="G",
                    help="time only muon_step over G parameters of 1024 x 4096 (update fused into the GEMM "
                         "program's epilogue), print the step time and exit")
    args = ap.parse_args()
    if args.record_traffic:
        return record_traffic(args.record_traffic, args.traffic_matrices)
    if args.only_muon:
        import torch
        import newton_schulz_gram_gb300 as gns
        gns.load()
        dev = torch.device("cuda", 0)
        print(json.dumps(muon_bucket_line(gns, torch, torch.cuda.current_stream(dev), dev, args.only_muon,
                                          max(3, args.steps // 4))))
        return
    if args.only_update:
        import torch
        import newton_schulz_gram_gb300 as gns
        gns.load()
        dev = torch.device("cuda", 0)
        r = update_rate(gns, torch, torch.cuda.current_stream(dev), dev, args.only_update, load_peaks(),
                        blocks=max(3, args.steps // 4))
        print(json.dumps({"kernel": "muon_update_kernel", **r}))
        return
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

    bucket = make_bucket(rank, world)
    host = torch.from_numpy(bucket).pin_memory()
    x = host.to(dev, non_blocking=False)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        torch.cuda.synchronize(dev)
        if dist is not None:
            dist.barrier()

    for _ in range(args.warmup):
        gns.gns_orthogonalize_batched(x, T_STEPS, RESTART)
    if gns.gns_get_status() != 0:
        raise SystemExit("device status error during warm-up")

    # Timed region: blocks of exactly K steps, each bracketed by a barrier and
    # a synchronization and timed with CUDA events on the launching stream;
    # at least 5 blocks, more until --min-timed-s is covered. The clocks are
    # sampled throughout.
    sampler = ClockSampler(smi_id(torch, local))
    sampler.start()
    time.sleep(0.3)
    block_ms, launches = [], 0
    while len(block_ms) < 5 or (sum(block_ms) < 1e3 * args.min_timed_s and len(block_ms) < 500):
        barrier()
        l0 = gns.gns_launch_count()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            gns.gns_orthogonalize_batched(x, T_STEPS, RESTART)
        e1.record(stream)
        barrier()
        launches = gns.gns_launch_count() - l0
        block_ms.append(max_over_ranks(e0.elapsed_time(e1), dist, dev))
    sampler.stop()
    status = gns.gns_get_status()
    if status != 0:
        raise SystemExit(f"device status {status} after the timed region")
    ms = median(block_ms)
    step_q = [b / args.steps for b in quantiles(block_ms)]

    # One more block with per-launch events, for the per-kernel roofline.
    gns.gns_profile_enable(True)
    gns.gns_profile_read()
    for _ in range(args.steps):
        gns.gns_orthogonalize_batched(x, T_STEPS, RESTART)
    torch.cuda.synchronize(dev)
    gns.gns_profile_enable(False)
    prof = gns.gns_profile_read()

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
    per_step_s = ms / 1e3 / args.steps
    value = job_throughput(G, world, per_step_s)
    alg = G * alg_flops_per_matrix(R, C)
    eff = G * eff_flops_per_matrix(R, C)
    gemm_n, gemm_ms = prof["gemm_tc"]
    achieved = (alg * args.steps) / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else None
    total_prof = max(1e-9, sum(v[1] for v in prof.values()))
    kernels = {k: {"launches": n, "total_ms": round(t, 4), "share": round(t / total_prof, 4)}
               for k, (n, t) in prof.items() if n}
    clocks = sampler.summary()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": per_step_s * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic (seeded N(0,1))", "config": config_dict(world),
        "timed_blocks": len(block_ms),
        "ms_per_step_quartiles": step_q,
        "algorithmic_tflops": alg * world / per_step_s / 1e12,
        "effective_tflops": eff * world / per_step_s / 1e12,
        "pct_fp16_peak_algorithmic": 100.0 * alg / per_step_s / 1e12 / peaks["tflops"],
        "pct_fp16_peak_effective": 100.0 * eff / per_step_s / 1e12 / peaks["tflops"],
        # The GEMM program is timed inside seconds of back-to-back calls under
        # the power cap, the condition of the sustained peak (a seconds-long
        # loop of bf16 matmuls); the burst-peak fraction is reported beside it.
        "roofline": {"kernel": "gemm_tc (tcgen05 grouped GEMM, all phases)", "bound": "tensor",
                     "achieved": achieved, "peak": peaks["tflops_sustained"], "unit": "TFLOP/s",
                     "frac": (achieved / peaks["tflops_sustained"]) if achieved else None,
                     "peak_source": f"{peaks['source']} dense bf16 sustained (seconds of back-to-back matmuls "
                                    f"under the power cap; fp16 rate taken equal)",
                     "peak_burst": peaks["tflops"],
                     "frac_of_burst": (achieved / peaks["tflops"]) if achieved else None,
                     "launches_per_step": gemm_n / args.steps,
                     "avg_launch_ms": gemm_ms / max(1, gemm_n),
                     "algorithmic_flops_per_launch": alg / max(1e-9, gemm_n / args.steps),
                     "traffic": profiled_traffic()},
        "kernels": kernels,
        "gpu_launches": launches,
        "clocks": clocks,
        "e2e": {"value": job_throughput(G * e2e_steps, world, e2e_s), "unit": UNIT, "h2d_bytes_per_step": G * R * C * 4,
                "d2h_bytes_per_step": G * R * C * 4},
    }
    if clocks.get("sm_mhz"):
        line["ms_x_sm_mhz"] = per_step_s * 1e3 * clocks["sm_mhz"]
    if rank == 0 and world == 1 and not args.no_configs:
        del x
        torch.cuda.empty_cache()
        line["configs"] = {
            "single_128x512": bucket_line(gns, torch, stream, dev, "single_128x512", 1, 128, 512, 200, peaks["tflops"]),
            "square_16x2048": bucket_line(gns, torch, stream, dev, "square_16x2048 (standard NS)", 16, 2048, 2048, 5,
                                          peaks["tflops"]),
            "moe_256x512x2048": bucket_line(gns, torch, stream, dev, "moe_256x512x2048", 256, 512, 2048, 5,
                                            peaks["tflops"]),
            "per_head_16x256x4096": bucket_line(gns, torch, stream, dev, "per_head_16x256x4096", 16, 256, 4096, 20,
                                                peaks["tflops"]),
            "llama7b_muon_step": llama7b_line(gns, torch, stream, dev, peaks),
        }
        line["configs"]["single_128x512"]["us_per_call"] = line["configs"]["single_128x512"]["ms_per_call"] * 1e3
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(bucket, args.cpu_budget)
        line["cpu_baseline_single_thread"] = single_thread_oracle()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
