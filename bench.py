"""Benchmark of the routed FP8 MoE decode layer (DeepSeek-V3 shape) on GB300.

One step = one routed-FP8 layer call at each of M = 1, 2, 4, 8 decode tokens
(hidden 7168, inter 2048, 256 experts, top_k 8, BF16 logits), every call with
fresh router logits so the touched expert set changes as in real decode. The
metric is the weight-stream bandwidth: the bytes of every unique expert the
calls touched (W13 + W2 + FP32 block scales, counted from the kernel's own
ids) over the device time. All weights (11.3 GB) are resident in HBM; each
call reads >= 352 MB of them, well above the 129 MB L2, so no flush is needed.

Launch: python bench.py [--gpus N --steps K --warmup W] (N > 1 under
torch.distributed.run: one independent replica per GPU, no collective on the
data path; the value is the sum over ranks of bytes over the max time).
--impl reference times the CPU oracle instead (host cores, bounded sample).
Prints one JSON line on rank 0.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MS = (1, 2, 4, 8)
EXPERT_BYTES = 4096 * 7168 + 7168 * 2048 + 4 * (32 * 56 + 56 * 16)  # 44,050,944
METRIC = "routed-MoE layer weight-stream HBM GB/s at M=1-8 tokens (DSv3-shaped routed FP8)"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="fme", choices=["fme", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-extras", action="store_true", help="skip the shared-expert / NVFP4 side measurements")
    ap.add_argument("--ref-seconds", type=float, default=10.0)
    ap.add_argument("--experts", type=int, default=256,
                    help="experts resident on the device (smaller for profiler captures; 32 x 44 MB = 1.4 GB)")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle leg")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end leg")
    ap.add_argument("--no-flushed", action="store_true", help="skip the L2-flushed per-M calls")
    ap.add_argument("--mx-launches", action="store_true",
                    help="only BF16- and MXFP8-token routed FP8 calls at M = 1, 2, 4, 8 (profiling)")
    ap.add_argument("--shared-launches", action="store_true",
                    help="only launch the FP8 shared expert alone twice at each of M = 1, 8 (for profiles)")
    ap.add_argument("--nvfp4-launches", action="store_true",
                    help="only launch the NVFP4 slot MoE twice at each of M = 1, 8, 64 (for profiler launch lists)")
    return ap.parse_args()


# --------------------------------------------------------------------------- CPU oracle leg
def oracle_prepare(seed=0):
    """Inputs of the CPU oracle sample: one DSv3 token's first route, its expert's
    bytes materialised (before any clock starts)."""
    from oracle import routing
    from synth import workloads as W

    cfg = W.DSV3
    w13h, w2h = W.fp8_weights_host(cfg, seed)
    s13, s2 = W.fp8_weight_scales(cfg, seed)
    # One token's first route, repeated: the oracle's work per route does not depend on
    # which expert it is, and generating a new 44 MB expert per route would dominate the
    # wall time of the sample.
    x, logits, bias = W.fp8_activations(cfg, 1, seed, 0)
    ids, _, _ = routing.route(logits, bias, cfg.top_k, cfg.scale)
    e = int(ids[0, 0])
    w13h[e], w2h[e]  # materialise this expert's bytes outside the timed region
    return cfg, (x, logits, bias, w13h, s13, w2h, s2)


def oracle_run(prep, seconds, max_routes=64):
    """Time whole DSv3 routes of the CPU oracle (one expert's GEMM1 + SwiGLU +
    GEMM2 for one token) until `seconds` of work or `max_routes` routes.
    Returns (GB/s of weight stream, routes, seconds)."""
    from oracle import moe_fp8

    cfg, (x, logits, bias, w13h, s13, w2h, s2) = prep
    done, t_total = 0, 0.0
    while t_total < seconds and done < max_routes:
        t0 = time.perf_counter()
        moe_fp8.routed_fp8(x, logits, bias, w13h, s13, w2h, s2, cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0,
                           routes=[0])
        t_total += time.perf_counter() - t0
        done += 1
    return done * EXPERT_BYTES / t_total / 1e9, done, t_total


def oracle_sample(seconds, seed=0):
    """oracle_prepare then oracle_run: (GB/s, routes, seconds)."""
    return oracle_run(oracle_prepare(seed), seconds)


_ONE_THREAD = dict(OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")


def run_oracle_subprocess(seconds):
    """Run the oracle sample in a child pinned to one thread; returns its dict."""
    env = dict(os.environ, **_ONE_THREAD)
    code = ("import json,sys; sys.path.insert(0, %r); import bench; g,n,t=bench.oracle_sample(%f); "
            "print(json.dumps({'gbs': g, 'routes': n, 'seconds': t}))" % (ROOT, seconds))
    out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, check=True)
    return json.loads(out.stdout.strip().splitlines()[-1])


def host_cores(cap=32):
    """Cores this process may run on (at most `cap`: each oracle process holds
    one expert, about 0.1 GB, in memory)."""
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        n = os.cpu_count() or 1
    return max(1, min(n, cap))


def run_oracle_parallel(seconds, workers, steps=1):
    """`workers` one-thread children time the oracle sample over common
    windows: each prepares its inputs once and reports ready; every step starts
    on a shared go. Returns one dict per step: {'gbs': routes of all children x
    expert bytes / the longest child's wall time, 'routes', 'seconds', 'workers'}."""
    env = dict(os.environ, **_ONE_THREAD)
    code = ("import json,sys,time; sys.path.insert(0, %r); import bench; p=bench.oracle_prepare(); "
            "print('ready', flush=True)\n"
            "for _ in range(%d):\n"
            "    sys.stdin.readline(); w0=time.perf_counter(); g,n,t=bench.oracle_run(p, %f)\n"
            "    print(json.dumps({'routes': n, 'seconds': t, 'wall': time.perf_counter()-w0}), flush=True)\n"
            % (ROOT, steps, seconds))
    procs = [subprocess.Popen([sys.executable, "-c", code], env=env, stdin=subprocess.PIPE,
                              stdout=subprocess.PIPE, text=True) for _ in range(workers)]
    out = []
    try:
        for p in procs:
            if p.stdout.readline().strip() != "ready":
                raise RuntimeError("oracle child failed before its sample")
        for _ in range(steps):
            for p in procs:
                p.stdin.write("go\n")
                p.stdin.flush()
            res = [json.loads(p.stdout.readline()) for p in procs]
            routes = sum(r["routes"] for r in res)
            wall = max(r["wall"] for r in res)
            out.append({"gbs": routes * EXPERT_BYTES / wall / 1e9, "routes": routes, "seconds": wall,
                        "workers": workers})
    finally:
        for p in procs:
            if p.stdin:
                p.stdin.close()
            p.wait()
    return out


def reference_arm(args, rank):
    if rank != 0:
        return
    steps = max(1, min(args.steps, 6))
    per = max(2.0, args.ref_seconds / steps)
    workers = host_cores()
    t0 = time.time()
    vals = run_oracle_parallel(per, workers, steps)
    gbs = sum(v["routes"] for v in vals) * EXPERT_BYTES / sum(v["seconds"] for v in vals) / 1e9
    ms_per_route = 1e3 * sum(v["seconds"] for v in vals) / sum(v["routes"] for v in vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
        "steps": steps, "warmup": 0, "ms_per_step": round(ms_per_route, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "dsv3_routed_fp8 (H 7168, I 2048, E 256, top_k 8)", "sample": "one route per "
                   "oracle call (one expert: 44,050,944 weight+scale bytes), one process per host core, "
                   "ms_per_step = wall ms per route, all processes together", "parallelism": "replicas"},
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": workers, "kind": "oracle",
                         "sample": f"{sum(v['routes'] for v in vals)} DSv3 routes over {workers} one-thread "
                                   f"processes, {time.time() - t0:.1f} s wall"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- replicas
def aggregate(total_bytes, elapsed_ms, dist=None, device="cpu"):
    """Whole-job weight-stream GB/s of N independent replicas: the bytes every
    rank streamed, summed, over the slowest rank's time (the only collective
    is this end-of-run reduction of two scalars)."""
    import torch

    if dist is not None and dist.is_initialized() and dist.get_world_size() > 1:
        t = torch.tensor([float(elapsed_ms)], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        b = torch.tensor([float(total_bytes)], dtype=torch.float64, device=device)
        dist.all_reduce(b)
        elapsed_ms, total_bytes = float(t.item()), float(b.item())
    return total_bytes, elapsed_ms, total_bytes / (elapsed_ms * 1e-3) / 1e9


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"fme_clocks_rank{index}_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            self.proc.wait(timeout=10)
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------- GPU arm
def gpu_arm(args, rank, world, local_rank):
    import torch

    import fp4_moe_expert_gb300 as fme
    from synth import workloads as W

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    import dataclasses
    cfg = dataclasses.replace(W.DSV3, E=args.experts)
    w13, s13, w2, s2 = W.fp8_weights_device(cfg, args.seed, dev)
    n_calls = (args.warmup + args.steps) * len(MS)
    pool = 64
    # Fresh logits for every call (a pool of distinct draws, cycled), fixed x per M.
    logits_pool = [torch.from_numpy(W.fp8_activations(cfg, 8, args.seed + 1000 * rank, step)[1]).to(dev)
                   .to(torch.bfloat16) for step in range(pool)]
    xs = {M: torch.from_numpy(W.fp8_activations(cfg, M, args.seed + 1000 * rank, 0)[0]).to(dev)
          .to(torch.bfloat16) for M in MS}
    bias = torch.from_numpy(W.fp8_activations(cfg, 1, args.seed, 0)[2]).to(dev)
    outs = {M: (torch.empty(M * cfg.top_k, cfg.H, dtype=torch.bfloat16, device=dev),
                torch.empty(M, cfg.top_k, dtype=torch.int32, device=dev),
                torch.empty(M, cfg.top_k, dtype=torch.float32, device=dev)) for M in MS}
    ws = fme.Workspace(fme.moe_routed_fp8_workspace(8, cfg.H, cfg.I, cfg.E, cfg.top_k), dev)
    # One ids buffer per timed call, so reading them back needs no copy inside the region.
    ids_log = torch.full((args.steps * len(MS), 8 * cfg.top_k), -1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps * len(MS))]

    def call(M, k, record=None):
        lg = logits_pool[k % pool][:M]
        out, ids, wts = outs[M]
        if record is not None:
            ids = ids_log[record, :M * cfg.top_k].view(M, cfg.top_k)
            ev[record][0].record(stream)
        fme.moe_routed_fp8(xs[M], lg, bias, w13, s13, w2, s2, cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0,
                           out=out, ids=ids, weights=wts, workspace=ws)
        if record is not None:
            ev[record][1].record(stream)

    k = 0
    for _ in range(args.warmup):
        for M in MS:
            call(M, k)
            k += 1
    torch.cuda.synchronize()
    code = ws.error()
    if code:
        raise SystemExit(f"device error word 0x{code:x} during warm-up: refusing to time a failing kernel")
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local_rank) as clocks:
        t_start.record(stream)
        rec = 0
        for _ in range(args.steps):
            for M in MS:
                call(M, k, rec)
                k += 1
                rec += 1
        t_end.record(stream)
        torch.cuda.synchronize()
    if dist:
        dist.barrier()
    elapsed_ms = t_start.elapsed_time(t_end)
    code = ws.error()
    if code:
        raise SystemExit(f"device error word 0x{code:x} in the timed region")
    launch_ms = np.array([a.elapsed_time(b) for a, b in ev])
    ids_np = ids_log.cpu().numpy()
    uniq = np.array([len(set(r[r >= 0].tolist())) for r in ids_np])
    bytes_call = uniq * EXPERT_BYTES
    total_bytes = float(bytes_call.sum())
    total_bytes, elapsed_ms, value = aggregate(total_bytes, elapsed_ms, dist, dev)
    per_m = {}
    for i, M in enumerate(MS):
        sel = slice(i, None, len(MS))
        t_us = launch_ms[sel] * 1e3
        per_m[str(M)] = {"us_median": round(float(np.median(t_us)), 2), "us_p10": round(float(np.percentile(t_us, 10)), 2),
                         "us_p90": round(float(np.percentile(t_us, 90)), 2),
                         "unique_experts_mean": round(float(uniq[sel].mean()), 2),
                         "GBps_median": round(float(np.median(bytes_call[sel] / (launch_ms[sel] * 1e-3) / 1e9)), 1)}
    peak, peak_kind = peaks()
    achieved = float(bytes_call.sum() / (launch_ms.sum() * 1e-3) / 1e9)
    for M in MS:
        per_m[str(M)]["pct_of_peak_median"] = round(100.0 * per_m[str(M)]["GBps_median"] / peak, 1)
    if not args.no_flushed:
        flushed_per_m(fme, torch, cfg, xs, logits_pool, bias, w13, s13, w2, s2, outs, ws, dev, per_m, peak)
    traffic = load_traffic()

    e2e = None if args.no_e2e else e2e_leg(fme, cfg, w13, s13, w2, s2, bias, dev, args)
    extras = {} if args.no_extras else side_measurements(fme, dev, args)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        try:
            workers = host_cores()
            r = run_oracle_parallel(args.ref_seconds, workers)[0]
            r1 = run_oracle_subprocess(args.ref_seconds)
            cpu = {"value": round(r["gbs"], 4), "unit": "GB/s", "cores": workers, "kind": "oracle",
                   "sample": f"{r['routes']} DSv3 routes (one expert each, 44.05 MB) over {workers} one-thread "
                             f"processes, {r['seconds']:.1f} s wall",
                   "single_core": {"value": round(r1["gbs"], 4), "unit": "GB/s",
                                   "sample": f"{r1['routes']} routes, {r1['seconds']:.1f} s"}}
        except Exception as exc:  # pragma: no cover - reported, not fatal
            cpu = {"value": None, "unit": "GB/s", "cores": None, "kind": "oracle", "sample": f"failed: {exc}"}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8-e4m3 x fp8-e4m3 -> f32", "data": "synthetic",
        "config": {"workload": "dsv3_routed_fp8: H 7168, I 2048, E 256, top_k 8, M in {1,2,4,8} per step, "
                   "BF16 logits, non-pow2 FP32 block scales", "global_batch": sum(MS) * world, "seq_len": 1,
                   "parallelism": "replicas" if world > 1 else "single-gpu",
                   "l2": "timed region: no flush, each call streams >= 352 MB of weights (> 129 MB L2) with "
                         "fresh routing; per_m also gives 50 calls per M with L2 flushed (512 MB read) before each",
                   "per_m": per_m, "unique_experts_per_step": round(float(uniq.sum() / args.steps), 2)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic, "peak_kind": peak_kind,
                     "kernel": "fp8_moe_tc_kernel", "bytes_per_launch": "unique experts x 44,050,944 B"},
        "clocks": clocks.summary(),
        "e2e": e2e,
        "gpu_launches": args.steps * len(MS),
        "cpu_baseline": cpu,
    }
    if extras:
        line["also"] = extras
    print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def flushed_per_m(fme, torch, cfg, xs, logits_pool, bias, w13, s13, w2, s2, outs, ws, dev, per_m, peak, calls=50):
    """Per M, `calls` more calls with L2 flushed before each (a 512 MB read,
    outside the events) and fresh logits each time: median microseconds and
    GB/s of the unique experts each call touched, beside the back-to-back
    figures of the timed region."""
    flush = torch.ones(128 * 1024 * 1024, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)
    for M in MS:
        out, ids, wts = outs[M]
        us, gbs = [], []
        for i in range(calls + 3):
            flush.amax()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fme.moe_routed_fp8(xs[M], logits_pool[(7 * i + M) % len(logits_pool)][:M], bias, w13, s13, w2, s2,
                               cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0, out=out, ids=ids, weights=wts,
                               workspace=ws)
            b.record(stream)
            torch.cuda.synchronize()
            if i >= 3:
                t = a.elapsed_time(b) * 1e3
                u = len(set(ids.reshape(-1).tolist()))
                us.append(t)
                gbs.append(u * EXPERT_BYTES / (t * 1e-6) / 1e9)
        if ws.error():
            raise SystemExit("device error word set in the flushed per-M calls")
        d = per_m[str(M)]
        d["us_median_l2_flushed"] = round(float(np.median(us)), 2)
        d["GBps_median_l2_flushed"] = round(float(np.median(gbs)), 1)
        d["pct_of_peak_median_l2_flushed"] = round(100.0 * float(np.median(gbs)) / peak, 1)
    del flush


def kernel_code_sha256(path):
    """sha256 of a CUDA source without its whole-line comments and blank lines:
    changes to the code change it, comment-only edits do not."""
    import hashlib
    with open(path) as f:
        lines = [ln.rstrip() for ln in f]
    code = [ln for ln in lines if ln.strip() and not ln.strip().startswith("//")]
    return hashlib.sha256("\n".join(code).encode()).hexdigest()


def load_traffic():
    """Mean DRAM bytes (read + write) per launch of the dominant kernel from the
    committed ncu launch list (profiles/traffic.json); None when the kernel
    code has changed since those counters were taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    src = os.path.join(ROOT, "fp4_moe_expert_gb300", "csrc", "fme_routed_fp8.cu")
    try:
        with open(path) as f:
            d = json.load(f)
        if kernel_code_sha256(src) != d.get("kernel_code_sha256"):
            return None
        return d.get("fp8_moe_kernel_dsv3_bytes_per_launch")
    except Exception:
        return None


def e2e_leg(fme, cfg, w13, s13, w2, s2, bias, dev, args):
    """Same metric through the public API with host buffers: per call, pinned
    x and logits go host->device, results come back device->host."""
    import torch
    from synth import workloads as W

    steps = max(5, min(50, args.steps))
    host = {}
    for M in MS:
        x, logits, _ = W.fp8_activations(cfg, M, args.seed + 7, M)
        host[M] = (torch.from_numpy(x).to(torch.bfloat16).pin_memory(),
                   torch.from_numpy(logits).to(torch.bfloat16).pin_memory(),
                   torch.empty(M * cfg.top_k, cfg.H, dtype=torch.bfloat16).pin_memory(),
                   torch.empty(M, cfg.top_k, dtype=torch.int32).pin_memory(),
                   torch.empty(M, cfg.top_k, dtype=torch.float32).pin_memory())
    stream = torch.cuda.current_stream(dev)
    uniq_total = 0

    def one(M):
        xh, lh, oh, ih, wh = host[M]
        xd = xh.to(dev, non_blocking=True)
        ld = lh.to(dev, non_blocking=True)
        out, ids, wts = fme.moe_routed_fp8(xd, ld, bias, w13, s13, w2, s2, cfg.top_k, cfg.limit, cfg.scale,
                                           cfg.ue8m0)
        oh.copy_(out, non_blocking=True)
        ih.copy_(ids, non_blocking=True)
        wh.copy_(wts, non_blocking=True)

    for M in MS:
        one(M)
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        for M in MS:
            one(M)
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b)
    for M in MS:
        uniq_total += len(set(host[M][3].numpy().reshape(-1).tolist()))
    h2d = sum(host[M][0].numel() * 2 + host[M][1].numel() * 2 for M in MS)
    d2h = sum(host[M][2].numel() * 2 + host[M][3].numel() * 4 + host[M][4].numel() * 4 for M in MS)
    gbs = steps * uniq_total * EXPERT_BYTES / (ms * 1e-3) / 1e9
    return {"value": round(gbs, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(ms / steps, 4)}


def _event_us(fn, flush, reps=25, skip=5):
    """Median device time of fn() in microseconds, L2 flushed before each call."""
    import torch
    ts = []
    for i in range(reps):
        flush.amax()  # reads 512 MB: L2 holds none of the weights, and no dirty lines
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        if i >= skip:
            ts.append(a.elapsed_time(b) * 1e3)
    return float(np.median(ts))


def layer_measurements(fme, dev, args, shared_w, shared_bytes, flush):
    """DSv3 ue8m0 routed experts plus the shared expert, M = 1, 2, 4, 8: the
    shared-expert call then the routed call on one stream, against the
    one-launch layer (fme_moe_layer_fp8). Bytes = unique routed experts x
    expert bytes + the shared expert's bytes."""
    import torch
    from synth import workloads as W

    import dataclasses
    cfg = dataclasses.replace(W.DSV3_UE8M0, E=args.experts)
    w13, s13, w2, s2 = W.fp8_weights_device(cfg, args.seed, dev)
    sw13, ss13, sw2, ss2 = shared_w
    res = {}
    for M in MS:
        x, logits, bias = W.fp8_activations(cfg, M, args.seed, 7)
        xd = torch.from_numpy(x).to(dev).to(torch.bfloat16)
        ld = torch.from_numpy(logits).to(dev).to(torch.bfloat16)
        bd = torch.from_numpy(bias).to(dev)
        routed = (xd, ld, bd, w13, s13, w2, s2, cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0)
        shared = (sw13, ss13, sw2, ss2, W.SHARED.limit, W.SHARED.ue8m0)
        ws_r = fme.Workspace(fme.moe_routed_fp8_workspace(M, cfg.H, cfg.I, cfg.E, cfg.top_k), dev)
        ws_s = fme.Workspace(fme.shared_expert_fp8_workspace(M, cfg.H, cfg.I), dev)
        ws_l = fme.Workspace(fme.moe_layer_fp8_workspace(M, cfg.H, cfg.I, cfg.E, cfg.top_k), dev)
        outs = {}

        def separate():
            outs["s"] = fme.shared_expert_fp8(xd, *shared, workspace=ws_s)
            outs["r"] = fme.moe_routed_fp8(*routed, workspace=ws_r)

        def fused():
            outs["l"] = fme.moe_layer_fp8(*routed, *shared, workspace=ws_l)

        us_sep = _event_us(separate, flush)
        us_fused = _event_us(fused, flush)
        us_shared = _event_us(lambda: fme.shared_expert_fp8(xd, *shared, workspace=ws_s), flush)
        # routed experts alone, BF16 tokens against MXFP8 tokens (E4M3 + per-32 E8M0)
        xq, xsc = fme.mxfp8_quantize(xd)
        us_routed = _event_us(lambda: fme.moe_routed_fp8(*routed, workspace=ws_r), flush)
        us_mx = _event_us(lambda: fme.moe_routed_fp8_mx(xq, xsc, *routed[1:], workspace=ws_r), flush)
        # local finalize of the layer's outputs: y = bf16(sum_r w * out + shared_out)
        lo, _, lw, lso = outs["l"]
        ybuf = torch.empty(M, cfg.H, dtype=torch.bfloat16, device=dev)
        us_fin = _event_us(lambda: fme.moe_finalize(lo, lw, lso, y=ybuf), flush)
        us_layer_y = _event_us(lambda: fme.moe_finalize(*(lambda r: (r[0], r[2], r[3]))(
            fme.moe_layer_fp8(*routed, *shared, workspace=ws_l)), y=ybuf), flush)
        fin_bytes = (M * cfg.top_k * cfg.H + 2 * M * cfg.H) * 2 + M * cfg.top_k * 4
        for w in (ws_r, ws_s, ws_l):
            if w.error() != 0:
                raise RuntimeError("device wait timed out in the layer measurement")
        if not torch.equal(outs["l"][1], outs["r"][1]):
            raise RuntimeError("one-launch layer routed differently from the separate call")
        uniq = len(set(outs["l"][1].reshape(-1).tolist()))
        nbytes = uniq * EXPERT_BYTES + shared_bytes
        res[f"dsv3_ue8m0_plus_shared_M{M}"] = {
            "unique_experts": uniq,
            "shared_only_us": round(us_shared, 2),
            "shared_then_routed_us": round(us_sep, 2),
            "one_launch_layer_us": round(us_fused, 2),
            "one_launch_layer_GBps": round(nbytes / (us_fused * 1e-6) / 1e9, 1),
            "shared_then_routed_GBps": round(nbytes / (us_sep * 1e-6) / 1e9, 1),
            "routed_bf16_input_us": round(us_routed, 2),
            "routed_mxfp8_input_us": round(us_mx, 2),
            "routed_mxfp8_input_GBps": round(uniq * EXPERT_BYTES / (us_mx * 1e-6) / 1e9, 1),
            "finalize_us": round(us_fin, 2),
            "finalize_GBps": round(fin_bytes / (us_fin * 1e-6) / 1e9, 1),
            "layer_plus_finalize_us": round(us_layer_y, 2),
        }
    del w13, w2
    return res


def latent_measurements(fme, dev, args, flush, calls=20):
    """Latent-MoE shape (H 3584, I 2048, 896 experts, top_k 16, FP32 logits, skewed
    bias N(0, 0.5)) at M = 1, 5, 16, 32: median microseconds of `calls` calls,
    L2 flushed before each, fresh logits each call; GB/s = unique experts x
    22,025,472 B over the call's time."""
    import torch
    from synth import workloads as W

    cfg = W.LATENT
    per_expert = 4096 * 3584 + 3584 * 2048 + 4 * (32 * 28 + 28 * 16)
    w13, s13, w2, s2 = W.fp8_weights_device(cfg, args.seed, dev)
    ws = fme.Workspace(fme.moe_routed_fp8_workspace(max(cfg.Ms), cfg.H, cfg.I, cfg.E, cfg.top_k), dev)
    res = {}
    for M in cfg.Ms:
        x, _, bias = W.fp8_activations(cfg, M, args.seed, 0)
        xd = torch.from_numpy(x).to(dev).to(torch.bfloat16)
        bd = torch.from_numpy(bias).to(dev)
        lgs = [torch.from_numpy(W.fp8_activations(cfg, M, args.seed, 100 + i)[1]).to(dev) for i in range(calls + 3)]
        us, gbs, uq = [], [], []
        for i, ld in enumerate(lgs):
            flush.amax()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            _, ids, _ = fme.moe_routed_fp8(xd, ld, bd, w13, s13, w2, s2, cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0,
                                           workspace=ws)
            b.record()
            torch.cuda.synchronize()
            if i >= 3:
                t = a.elapsed_time(b) * 1e3
                u = len(set(ids.reshape(-1).tolist()))
                us.append(t)
                uq.append(u)
                gbs.append(u * per_expert / (t * 1e-6) / 1e9)
        if ws.error():
            raise RuntimeError("device wait timed out in the latent measurement")
        res[f"latent_routed_fp8_M{M}"] = {"us_median": round(float(np.median(us)), 2),
                                         "unique_experts_mean": round(float(np.mean(uq)), 2),
                                         "GBps_median": round(float(np.median(gbs)), 1)}
    del w13, w2
    return res


def side_measurements(fme, dev, args):
    """Shared expert (UE8M0, H 7168 / I 2048) and NVFP4 slot MoE latencies."""
    import torch
    from synth import workloads as W

    res = {}
    cfg = W.SHARED
    w13, s13, w2, s2 = W.shared_weights_host(cfg, args.seed)
    w13, s13, w2, s2 = (torch.from_numpy(v).to(dev) for v in (w13, s13, w2, s2))
    shared_bytes = w13.numel() + w2.numel() + 4 * (s13.numel() + s2.numel())
    flush = torch.ones(128 * 1024 * 1024, dtype=torch.int32, device=dev)
    res.update(layer_measurements(fme, dev, args, (w13, s13, w2, s2), shared_bytes, flush))
    res.update(latent_measurements(fme, dev, args, flush))
    for M in (1, 8):
        x = torch.from_numpy(W.fp8_activations(W.DSV3, M, args.seed, 3)[0]).to(dev).to(torch.bfloat16)
        ts = []
        for i in range(30):
            flush.amax()  # evict the 44 MB of weights from L2 between calls (reads only)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fme.shared_expert_fp8(x, w13, s13, w2, s2, cfg.limit, cfg.ue8m0)
            b.record()
            torch.cuda.synchronize()
            if i >= 5:
                ts.append(a.elapsed_time(b) * 1e3)
        us = float(np.median(ts))
        res[f"shared_expert_fp8_M{M}"] = {"us_median": round(us, 2),
                                         "GBps": round(shared_bytes / (us * 1e-6) / 1e9, 1)}
    # NVFP4 slot MoE: 48 local experts of a 384-expert router (bytes = unique
    # local experts x 37,158,912 B of packed E2M1 weights + UE4M3 scales).
    # Routing fused in (fme_moe_layer_nvfp4): the router's logits and bias over its
    # 384 experts pick the routes; unique local experts counted from the kernel's ids.
    ncfg = W.NVFP4
    nw = W.nvfp4_weights_device(ncfg, args.seed, dev)
    per_expert = 6144 * 3584 + 7168 * 1536 + 6144 * 448 + 7168 * 192
    for M in ncfg.Ms:
        x, logits, rbias = W.nvfp4_activations(ncfg, M, args.seed, 5)
        xd = torch.from_numpy(x).to(dev).to(torch.bfloat16)
        ld, bd = torch.from_numpy(logits).to(dev), torch.from_numpy(rbias).to(dev)
        _, ids, _ = fme.moe_layer_nvfp4(xd, ld, bd, *nw, ncfg.e0, ncfg.top_k, 1.0, ncfg.limit)
        uniq = len({int(e) for e in ids.reshape(-1).tolist() if ncfg.e0 <= e < ncfg.e0 + ncfg.L})
        ts = []
        for i in range(25):
            flush.amax()  # reads 512 MB: L2 holds none of the weights, and no dirty lines
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record()
            fme.moe_layer_nvfp4(xd, ld, bd, *nw, ncfg.e0, ncfg.top_k, 1.0, ncfg.limit)
            b.record()
            torch.cuda.synchronize()
            if i >= 5:
                ts.append(a.elapsed_time(b) * 1e3)
        us = float(np.median(ts))
        res[f"nvfp4_slot_moe_M{M}"] = {"us_median": round(us, 2), "unique_local_experts": uniq,
                                       "GBps": round(uniq * per_expert / (us * 1e-6) / 1e9, 1) if uniq else 0.0}
    # Single-GPU forms of the expert-parallel dispatch quantiser and the combine's
    # reduction + RMSNorm on the latent shape (H 3584, 16 ranks), T = 8 and 64 tokens.
    H = 3584
    for T in (8, 64):
        rng = np.random.default_rng(args.seed + T)
        x = torch.from_numpy(rng.normal(size=(T, H)).astype(np.float32)).to(dev).to(torch.bfloat16)
        parts = torch.from_numpy(rng.normal(size=(T, 16, H)).astype(np.float32)).to(dev).to(torch.bfloat16)
        gam = torch.from_numpy(rng.uniform(0.5, 1.5, H).astype(np.float32)).to(dev).to(torch.bfloat16)
        us_q = _event_us(lambda: fme.mxfp8_quantize(x), flush)
        us_c = _event_us(lambda: fme.combine_rmsnorm(parts, gam, 1e-5), flush)
        res[f"mxfp8_quantize_T{T}"] = {"us_median": round(us_q, 2),
                                       "GBps": round(T * H * (2 + 1 + 1 / 32) / (us_q * 1e-6) / 1e9, 1)}
        res[f"combine_rmsnorm_N16_T{T}"] = {"us_median": round(us_c, 2),
                                            "GBps": round((T * 16 * H + 2 * T * H + H) * 2 / (us_c * 1e-6) / 1e9, 1)}
    del flush
    return res


def nvfp4_launches(args):
    """Two NVFP4 slot-MoE calls (routing fused in) at each of M = 1, 8, 64 on the
    48-expert workload, nothing else: the command the profiler launch lists of this
    kernel are taken on."""
    import torch
    import fp4_moe_expert_gb300 as fme
    from synth import workloads as W
    dev = torch.device("cuda", 0)
    ncfg = W.NVFP4
    nw = W.nvfp4_weights_device(ncfg, args.seed, dev)
    for M in (1, 8, 64):
        x, logits, rbias = W.nvfp4_activations(ncfg, M, args.seed, 5)
        xd = torch.from_numpy(x).to(dev).to(torch.bfloat16)
        ld, bd = torch.from_numpy(logits).to(dev), torch.from_numpy(rbias).to(dev)
        for _ in range(2):
            fme.moe_layer_nvfp4(xd, ld, bd, *nw, ncfg.e0, ncfg.top_k, 1.0, ncfg.limit)
        torch.cuda.synchronize()
    print(json.dumps({"nvfp4_launches": 6}))


def shared_launches(args):
    """The FP8 shared expert alone (UE8M0, H 7168 / I 2048), two calls at each of
    M = 1 and 8, nothing else: the command the profiles of that launch are taken on."""
    import torch
    import fp4_moe_expert_gb300 as fme
    from synth import workloads as W
    dev = torch.device("cuda", 0)
    cfg = W.SHARED
    w13, s13, w2, s2 = (torch.from_numpy(v).to(dev) for v in W.shared_weights_host(cfg, args.seed))
    for M in (1, 8):
        x = torch.from_numpy(W.fp8_activations(W.DSV3, M, args.seed, 3)[0]).to(dev).to(torch.bfloat16)
        for _ in range(2):
            fme.shared_expert_fp8(x, w13, s13, w2, s2, cfg.limit, cfg.ue8m0)
        torch.cuda.synchronize()
    print(json.dumps({"shared_launches": 4}))


def mx_launches(args):
    """Per M = 1, 2, 4, 8: one BF16-token and one MXFP8-token routed FP8 call on the
    DeepSeek-V3 shape (``--experts`` resident), nothing else: the command the
    profiles comparing the two instantiations are taken on."""
    import dataclasses

    import torch
    import fp4_moe_expert_gb300 as fme
    from synth import workloads as W
    dev = torch.device("cuda", 0)
    cfg = dataclasses.replace(W.DSV3_UE8M0, E=args.experts)
    w13, s13, w2, s2 = W.fp8_weights_device(cfg, args.seed, dev)
    for M in MS:
        x, logits, bias = W.fp8_activations(cfg, M, args.seed, 7)
        xd = torch.from_numpy(x).to(dev).to(torch.bfloat16)
        ld = torch.from_numpy(logits).to(dev).to(torch.bfloat16)
        bd = torch.from_numpy(bias).to(dev)
        xq, xsc = fme.mxfp8_quantize(xd)
        rest = (ld, bd, w13, s13, w2, s2, cfg.top_k, cfg.limit, cfg.scale, cfg.ue8m0)
        fme.moe_routed_fp8(xd, *rest)
        fme.moe_routed_fp8_mx(xq, xsc, *rest)
        torch.cuda.synchronize()
    print(json.dumps({"mx_launches": 2 * len(MS)}))


def main():
    args = parse_args()
    if args.mx_launches:
        mx_launches(args)
        return
    if args.nvfp4_launches:
        nvfp4_launches(args)
        return
    if args.shared_launches:
        shared_launches(args)
        return
    rank = int(os.environ.get("RANK", 0))
    world = int(os.environ.get("WORLD_SIZE", 1))
    local_rank = int(os.environ.get("LOCAL_RANK", 0))
    if args.impl == "reference":
        reference_arm(args, rank)
        return
    gpu_arm(args, rank, world, local_rank)


if __name__ == "__main__":
    main()
