"""Benchmark of the fused FP8 AdamW + DRE step on GB300.

Default workload: the Llama-2-7B-shaped parameter set (6,738,415,616 params,
G = 128), synthetic fp32 master weights and bf16 gradients (no model weights
or data).  A step is one launch of the fused kernel over the whole flat
buffer.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload llama7b]
                  [--G 128] [--impl ours|reference]

Metric: parameters updated per second (whole job), with the dominant
kernel's achieved HBM bandwidth against the measured copy peak.
--impl reference times the float64 CPU oracle on the host cores instead (a
deliberately slow baseline, bounded sample of the same workload).
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
sys.path.insert(0, ROOT)

METRIC = "FP8 AdamW+DRE step: params/s and achieved HBM GB/s (% of GB300 peak), 1 GPU"
UNIT = "params/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
KERNEL = "step_kernel_cta"
L2_BYTES = 129 * 2 ** 20


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--workload", default="llama7b")
    p.add_argument("--G", type=int, default=128)
    p.add_argument("--grads", type=int, default=3,
                   help="distinct seeded gradients generated before timing and cycled through")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--e2e-steps", type=int, default=3)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--report", default=None, choices=["dre-mse", "act-quant", "g-sweep", "linear"],
                   help="dre-mse: quantization error with and without the expansion on "
                        "AdamW-like moments, and the codec kernels' bandwidth; act-quant: "
                        "bandwidth of the per-group FP8 activation quantizer (one GPU); "
                        "g-sweep: the step over --sweep-workload for G in --sweep-G, one "
                        "JSON line per G with its roofline and clocks; linear: the FP8 linear "
                        "layer with per-group FP8 output on Llama-2-7B layer shapes, one JSON "
                        "line per shape against the tensor-core roofline")
    p.add_argument("--lin-tokens", type=int, default=8192, help="M (tokens) of the linear report")
    p.add_argument("--lin-G", type=int, default=16, help="output group size of the linear report")
    p.add_argument("--lin-shapes", default="attn_qkvo,mlp_up_gate,mlp_down,square_16k_8k_8k",
                   help="layers of the linear report (comma-separated)")
    p.add_argument("--sweep-workload", default="llama13b")
    p.add_argument("--sweep-G", default="16,32,64,128,256")
    p.add_argument("--rows", type=int, default=32768, help="M of the act-quant report")
    p.add_argument("--cols", type=int, default=8192, help="N of the act-quant report")
    p.add_argument("--params", type=int, default=1 << 30,
                   help="parameters of the dre-mse report")
    return p.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(total_ms: float, params_per_rank: int, steps: int, device=None):
    """Whole-job rate of independent replicas: every rank updates its own
    parameter set; the job takes as long as its slowest rank.

    Returns (max_ms_over_ranks, params_per_second_over_all_ranks).  With one
    process (or no process group) it is the local figure.
    """
    import torch
    ws = 1
    if torch.distributed.is_available() and torch.distributed.is_initialized():
        import torch.distributed as dist
        ws = dist.get_world_size()
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
        n = torch.tensor([float(params_per_rank)], dtype=torch.float64, device=device)
        dist.all_reduce(n, op=dist.ReduceOp.SUM)
        total_params = float(n.item())
    else:
        total_params = float(params_per_rank)
    return total_ms, total_params * steps / (total_ms / 1e3)


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "coat_fp8_adamw_gb300", "csrc")
    # every file the step kernel is compiled from (the C ABI header only declares)
    for name in ("adamw_dre_step.cu", "coat_device.cuh", "coat_df.cuh", "coat_round.cuh",
                 "coat_tables.inc", "coat_kernels.h"):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, G: int):
    """DRAM bytes per parameter of the step kernel from a committed ncu summary,
    if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(p):
        return None
    digest = kernel_source_digest()
    for line in open(p):
        f = line.split()
        if len(f) >= 4 and not line.startswith("#") and f[0] == digest and int(f[1]) == G:
            return float(f[3])  # bytes per parameter
    return None


# ---------------------------------------------------------------------------
# CPU baseline: the float64 oracle on a bounded sample of the workload
# ---------------------------------------------------------------------------
_CPU_SAMPLE = {}


def cpu_baseline(workload: str, G: int, seconds: float):
    import numpy as np

    import oracle
    from coat_fp8_adamw_gb300 import synth
    wl = synth.workload(workload, G)
    sample = min(wl.n, 1 << 24)          # a fixed contiguous slice of 2^24 parameters
    key = (sample, G)
    if key not in _CPU_SAMPLE:           # generated once per process (reference-arm steps reuse it)
        rng = np.random.default_rng(0)
        w0 = (rng.standard_normal(sample) * 0.02).astype(np.float32)
        g0 = synth.f32_to_bf16_bits((rng.standard_normal(sample) * 1e-3).astype(np.float32))
        _CPU_SAMPLE.clear()
        _CPU_SAMPLE[key] = (w0, g0) + tuple(synth.random_state_np(sample, G, seed=1))
    w0, g, mq0, vq0, meta0 = _CPU_SAMPLE[key]
    w, mq, vq, meta = w0.copy(), mq0.copy(), vq0.copy(), meta0.copy()
    hp = synth.HYPER
    threads = oracle.threads(0)
    done, t0, step = 0, time.perf_counter(), 1
    while True:
        oracle.adamw_step(w, g, mq, vq, meta, G, hp["beta1"], hp["beta2"], hp["lr"], hp["eps"],
                          hp["weight_decay"], step, nthreads=threads)
        done += sample
        step += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return {"value": done / el, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": f"{step - 1} steps over a contiguous slice of {sample} params "
                      f"({workload}-shaped, G={G}; w ~ N(0, 0.02^2), g ~ N(0, 1e-3^2), random "
                      f"stored state), {el:.1f} s of float64 CPU work; full-size step time "
                      f"extrapolated"}


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    t0 = time.perf_counter()
    per_step = []
    base = None
    for i in range(args.warmup + args.steps):
        b = cpu_baseline(args.workload, args.G, max(1.0, args.cpu_seconds / 4))
        if i >= args.warmup:
            per_step.append(b["value"])
        base = b
    value = statistics.median(per_step) if per_step else base["value"]
    from coat_fp8_adamw_gb300 import synth
    n = synth.workload(args.workload, args.G).n
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": n / value * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{args.workload}-shaped parameter set", "G": args.G,
                       "params": n, "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": base["cores"],
                             "kind": "oracle", "sample": base["sample"]},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "wall_s": time.perf_counter() - t0}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def quantile(xs, q: float) -> float:
    """Nearest-rank quantile of a list of launch times."""
    ys = sorted(xs)
    return ys[min(len(ys) - 1, max(0, int(round(q * (len(ys) - 1)))))]


def l2_note(working_set_bytes: float) -> str:
    if working_set_bytes > 10 * L2_BYTES:
        return "working set %.1f GB >> 129 MB L2: no flush needed" % (working_set_bytes / 1e9)
    return ("working set %.2f GB is comparable to the 129 MB L2: timings are L2-affected "
            "(a parity case, not a bench configuration)" % (working_set_bytes / 1e9))


def run_ours(args):
    import torch

    import coat_fp8_adamw_gb300 as coat
    from coat_fp8_adamw_gb300 import synth

    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    coat.lib()  # fail loudly if the library is missing

    wl = synth.workload(args.workload, args.G)
    n, G = wl.n, wl.G
    ng = coat.num_groups(n, G)
    hp = synth.HYPER
    w = synth.init_weights_torch(wl, dev)
    # a training run sees a new gradient every step: K distinct seeded
    # gradients are generated before the timed region and cycled through
    grads = [synth.grad_torch(wl, 1 + i, dev) for i in range(max(1, args.grads))]
    n_grads = len(grads)
    g = grads[0]
    mq = torch.zeros(n, dtype=torch.uint8, device=dev)
    vq = torch.zeros(n, dtype=torch.uint8, device=dev)
    meta = torch.zeros(ng, 4, dtype=torch.float32, device=dev)
    meta[:, 1] = 1.0
    meta[:, 3] = 1.0
    torch.cuda.synchronize()

    stream = torch.cuda.current_stream(dev)

    def step(t):
        coat.coat_fp8_adamw_step(w, grads[(t - 1) % len(grads)], mq, vq, meta, G, hp["beta1"],
                                 hp["beta2"], hp["lr"], hp["eps"], hp["weight_decay"], t,
                                 stream=stream)

    t = 0
    for _ in range(args.warmup):
        t += 1
        step(t)
    torch.cuda.synchronize()

    def barrier():
        if ws > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier()
    # the timed region is the profiler's capture range (ncu --profile-from-start off)
    torch.cuda.profiler.start()
    t_begin = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_begin.record(stream)
    for i in range(args.steps):
        t += 1
        starts[i].record(stream)
        step(t)
        ends[i].record(stream)
    t_end.record(stream)
    barrier()
    torch.cuda.profiler.stop()
    clk = clocks.stop()
    total_ms = t_begin.elapsed_time(t_end)
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms, value = aggregate(total_ms, n, args.steps, device=dev)
    ms_per_step = total_ms / args.steps
    avg_launch = statistics.mean(launch_ms)
    bpp = coat.bytes_per_param(G)
    achieved = bpp * n / (avg_launch / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    traffic_bpp = recorded_traffic(args.workload, G)

    del grads[1:]            # the end-to-end leg streams the first gradient only
    torch.cuda.empty_cache()

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e and args.e2e_steps > 0:
        e2e = e2e_leg(args, coat, synth, torch, dev, w, g, mq, vq, meta, n, G, ng, hp, t)

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(args.workload, G, args.cpu_seconds)

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "data": "synthetic",
                "config": {"workload": f"{args.workload}-shaped parameter set", "G": G,
                           "params": n, "groups": ng, "bytes_per_param": bpp,
                           "parallelism": "replicas" if ws > 1 else "single GPU",
                           "gradients": f"{n_grads} distinct seeded gradients, cycled",
                           "l2": l2_note(bpp * n)},
                "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                             "unit": "GB/s", "frac": achieved / peak,
                             "peak_kind": f"{peak_kind} (copy bandwidth)",
                             "traffic": (traffic_bpp * n) if traffic_bpp else None,
                             "kernel": KERNEL, "avg_launch_ms": avg_launch,
                             "median_launch_ms": statistics.median(launch_ms),
                             "p10_launch_ms": quantile(launch_ms, 0.1),
                             "p90_launch_ms": quantile(launch_ms, 0.9),
                             "min_launch_ms": min(launch_ms), "max_launch_ms": max(launch_ms)},
                "gpu_launches": args.steps,
                "clocks": clk,
                "e2e": e2e,
                "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def e2e_leg(args, coat, synth, torch, dev, w, g, mq, vq, meta, n, G, ng, hp, t):
    """The same step through the library's host-buffer entry point: w, g,
    codes and meta live in pinned host memory, and coat_fp8_adamw_step_host
    streams them through a device workspace (chunks on three streams, copies in
    both directions overlapping the kernel).  Every step moves the whole state
    host->device and back; the call returns when the host holds the result."""
    chunk = min(n, 1 << 27)
    try:
        hw = torch.empty(n, dtype=torch.float32, pin_memory=True)
        hg = torch.empty(n, dtype=torch.bfloat16, pin_memory=True)
        hmq = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        hvq = torch.empty(n, dtype=torch.uint8, pin_memory=True)
        hmeta = torch.empty(ng, 4, dtype=torch.float32, pin_memory=True)
    except RuntimeError as e:
        return {"error": f"pinned host allocation failed: {e}"}
    hw.copy_(w)
    hg.copy_(g)
    hmq.copy_(mq)
    hvq.copy_(vq)
    hmeta.copy_(meta)
    ws = torch.empty(coat.coat_fp8_adamw_step_host_workspace_bytes(chunk, G), dtype=torch.uint8,
                     device=dev)

    def one_step(step_t):
        coat.coat_fp8_adamw_step_host(hw, hg, hmq, hvq, hmeta, G, hp["beta1"], hp["beta2"],
                                      hp["lr"], hp["eps"], hp["weight_decay"], step_t, ws)

    one_step(t + 1)  # warm-up
    torch.cuda.profiler.start()
    t0 = time.perf_counter()
    for i in range(args.e2e_steps):
        one_step(t + 2 + i)
    el = time.perf_counter() - t0
    torch.cuda.profiler.stop()
    h2d = n * (4 + 2 + 1 + 1) + ng * 16
    d2h = n * (4 + 1 + 1) + ng * 16
    link = link_bandwidth(torch, dev, hw, ws)
    # the step's time if the copies ran at the measured link rates and the
    # kernel were free: whichever of one direction alone and both together binds
    bound_s = max(h2d / (link["h2d_gbs"] * 1e9), d2h / (link["d2h_gbs"] * 1e9),
                  (h2d + d2h) / (link["bidir_gbs"] * 1e9))
    per_step = el / args.e2e_steps
    return {"value": n * args.e2e_steps / el, "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "chunk_params": chunk,
            "link_gbs": link, "link_bound_params_per_s": n / bound_s,
            "e2e_frac_of_link": bound_s / per_step,
            "note": "coat_fp8_adamw_step_host on pinned host buffers (state offloaded to host "
                    "memory), host wall clock per call; link_gbs: plain pinned copies measured "
                    "in the same process just after (one direction, then both at once)"}


def link_bandwidth(torch, dev, host_pinned, dev_buf, reps=4):
    """Raw host<->device copy rates between pinned host memory and the device:
    host->device, device->host, and both at once on two streams (each direction
    its own buffers).  Timed with CUDA events on the copying streams, best of
    three timings each."""
    nb = min(dev_buf.numel() // 2, host_pinned.numel() * host_pinned.element_size() // 2, 1 << 30)
    hb = host_pinned.view(torch.uint8)[: 2 * nb]
    h_in, h_out = hb[:nb], hb[nb: 2 * nb]
    d_in, d_out = dev_buf[:nb], dev_buf[nb: 2 * nb]
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def timed(fn, streams):
        for s in streams:
            s.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in streams]
        for (a, _), s in zip(evs, streams):
            a.record(s)
        fn()
        for (_, b), s in zip(evs, streams):
            b.record(s)
        torch.cuda.synchronize()
        return max(a.elapsed_time(b) for a, b in evs) / 1e3

    def h2d():
        with torch.cuda.stream(s1):
            for _ in range(reps):
                d_in.copy_(h_in, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            for _ in range(reps):
                h_out.copy_(d_out, non_blocking=True)

    def both():
        h2d()
        d2h()

    both()
    # best of three of each: a single timing has come out several times low
    t_h2d = min(timed(h2d, [s1]) for _ in range(3))
    t_d2h = min(timed(d2h, [s2]) for _ in range(3))
    t_both = min(timed(both, [s1, s2]) for _ in range(3))
    return {"h2d_gbs": reps * nb / t_h2d / 1e9, "d2h_gbs": reps * nb / t_d2h / 1e9,
            "bidir_gbs": 2 * reps * nb / t_both / 1e9, "bytes_per_copy": int(nb)}


def report_dre_mse(args):
    """Quantization MSE of AdamW-like first and second moments stored as E4M3
    codes with and without Dynamic Range Expansion (the section 4 table of the
    COAT review page credits the expansion with a 1.63x lower MSE), plus the
    achieved bandwidth of the three codec kernels.  Everything runs on the GPU
    through the C ABI; the oracle cross-checks the same numbers in the tests."""
    import torch

    import coat_fp8_adamw_gb300 as coat
    from coat_fp8_adamw_gb300 import synth
    coat.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    n, G = args.params, args.G
    ng = coat.num_groups(n, G)
    stream = torch.cuda.current_stream()
    out = {"report": "dre-mse", "params": n, "G": G, "data": "synthetic AdamW-like moments",
           "moments": {}, "kernels": {}}
    peak, peak_kind = measured_peak()
    q = torch.empty(n, dtype=torch.uint8, device=dev)
    S = torch.empty(ng, dtype=torch.float32, device=dev)
    k = torch.empty(ng, dtype=torch.float32, device=dev)
    ones = torch.ones(ng, dtype=torch.float32, device=dev)
    back = torch.empty(n, dtype=torch.float32, device=dev)

    def timed(fn, bytes_moved):
        for _ in range(3):
            fn()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        torch.cuda.synchronize()
        ev[0].record(stream)
        reps = 10
        for _ in range(reps):
            fn()
        ev[1].record(stream)
        torch.cuda.synchronize()
        ms = ev[0].elapsed_time(ev[1]) / reps
        gbs = bytes_moved / (ms / 1e3) / 1e9
        return {"ms": ms, "achieved_gbs": gbs, "peak_gbs": peak, "frac": gbs / peak,
                "peak_kind": peak_kind}

    m, v = synth.adamw_like_moments_torch(n, G, 11, dev)
    for name, x in (("m", m), ("v", v)):
        xd = x.double()
        norm = float((xd * xd).mean())
        coat.coat_dre_quantize(x, G, q, S, k)
        coat.coat_dre_dequantize(q, S, k, G, back)
        mse_dre = float(((back.double() - xd) ** 2).mean())
        kk = k.double()
        coat.coat_fp8_quantize_absmax(x, G, q, S)
        coat.coat_dre_dequantize(q, S, ones, G, back)
        mse_abs = float(((back.double() - xd) ** 2).mean())
        out["moments"][name] = {"mse_dre": mse_dre, "mse_no_dre": mse_abs,
                                "relative_mse_dre": mse_dre / norm,
                                "relative_mse_no_dre": mse_abs / norm,
                                "no_dre_over_dre": mse_abs / mse_dre,
                                "k_median": float(kk.median()), "k_p10": float(kk.quantile(0.1)),
                                "k_p90": float(kk.quantile(0.9))}
    x = v
    out["kernels"]["dre_quantize"] = timed(lambda: coat.coat_dre_quantize(x, G, q, S, k),
                                           n * 5 + ng * 8)
    out["kernels"]["fp8_quantize_absmax"] = timed(lambda: coat.coat_fp8_quantize_absmax(x, G, q, S),
                                                  n * 5 + ng * 4)
    out["kernels"]["dre_dequantize"] = timed(lambda: coat.coat_dre_dequantize(q, S, k, G, back),
                                             n * 5 + ng * 8)
    print(json.dumps(out), flush=True)


def report_act_quant(args):
    """Achieved HBM bandwidth of the per-group (1 x G) FP8 activation quantizer
    with its transposed second output, over the group sizes of the section 5
    table, on a synthetic bf16 activation of --rows x --cols."""
    import torch

    import coat_fp8_adamw_gb300 as coat
    coat.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    M, N = args.rows, args.cols
    gen = torch.Generator(device=dev).manual_seed(7)
    x = torch.randn(M, N, generator=gen, device=dev)
    x = (x * torch.pow(10.0, torch.rand(M, 1, generator=gen, device=dev) * 4 - 3)).to(torch.bfloat16)
    q = torch.empty((M, N), dtype=torch.uint8, device=dev)
    qt = torch.empty((N, M), dtype=torch.uint8, device=dev)
    peak, peak_kind = measured_peak()
    stream = torch.cuda.current_stream()
    out = {"report": "act-quant", "rows": M, "cols": N, "data": "synthetic bf16 activation",
           "dtype": "bf16 in, e4m3 out", "by_G": {}}
    for G in (4, 8, 16, 32, 64, 128):
        S = torch.empty((M, N // G), dtype=torch.float32, device=dev)
        for _ in range(3):
            coat.coat_act_quantize_fp8(x, G, q, S, qt)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        torch.cuda.synchronize()
        ev[0].record(stream)
        reps = 10
        for _ in range(reps):
            coat.coat_act_quantize_fp8(x, G, q, S, qt)
        ev[1].record(stream)
        torch.cuda.synchronize()
        ms = ev[0].elapsed_time(ev[1]) / reps
        bytes_moved = M * N * (2 + 1 + 1) + (M * N // G) * 4
        gbs = bytes_moved / (ms / 1e3) / 1e9
        out["by_G"][str(G)] = {"ms": ms, "elements_per_s": M * N / (ms / 1e3),
                               "achieved_gbs": gbs, "peak_gbs": peak, "frac": gbs / peak,
                               "bytes_per_element": 4 + 4 / G, "peak_kind": peak_kind}
    print(json.dumps(out), flush=True)


def measured_fp8_peaks():
    """Dense FP8 tensor peaks (burst, sustained): the measured bf16 GEMM rates
    times the nominal FP8:bf16 ratio of 2 (4.5 / 2.25 PFLOP/s dense)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as fh:
            d = json.load(fh)
        burst = 2.0 * float(d["bf16_tflops"])
        sust = 2.0 * float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))
        return burst, sust, "measured bf16 x 2 (nominal fp8:bf16)"
    except (OSError, KeyError, ValueError):
        return 2.0 * FALLBACK_BF16_TFLOPS, 2.0 * FALLBACK_BF16_TFLOPS, "fallback bf16 x 2"


def report_linear(args):
    """The FP8 linear layer with a per-group FP8 output (coat_fp8_linear_group_quantize)
    on the linear layers of a Llama-2-7B block over --lin-tokens tokens (q/k/v/o,
    MLP up/gate, MLP down) and one 16384 x 8192 x 8192 product, one JSON line per
    shape.  Burst: 20 back-to-back launches (CUDA events on the launching
    stream) against the burst FP8 peak, with a plain FP8 GEMM from the library
    (torch._scaled_mm, bf16 output, no group quantization) timed the same way
    just before for context.  Sustained: launches for half a second with the
    clocks sampled, against the sustained (power-capped) peak."""
    import torch

    import coat_fp8_adamw_gb300 as coat
    from coat_fp8_adamw_gb300 import synth
    coat.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    T, G = args.lin_tokens, args.lin_G
    peak_b, peak_s, peak_kind = measured_fp8_peaks()
    stream = torch.cuda.current_stream(dev)
    shapes = [("attn_qkvo", T, 4096, 4096), ("mlp_up_gate", T, 11008, 4096),
              ("mlp_down", T, 4096, 11008), ("square_16k_8k_8k", 16384, 8192, 8192)]
    wanted = set(args.lin_shapes.split(","))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]

    def timed(fn, reps):
        ev[0].record(stream)
        for _ in range(reps):
            fn()
        ev[1].record(stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]) / reps

    for name, M, N, K in shapes:
        if name not in wanted:
            continue
        xq = torch.from_numpy(synth.fp8_operand_codes_np(M, K, 1)).to(dev)
        wq = torch.from_numpy(synth.fp8_operand_codes_np(N, K, 2)).to(dev)
        q = torch.empty((M, N), dtype=torch.uint8, device=dev)
        S = torch.empty((M, N // G), dtype=torch.float32, device=dev)
        sx, sw = 0.02, 0.003
        flops = 2.0 * M * N * K

        def run():
            coat.coat_fp8_linear_group_quantize(xq, sx, wq, sw, G, q, S, stream=stream)

        lib = None
        try:
            a8, b8 = xq.view(torch.float8_e4m3fn), wq.view(torch.float8_e4m3fn)
            one = torch.ones((), device=dev)

            def run_lib():
                torch._scaled_mm(a8, b8.t(), scale_a=one, scale_b=one, out_dtype=torch.bfloat16)

            timed(run_lib, 3)
            lib_ms = timed(run_lib, 20)
            lib = {"what": "torch._scaled_mm, bf16 output, no group quantization, burst",
                   "ms": lib_ms, "tflops": flops / (lib_ms / 1e3) / 1e12}
        except (RuntimeError, AttributeError, TypeError):
            pass
        timed(run, 3)
        coat.coat_kernel_wait_timeouts(reset=True)
        ms_b = timed(run, 20)
        tf_b = flops / (ms_b / 1e3) / 1e12
        reps = max(20, int(500.0 / max(ms_b, 1e-3)))   # half a second of clock samples
        clocks = ClockSampler(0)
        clocks.start()
        ms_s = timed(run, reps)
        clk = clocks.stop()
        tf_s = flops / (ms_s / 1e3) / 1e12
        timeouts = coat.coat_kernel_wait_timeouts(reset=True)
        print(json.dumps({
            "report": "linear", "layer": name, "M": M, "N": N, "K": K, "G": G,
            "metric": "fp8_linear_group_quantize_tflops", "value": tf_b, "unit": "TFLOP/s",
            "ms": ms_b, "data": "synthetic E4M3 codes (activation-like magnitudes)",
            "dtype": "e4m3 x e4m3 -> f32 accumulate -> e4m3 codes + f32 group scales",
            "roofline": {"bound": "tensor", "achieved": tf_b, "peak": peak_b, "unit": "TFLOP/s",
                         "frac": tf_b / peak_b, "peak_kind": peak_kind + ", burst",
                         "traffic": None, "kernel": "linear_fp8_kernel"},
            "sustained": {"launches": reps, "ms": ms_s, "tflops": tf_s, "peak": peak_s,
                          "frac": tf_s / peak_s, "clocks": clk},
            "output_bytes": M * N + 4 * (M * N // G),
            "library_fp8_gemm": lib, "wait_timeouts": timeouts}), flush=True)


def report_g_sweep(args):
    """The step over one model-shaped parameter set for several group sizes
    (the 13B configuration sweeps G = 16 ... 256): weights and three cycled
    gradients are generated once, the state is reset for every G, and each G
    gets warm-up steps, timed steps (CUDA events per launch on the launching
    stream), clocks sampled while they run, and its roofline line."""
    import torch

    import coat_fp8_adamw_gb300 as coat
    from coat_fp8_adamw_gb300 import synth
    coat.lib()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    wl0 = synth.workload(args.sweep_workload)
    n = wl0.n
    w = synth.init_weights_torch(wl0, dev)
    grads = [synth.grad_torch(wl0, 1 + i, dev) for i in range(max(1, args.grads))]
    hp = synth.HYPER
    peak, peak_kind = measured_peak()
    stream = torch.cuda.current_stream(dev)
    for G in (int(x) for x in args.sweep_G.split(",")):
        ng = coat.num_groups(n, G)
        mq = torch.zeros(n, dtype=torch.uint8, device=dev)
        vq = torch.zeros(n, dtype=torch.uint8, device=dev)
        meta = torch.zeros(ng, 4, dtype=torch.float32, device=dev)
        meta[:, 1] = 1.0
        meta[:, 3] = 1.0
        t = 0

        def step():
            nonlocal t
            t += 1
            coat.coat_fp8_adamw_step(w, grads[(t - 1) % len(grads)], mq, vq, meta, G, hp["beta1"],
                                     hp["beta2"], hp["lr"], hp["eps"], hp["weight_decay"], t,
                                     stream=stream)

        for _ in range(args.warmup):
            step()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        clocks = ClockSampler(0)
        clocks.start()
        time.sleep(0.3)
        for a, b in evs:
            a.record(stream)
            step()
            b.record(stream)
        torch.cuda.synchronize()
        clk = clocks.stop()
        ms = [a.elapsed_time(b) for a, b in evs]
        avg = statistics.mean(ms)
        bpp = coat.bytes_per_param(G)
        achieved = bpp * n / (avg / 1e3) / 1e9
        print(json.dumps({"report": "g-sweep", "metric": METRIC, "value": n / (avg / 1e3),
                          "unit": UNIT, "config": {"workload": f"{args.sweep_workload}-shaped "
                                                   "parameter set", "G": G, "params": n,
                                                   "groups": ng, "bytes_per_param": bpp,
                                                   "gradients": f"{len(grads)} distinct seeded "
                                                                "gradients, cycled"},
                          "steps": args.steps, "warmup": args.warmup,
                          "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                                       "unit": "GB/s", "frac": achieved / peak,
                                       "peak_kind": f"{peak_kind} (copy bandwidth)",
                                       "kernel": KERNEL, "avg_launch_ms": avg,
                                       "median_launch_ms": statistics.median(ms),
                                       "min_launch_ms": min(ms), "max_launch_ms": max(ms)},
                          "clocks": clk}), flush=True)
        del mq, vq, meta
        torch.cuda.empty_cache()


def main():
    args = parse()
    if args.report == "g-sweep":
        report_g_sweep(args)
        return
    if args.report == "linear":
        report_linear(args)
        return
    if args.report == "dre-mse":
        report_dre_mse(args)
        return
    if args.report == "act-quant":
        report_act_quant(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
