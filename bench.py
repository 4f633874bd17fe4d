"""Benchmark of the FFN-server MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config qwen3_bf16] [--B 395] [--M 8] [--n-micro 1]

One step = one pass of the whole layer (router -> routing tables -> pack ->
gate/up GEMM -> down GEMM -> combine) over one aggregated batch of T = B*M
tokens from M source buffers, inputs already resident in HBM.  The default
workload is the Qwen3-235B-A22B-shaped bf16 layer at its largest aggregated
decode batch (B=395 per attention instance, M=8 instances, T=3160).

Prints ONE JSON line (rank 0).  ``value`` is whole-job tokens/s; ``tflops``
and ``layer_roofline`` give TFLOPS and the fraction of the layer roofline
(slower of FLOPs at the measured bf16 tensor peak and algorithmic bytes at
the measured HBM bandwidth); ``roofline`` is the dominant kernel's (the
grouped gate/up GEMM) achieved HBM bandwidth against the measured peak.
``e2e`` is the same metric through the host-buffer entry points with pinned
host buffers, every step's copies in the timed region: the asynchronous call
(consecutive batches, one's copies overlapping the previous one's compute),
with the synchronous call's rate under ``e2e.sync``.  ``cpu_baseline`` is the CPU oracle on
a bounded sample of the same workload.

``--impl reference`` times the CPU oracle itself (the reference of this
build) on a bounded sample of the workload per step.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from ffn_side_attention_gb300 import roofline, synth  # noqa: E402

METRIC = "MoE-FFN tokens/s and TFLOPS on 1 GB300; fraction of roofline per batch size"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def recorded_traffic(kernel_file: str, cfg):
    """ncu capture records of the gate/up GEMM launch for the layer's shapes (H, I,
    dtype), from the committed summaries of that kernel; empty when its source changed
    since the captures."""
    import hashlib

    p = os.path.join(ROOT, "profiles", "traffic.json")
    src = os.path.join(ROOT, "ffn_side_attention_gb300", "csrc", kernel_file)
    if not (os.path.exists(p) and os.path.exists(src)):
        return []
    with open(p) as f:
        recs = json.load(f).get(kernel_file) or []
    with open(src, "rb") as f:
        h = hashlib.sha256(f.read()).hexdigest()
    return [r for r in recs if r.get("source_sha256") == h and
            (r.get("H"), r.get("I"), r.get("dtype")) == (cfg.H, cfg.I, cfg.dtype)]


def tc_peak(peaks, dtype):
    """Dense tensor peak for the layer's dtype, TFLOP/s (fp8 = 2x the bf16 measurement, the nominal ratio)."""
    bf16 = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
    return bf16 * (2.0 if dtype == "fp8" else 1.0)


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.lines = []
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "100"]
        uuid = getattr(torch.cuda.get_device_properties(device_index), "uuid", None)
        if uuid is not None:
            u = str(uuid)
            cmd.insert(1, f"--id={u if u.startswith('GPU-') else 'GPU-' + u}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in out.strip().splitlines():
            p = [x.strip() for x in ln.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                mx.append(float(p[2]))
                pw.append(float(p[3]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        # samples under load: power above the midpoint of the observed range
        thr = (min(pw) + max(pw)) / 2 if pw else 0
        load = [s for s, w in zip(sm, pw) if w >= thr] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "samples_under_load": len(load), "power_w_max": max(pw)}


# ------------------------------------------------------------------ distributed
# One process per GPU (torchrun), each an independent replica of the layer:
# the path has no exchange step, so the only collectives are the barrier
# around the timed region and the max of the ranks' times.  NCCL on GPUs,
# gloo where there is no GPU (the multi-rank logic is tested that way).
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        if torch.cuda.is_available():
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        else:
            dist.init_process_group("gloo")
    return world, rank, local


def _reduce_device():
    import torch.distributed as dist

    return "cuda" if dist.get_backend() == "nccl" else "cpu"


def barrier_max(world, seconds: float) -> float:
    """Largest of the ranks' times (every rank gets it)."""
    if world == 1:
        return seconds
    import torch.distributed as dist

    t = torch.tensor([seconds], device=_reduce_device(), dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def job_rate(world, units_per_rank, seconds):
    """Whole-job throughput: the units all replicas processed / the slowest rank's time."""
    return world * units_per_rank / seconds


# ------------------------------------------------------------------ CPU oracle leg
def oracle_sample(cfg, srcs_dev, weights_dev, n_tokens):
    """Oracle (all host cores) on the first n_tokens of the workload, whole
    layer (routing + experts + combine).  -> (seconds, tokens, cores)"""
    import oracle

    oracle.build()
    x = torch.cat([s for s in srcs_dev])[:n_tokens]
    src = [synth.to_numpy_bits(x)]
    w = synth.weights_numpy(weights_dev)
    c = dict(H=cfg.H, I=cfg.I, E=cfg.E, k=cfg.k, S=cfg.S, dtype=cfg.dtype)
    t0 = time.perf_counter()
    oracle.moe_forward(c, src, w)
    dt = time.perf_counter() - t0
    return dt, n_tokens, oracle.num_threads(), w, c, src


def default_sample_tokens(cfg):
    # about 10-20 s of oracle work on 16 host cores
    per_tok = 6.0 * (cfg.k + cfg.S) * cfg.H * cfg.I  # FLOPs per token
    return max(8, min(cfg.T, int(16 * 12 * 0.75e9 / per_tok)))


# ------------------------------------------------------------------ roofline of one workload
def routing_roofline(layer, cfg, xall, n_mb, stream, peaks):
    """Touched experts per micro-batch (from one forward of each micro-batch's tokens) and
    the layer roofline summed over micro-batches: each micro-batch is its own forward and
    streams its own experts' weights."""
    T = xall.shape[0]
    ptc = tc_peak(peaks, cfg.dtype)
    q, rem = divmod(T, n_mb)
    sizes = [q + (1 if i < rem else 0) for i in range(n_mb)]
    flops = lbytes = t_roof = 0.0
    touched_list = []
    bound = "hbm"
    t0_ = 0
    for sz in sizes:
        sub = [xall[t0_:t0_ + sz]]
        layer.forward(sub, [torch.empty_like(sub[0])], stream=stream)
        r = layer.routing(sz)
        tch = int((r["counts"].cpu() > 0).sum().item())
        touched_list.append(tch)
        f_i = roofline.layer_flops(cfg, sz)
        b_i = roofline.layer_bytes(cfg, sz, tch)
        tr_i, bound = roofline.t_roof(f_i, b_i, ptc, peaks["hbm_gbs"])
        flops += f_i
        lbytes += b_i
        t_roof += tr_i
        t0_ += sz
    return dict(sizes=sizes, touched=touched_list, flops=flops, bytes=lbytes, t_roof=t_roof, bound=bound, ptc=ptc)


def gemm_roofline(cfg, size0, touched0, k_avg, peaks):
    """Roofline of the two GEMM launches of one (micro-)batch against their profiled times."""
    ptc = tc_peak(peaks, cfg.dtype)
    gu_bytes = roofline.gateup_bytes(cfg, size0, touched0)
    dn_bytes = roofline.down_bytes(cfg, size0, touched0)
    t_gemm = (k_avg["gemm_gateup"] + k_avg["gemm_down"]) / 1e3
    t_r, _ = roofline.t_roof(roofline.layer_flops(cfg, size0), gu_bytes + dn_bytes, ptc, peaks["hbm_gbs"])
    return dict(t_roof_ms=t_r * 1e3, t_ms=t_gemm * 1e3, frac=t_r / t_gemm if t_gemm > 0 else None), gu_bytes, dn_bytes


def profile_kernels(layer, fwd, n):
    """Average per-kernel milliseconds over n forwards run by fwd(i) with CUDA events around
    each kernel (an untimed pass first creates the library's events)."""
    layer.profile_begin()
    for i in range(n):
        fwd(i)
    layer.profile_end()
    torch.cuda.synchronize()
    layer.profile_begin()
    for i in range(n):
        fwd(i)
    kms, nf = layer.profile_end()
    return {k: v / max(nf, 1) for k, v in kms.items()}


# ------------------------------------------------------------------ per-batch sweep
# Every decode batch of the workloads, one entry each: the Qwen3 bf16 layer at
# B in {6, 48, 197, 395} x M in {1, 4, 8}, its fp8 variant at 4 x 395, the
# DeepSeek-V3 fp8 layer at T in {512, 2048, 4096}, the Step3 layer as three
# micro-batches of 8 x 256, and the tiny fp32 layer.
def sweep_points():
    pts = [("qwen3_bf16", b, m, 1) for (b, m) in synth.CONFIGS["qwen3_bf16"].batches]
    pts.append(("qwen3_fp8", 395, 4, 1))
    pts += [("dsv3_fp8", b, m, 1) for (b, m) in synth.CONFIGS["dsv3_fp8"].batches]
    pts.append(("step3_bf16", 256, 8, 3))
    pts.append(("tiny_fp32", 32, 2, 1))
    return pts


def measure_point(layer, cfg, n_micro, peaks, stream, local, min_s=0.3):
    """One per-batch entry: tokens/s over a timed run of at least min_s seconds (CUDA
    events on the launching stream, clocks sampled during it), the layer and GEMM
    rooflines and the per-kernel split."""
    T = cfg.T
    inputs = [synth.make_sources(cfg, "cuda", seed=s) for s in range(4)]
    outs = [[torch.empty_like(x) for x in srcs] for srcs in inputs]

    def step(i):
        layer.forward(inputs[i % 4], outs[i % 4], stream=stream, n_micro=n_micro)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(5):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    est = max(e0.elapsed_time(e1) / 5e3, 1e-6)
    steps = int(min(2000, max(20, min_s / est)))
    sampler = ClockSampler(local)
    time.sleep(0.2)
    t_spin = time.perf_counter()
    i = 0
    while time.perf_counter() - t_spin < 0.15:
        step(i)
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    layer.check()
    ms = e0.elapsed_time(e1) / steps
    xall = torch.cat(inputs[0])
    rl = routing_roofline(layer, cfg, xall, n_micro, stream, peaks)
    size0 = rl["sizes"][0]
    prof_in = [xall[:size0]]
    prof_out = [torch.empty_like(prof_in[0])]
    if n_micro == 1:
        k_avg = profile_kernels(layer, step, min(steps, 30))
    else:
        k_avg = profile_kernels(layer, lambda i: layer.forward(prof_in, prof_out, stream=stream), min(steps, 30))
    gr, _, _ = gemm_roofline(cfg, size0, rl["touched"][0], k_avg, peaks)
    return {
        "workload": f"{cfg.name} B={cfg.B} M={cfg.M} T={T}" + (f" n_micro={n_micro}" if n_micro > 1 else ""),
        "T": T, "n_micro": n_micro, "steps": steps, "ms_per_step": ms, "value": T / (ms / 1e3),
        "unit": "tokens/s", "tflops": rl["flops"] / (ms / 1e3) / 1e12,
        "layer_roofline": {"t_roof_ms": rl["t_roof"] * 1e3, "bound": rl["bound"], "frac": rl["t_roof"] / (ms / 1e3),
                           "touched_experts": rl["touched"][0] if n_micro == 1 else rl["touched"]},
        "gemm_roofline": gr,
        "kernel_ms": k_avg,
        "gpu_launches_per_step": sum(layer.launches_per_forward(sz) for sz in rl["sizes"]),
        "clocks": clocks,
    }


def per_batch_sweep(peaks, stream, local, reuse=None):
    """All sweep points, grouped by layer so each layer's weights are made once.  `reuse`
    = (cfg, layer) of a layer already built for the largest batch of its workload."""
    from ffn_side_attention_gb300 import afd

    entries = []
    by_name = {}
    for name, b, m, nm in sweep_points():
        by_name.setdefault(name, []).append((b, m, nm))
    for name, pts in by_name.items():
        base = synth.CONFIGS[name]
        max_t = max(b * m for b, m, _ in pts)
        max_m = max(m for _, m, _ in pts)
        if reuse is not None and reuse[0].name == name and reuse[0].T >= max_t and reuse[0].M >= max_m:
            layer, own = reuse[1], False
        else:
            w = synth.make_weights(base, "cuda")
            layer = afd.MoELayer(base.H, base.I, base.E, base.k, base.dtype, w, n_shared=base.S, max_tokens=max_t,
                                 max_sources=max_m)
            del w
            torch.cuda.empty_cache()
            own = True
        for b, m, nm in pts:
            entries.append(measure_point(layer, base.with_batch(b, m), nm, peaks, stream, local))
        if own:
            layer.close()
            del layer
            torch.cuda.empty_cache()
    return entries


# ------------------------------------------------------------------ main legs
def run_reference(args, world, rank):
    if rank != 0:
        return
    cfg = synth.CONFIGS[args.config].with_batch(args.B, args.M)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    srcs = synth.make_sources(cfg, dev)
    w = synth.make_weights(cfg, dev)
    import oracle

    oracle.build()
    wn = synth.weights_numpy(w)
    c = dict(H=cfg.H, I=cfg.I, E=cfg.E, k=cfg.k, S=cfg.S, dtype=cfg.dtype)
    xall = torch.cat(srcs)
    if args.cpu_sample:
        n = args.cpu_sample
    else:
        # size each step so that warmup + steps take about two minutes (at most 2 s a step)
        n0 = min(8, cfg.T)
        t0 = time.perf_counter()
        oracle.moe_forward(c, [synth.to_numpy_bits(xall[:n0])], wn)
        per_tok = (time.perf_counter() - t0) / n0
        budget = min(2.0, 120.0 / max(args.steps + args.warmup, 1))
        n = int(max(1, min(cfg.T, budget / max(per_tok, 1e-9))))
    src = [synth.to_numpy_bits(xall[:n])]
    for _ in range(args.warmup):
        oracle.moe_forward(c, src, wn)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.moe_forward(c, src, wn)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    value = n / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{cfg.name} B={cfg.B} M={cfg.M} T={cfg.T}", "sample_tokens": n,
                   "H": cfg.H, "I": cfg.I, "E": cfg.E, "k": cfg.k, "S": cfg.S, "layer_dtype": cfg.dtype},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"first {n} tokens of the workload, whole layer, per step"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    from ffn_side_attention_gb300 import afd

    torch.cuda.set_device(local)
    cfg = synth.CONFIGS[args.config].with_batch(args.B, args.M)
    T = cfg.T
    peaks, peak_src = load_peaks()
    w = synth.make_weights(cfg, "cuda")
    n_sets = 4  # rotating input sets
    inputs = [synth.make_sources(cfg, "cuda", seed=s) for s in range(n_sets)]
    outs = [[torch.empty_like(x) for x in srcs] for srcs in inputs]
    layer = afd.MoELayer(cfg.H, cfg.I, cfg.E, cfg.k, cfg.dtype, w, n_shared=cfg.S, max_tokens=T,
                         max_sources=max(cfg.M, 1))
    stream = torch.cuda.current_stream()

    def step(i):
        layer.forward(inputs[i % n_sets], outs[i % n_sets], stream=stream, n_micro=args.n_micro)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    layer.check()

    # --graph: the timed steps replay CUDA graphs that captured one forward per input set
    # (the library enqueues no host synchronisation and keeps no per-launch host state on
    # the device path, so a capture replays the forward exactly); the per-kernel profile
    # and the end-to-end legs stay eager.
    timed_step = step
    if args.graph:
        graphs = []
        for j in range(n_sets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                layer.forward(inputs[j], outs[j], stream=torch.cuda.current_stream(), n_micro=args.n_micro)
            graphs.append(g)
        torch.cuda.synchronize()

        def timed_step(i):
            graphs[i % n_sets].replay()

        for i in range(args.warmup):
            timed_step(i)
        torch.cuda.synchronize()
        layer.check()

    sampler = ClockSampler(local) if rank == 0 else None
    if sampler is not None:
        time.sleep(0.3)
    # a short spin-up so the clock samples see the load
    t_spin = time.perf_counter()
    i = 0
    while time.perf_counter() - t_spin < 0.5:
        timed_step(i)
        i += 1
        if i % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()

    # The value: K steps with nothing recorded between the kernels (each kernel's
    # launch overlaps the previous one's tail through programmatic dependent launch).
    n_mb = max(args.n_micro, 1)
    barrier(world)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(args.steps):
        timed_step(i)
    ev1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    elapsed = barrier_max(world, ev0.elapsed_time(ev1) / 1e3)
    clocks = sampler.stop() if sampler is not None else None
    layer.check()
    ms_step = elapsed / max(args.steps, 1) * 1e3

    # Step-time spread: K more steps with an event between consecutive forwards (the
    # event keeps the next forward's first kernel from launching during the previous
    # one's last), for the median and p10 / p90 of single steps.
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    evs[0].record(stream)
    for i in range(args.steps):
        timed_step(i)
        evs[i + 1].record(stream)
    torch.cuda.synchronize()
    per_step = sorted(evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps))

    def pct(q):
        return per_step[min(len(per_step) - 1, int(q * (len(per_step) - 1) + 0.5))] if per_step else None

    # Per-kernel times (the roofline's kernel): K more steps on one stream with CUDA
    # events recorded around every kernel.  The events serialise the launches, so these
    # steps run slightly slower than the value's.  The library creates the events on
    # first use, so an untimed pass creates them first.
    prof_timed = n_mb == 1
    if prof_timed:
        k_avg = profile_kernels(layer, step, args.steps)

    # routing statistics of input set 0 (touched experts), per micro-batch:
    # each micro-batch is its own forward and streams its own experts' weights
    xall = torch.cat(inputs[0])
    rl = routing_roofline(layer, cfg, xall, n_mb, stream, peaks)
    sizes, touched_list = rl["sizes"], rl["touched"]
    flops, lbytes, t_roof, bound, ptc = rl["flops"], rl["bytes"], rl["t_roof"], rl["bound"], rl["ptc"]
    touched = touched_list[0] if n_mb == 1 else touched_list

    # with micro-batches (three streams), per-kernel times come from a separate
    # pass of the first micro-batch alone on one stream
    if not prof_timed:
        prof_in = [xall[:sizes[0]]]
        prof_out = [torch.empty_like(prof_in[0])]
        k_avg = profile_kernels(layer, lambda i: layer.forward(prof_in, prof_out, stream=stream),
                                min(args.steps, 50))
    step_s = ms_step / 1e3
    gr, gu_bytes, dn_bytes = gemm_roofline(cfg, sizes[0], touched_list[0], k_avg, peaks)
    gu_s = k_avg["gemm_gateup"] / 1e3
    dn_s = k_avg["gemm_down"] / 1e3
    # the gate/up launch's own bound: tensor if its FLOPs at the dense tensor
    # peak take longer than its algorithmic bytes at the HBM peak
    gu_flops = roofline.gateup_flops(cfg, sizes[0])
    gu_tensor = gu_flops / (ptc * 1e12) > gu_bytes / (peaks["hbm_gbs"] * 1e9)
    if gu_tensor:
        achieved = gu_flops / gu_s / 1e12 if gu_s > 0 else None
        rf_peak, rf_unit = ptc, "TFLOP/s"
    else:
        achieved = gu_bytes / gu_s / 1e9 if gu_s > 0 else None
        rf_peak, rf_unit = peaks["hbm_gbs"], "GB/s"
    recs = recorded_traffic("gemm_fp8.cu" if cfg.dtype == "fp8" else "gemm_tc.cu", cfg)
    exact = [r for r in recs if r.get("workload") == cfg.name and r.get("T") == sizes[0]]
    scaled = [r for r in recs if r.get("dram_bytes_per_touched_expert")]
    traffic = None
    if args.traffic is not None:
        traffic = args.traffic
    elif exact:
        traffic = exact[0]["dram_bytes_per_launch"]
    elif scaled:
        # a capture of the same shapes on fewer experts, scaled by the touched experts
        # (the bf16 gate/up traffic is weight-dominated)
        traffic = scaled[0]["dram_bytes_per_touched_expert"] * (touched_list[0] + cfg.S)

    # End to end through the host-buffer entry points (pinned memory, two input sets
    # alternating).  Every step copies its sources in and its outputs out inside the
    # timed region.  The headline uses the asynchronous call, as a serving loop would:
    # batch i+1's copies cross the host link while batch i computes.  The synchronous
    # call (copies and compute back to back) is reported beside it.
    h_in = [[x.cpu().pin_memory() for x in inputs[j]] for j in range(2)]
    h_out = [[torch.empty_like(x).pin_memory() for x in h_in[j]] for j in range(2)]
    e2e_steps = max(3, min(args.steps, 50))
    for i in range(max(2, args.warmup // 2)):
        layer.forward_host(h_in[i % 2], h_out[i % 2], stream=stream, n_micro=args.n_micro)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        layer.forward_host(h_in[i % 2], h_out[i % 2], stream=stream, n_micro=args.n_micro)
    e2e_sync_s = barrier_max(world, time.perf_counter() - t0) / e2e_steps
    for i in range(max(2, args.warmup // 2)):
        layer.forward_host_async(h_in[i % 2], h_out[i % 2], n_micro=args.n_micro)
    layer.host_wait()
    barrier(world)
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        layer.forward_host_async(h_in[i % 2], h_out[i % 2], n_micro=args.n_micro)
    layer.host_wait()
    e2e_s = barrier_max(world, time.perf_counter() - t0) / e2e_steps
    layer.check()
    io_bytes = T * cfg.H * (4 if cfg.dtype == "fp32" else 2)

    line = {
        "metric": METRIC, "value": job_rate(world, T, step_s), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": {"fp32": "f32", "bf16": "bf16", "fp8": "e4m3"}[cfg.dtype], "data": "synthetic",
        "config": {"workload": f"{cfg.name} B={cfg.B} M={cfg.M} T={T}", "H": cfg.H, "I": cfg.I, "E": cfg.E,
                   "k": cfg.k, "S": cfg.S, "n_micro": args.n_micro, "cuda_graph": bool(args.graph),
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs > L2: expert weights streamed every step; 4 rotating input sets"},
        "tflops": flops / step_s / 1e12,
        "step_ms": {"p10": pct(0.1), "p50": pct(0.5), "p90": pct(0.9), "n": len(per_step),
                    "how": "CUDA events between consecutive forwards (separate pass)"},
        "layer_roofline": {"t_roof_ms": t_roof * 1e3, "bound": bound, "frac": t_roof / step_s,
                           "flops": flops, "bytes": lbytes, "touched_experts": touched,
                           "peak_tflops": ptc, "peak_gbs": peaks["hbm_gbs"], "peaks": peak_src},
        "gemm_roofline": gr,
        "roofline": {"kernel": "gemm_gateup", "bound": "tensor" if gu_tensor else "hbm", "achieved": achieved,
                     "peak": rf_peak, "unit": rf_unit, "frac": achieved / rf_peak if achieved else None,
                     "traffic": traffic, "peak_src": peak_src},
        "kernel_ms": k_avg,
        "e2e": {"value": job_rate(world, T, e2e_s), "unit": "tokens/s", "h2d_bytes_per_step": io_bytes,
                "d2h_bytes_per_step": io_bytes, "steps": e2e_steps,
                "api": "afd_ffn_forward_host_async + afd_ffn_host_wait (consecutive batches: one's copies "
                       "overlap the previous one's compute)",
                "sync": {"value": job_rate(world, T, e2e_sync_s), "unit": "tokens/s",
                         "api": "afd_ffn_forward_host (copies and compute back to back)"}},
        "gpu_launches": args.steps * sum(layer.launches_per_forward(sz) for sz in sizes),
        "clocks": clocks,
    }
    if world == 1 and not args.no_per_batch:
        # the per-batch roofline sweep (one GPU: the metric is per GB300); the headline's
        # layer serves the workload it was built for
        del w
        torch.cuda.empty_cache()
        line["per_batch"] = per_batch_sweep(peaks, stream, local, reuse=(cfg, layer) if n_mb == 1 else None)
        w = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        n = args.cpu_sample or default_sample_tokens(cfg)
        if w is None:
            w = synth.make_weights(cfg, "cuda")
        dt, n, cores, *_ = oracle_sample(cfg, inputs[0], w, n)
        line["cpu_baseline"] = {"value": n / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                                "sample": f"first {n} of {T} tokens, whole layer (routing + experts + combine)"}
        if T <= 64:  # small batches: the oracle on one core as well
            import oracle

            oracle.set_num_threads(1)
            dt1, n1, *_ = oracle_sample(cfg, inputs[0], w, n)
            oracle.set_num_threads(cores)
            line["cpu_baseline"]["one_core"] = {"value": n1 / dt1, "unit": "tokens/s", "cores": 1}
    if rank == 0:
        print(json.dumps(line), flush=True)
    layer.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="qwen3_bf16", choices=sorted(synth.CONFIGS))
    ap.add_argument("--B", type=int, default=None)
    ap.add_argument("--M", type=int, default=None)
    ap.add_argument("--n-micro", type=int, default=None)
    ap.add_argument("--graph", action="store_true",
                    help="time CUDA-graph replays of captured forwards instead of eager launches")
    ap.add_argument("--E", type=int, default=None, help="override the expert count (small profiling cases)")
    ap.add_argument("--I", type=int, default=None, help="override the expert intermediate size (profiling cases)")
    ap.add_argument("--cpu-sample", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-batch", action="store_true",
                    help="skip the per-batch roofline sweep over every workload's decode batches")
    ap.add_argument("--traffic", type=float, default=None,
                    help="ncu dram bytes per gate/up launch, when taken for the current kernel")
    args = ap.parse_args()
    base = synth.CONFIGS[args.config]
    if args.E is not None or args.I is not None:
        import dataclasses

        E = args.E if args.E is not None else base.E
        I = args.I if args.I is not None else base.I
        synth.CONFIGS[args.config] = base = dataclasses.replace(base, E=E, I=I, name=f"{base.name}_E{E}_I{I}")
    args.B = args.B if args.B is not None else base.B
    args.M = args.M if args.M is not None else base.M
    args.n_micro = args.n_micro if args.n_micro is not None else base.n_micro
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.gpus != world:
        sys.exit(f"bench.py: --gpus {args.gpus} but WORLD_SIZE={world}; launch N > 1 ranks with "
                 f"torchrun --nproc-per-node N")
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
