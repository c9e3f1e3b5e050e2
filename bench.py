#!/usr/bin/env python
"""Benchmark of the W4A4 MoE expert layer (per-token NVFP4 activations,
block-scaled grouped GEMMs on tcgen05) on GB300.

A step is one pass of the whole path -- route, metadata, per-token
quantization, permute, FC1 + SwiGLU + row amax, requant, FC2, weighted
combine -- over one batch of the 32768-token Qwen3-30B-A3B-shaped layer
(hidden 2048, 128 experts, top-8, FFN 768, router bias ~N(0, 2^2)), with
seeded synthetic inputs resident in HBM and the weights quantized once
before timing.  L2 is flushed (256 MiB write, then a 256 MiB read) between timed steps, outside
the timed region; each step is timed with CUDA events on the launching
stream, and per-stage events recorded by the library give the kernels'
durations live.

--gpus N runs N independent replicas (one process per GPU under torchrun):
the layer is not sharded, nothing is exchanged on the data path; the only
collectives are the barrier and the max over ranks of the timed region.
--impl reference times the CPU oracle on a bounded sample of the same
workload (rank 0 only).
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

# The CPU oracle's fp64 GEMMs go through numpy's BLAS: one BLAS thread per
# calling thread, so that the oracle's single-thread and all-core timings use
# exactly the threads they report (the all-core figure runs one oracle
# thread per core; the C oracle and BLAS release the GIL).
for _v in ("OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "MoE W4A4 expert-layer tokens/s"
T, H, F, E, K_TOP = 32768, 2048, 768, 128, 8
WORKLOAD = "moe_expert_layer_32k"
CONFIG = {"workload": WORKLOAD, "tokens": T, "hidden": H, "ffn": F, "experts": E, "topk": K_TOP,
          "router_bias_std": 2.0, "token_expert_rows": T * K_TOP, "weights": "pre-quantized NVFP4, static",
          "l2": "flushed between timed steps (256 MiB write, then a 256 MiB read so no dirty lines remain)",
          "seed": 3}
FLUSH_BYTES = 256 << 20


class L2Flush:
    """Write a buffer larger than L2, then read another one: the next timed
    kernel starts with cold inputs and without dirty lines to write back."""

    def __init__(self, dev):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.sink = self.r.sum()
FP4_OVER_BF16 = 13.5 / 2.25  # nominal dense FP4 : BF16 tensor rate


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--quick", action="store_true", help="profiling runs: no e2e, no oracle, no clocks")
    p.add_argument("--tokens", type=int, choices=[8192, 32768], default=32768,
                   help="--only backward: the layer whose backward is timed (8192: a smaller case for profiling)")
    p.add_argument("--only", choices=["all", "quant", "dequant", "backward"], default="all",
                   help="quant / dequant: time only the 16384 x 2048 quantizer / dequantizer workload; backward: "
                        "only the FC1 backward GEMMs of the 32768-token layer (for profiling)")
    return p.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() and args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available() and args.impl == "ours":
        torch.cuda.set_device(local)
    return rank, world, local


def reduce_max(value, world, device):
    """Max of a float over ranks (identity on one rank)."""
    if world == 1:
        return value
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 20 ms) of SM clock, power and throttle
    reasons while running; each sample keeps its host time, so a summary can
    be taken over one timed window."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_MS = 20

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.PERIOD_MS)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.reader = threading.Thread(target=self._read, daemon=True)
            self.reader.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.monotonic(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=2)

    def summary(self, t0=None, t1=None):
        """Median SM clock, max clock, max power and the throttle reasons seen
        in samples taken in [t0, t1] (host monotonic seconds; all when None)."""
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, ln in self.lines:
            if (t0 is not None and ts < t0) or (t1 is not None and ts > t1):
                continue
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
                pw.append(float(f[3]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(pw), "sample_period_ms": self.PERIOD_MS}


# ---------------------------------------------------------------- workload

def make_inputs():
    d = workloads.moe_32k()
    return d


def recorded_traffic(stage):
    """DRAM bytes per launch of a stage's kernel from the committed ncu record,
    or None when the kernel's sources changed since the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        rec = json.load(f)["kernels"].get(stage)
    if rec is None:
        return None
    h = hashlib.sha256()
    for src in rec["sources"]:
        with open(os.path.join(ROOT, "nvfp4_quantized_moe_token_gb300", src), "rb") as f:
            h.update(f.read())
    if h.hexdigest()[:16] != rec["source_sha256_16"]:
        return None
    return rec["dram_read_bytes"] + rec["dram_write_bytes"]


def algorithmic(T_, R):
    """Per-launch algorithmic work of each stage (bytes or flops) of a layer of
    T_ tokens and R = T_ k token-expert rows."""
    b16, f32 = 2, 4
    q_row = H // 2 + H // 16 + f32
    return {
        # the router top-k runs in the quantize launch (independent work, one launch)
        "quantize": ("hbm", T_ * H * b16 + T_ * q_row + T_ * E * f32 + E * f32 + T_ * K_TOP * 8),
        "route": ("hbm", T_ * q_row + R * q_row + R * 8),
        "fc1": ("tensor", 2.0 * R * (2 * F) * H),
        "requant": ("hbm", R * F * b16 + R * f32 + R * (F // 2 + F // 16 + f32)),
        "fc2": ("tensor", 2.0 * R * H * F),
        "combine": ("hbm", R * H * b16 + T_ * K_TOP * 8 + T_ * H * b16),
    }


def run_e2e(args, nv, d, w1q, w2q, ws, world, dev):
    """Tokens/s end to end through the public call with host buffers: every
    step copies its inputs (X, logits, bias) from pinned host memory to the
    device, runs moe_expert_forward and copies the output back.  Steps are
    pipelined the way a serving or training loop would run them: the inputs
    of step i + 1 are copied in on one copy stream and the output of step
    i - 1 is copied out on another while step i computes (two device buffer
    sets alternate).  The timed region runs from the first input copy to the
    last output copy, so every step's copies are inside it; no L2 flush (the
    step touches well over 1 GB)."""
    xh = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).pin_memory()
    lh = torch.from_numpy(d["logits"]).pin_memory()
    bh = torch.from_numpy(d["bias"]).pin_memory()
    oh = [torch.empty((T, H), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xd = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    ld_ = [torch.empty((T, E), dtype=torch.float32, device=dev) for _ in range(2)]
    bd = [torch.empty((E,), dtype=torch.float32, device=dev) for _ in range(2)]
    od = [torch.empty((T, H), dtype=torch.bfloat16, device=dev) for _ in range(2)]
    comp = torch.cuda.current_stream(dev)
    cin, cout = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    # the layer call of each buffer set, captured once into a CUDA graph (as the
    # headline step is run); the copies stay explicit on their own streams
    for b in range(2):
        xd[b].copy_(xh)
        ld_[b].copy_(lh)
        bd[b].copy_(bh)
        nv.moe_expert_forward(xd[b], ld_[b], bd[b], w1q, w2q, F, K_TOP, out=od[b], ws=ws, stream=comp)
    torch.cuda.synchronize()
    graphs = []
    for b in range(2):
        side = torch.cuda.Stream(dev)
        side.wait_stream(comp)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            nv.moe_expert_forward(xd[b], ld_[b], bd[b], w1q, w2q, F, K_TOP, out=od[b], ws=ws)
        comp.wait_stream(side)
        graphs.append(g)
    torch.cuda.synchronize()

    def run(n):
        in_ready = [torch.cuda.Event() for _ in range(2)]
        done = [None, None]      # compute of the step that last used buffer set b
        copied = [None, None]    # output copy of the step that last used buffer set b
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(cin)
        for i in range(n):
            b = i & 1
            if done[b] is not None:
                cin.wait_event(done[b])
            with torch.cuda.stream(cin):
                xd[b].copy_(xh, non_blocking=True)
                ld_[b].copy_(lh, non_blocking=True)
                bd[b].copy_(bh, non_blocking=True)
            in_ready[b].record(cin)
            comp.wait_event(in_ready[b])
            if copied[b] is not None:
                comp.wait_event(copied[b])
            with torch.cuda.stream(comp):
                graphs[b].replay()
            done[b] = torch.cuda.Event()
            done[b].record(comp)
            cout.wait_event(done[b])
            with torch.cuda.stream(cout):
                oh[b].copy_(od[b], non_blocking=True)
            copied[b] = torch.cuda.Event()
            copied[b].record(cout)
        end.record(cout)
        return start, end

    run(max(args.warmup, 3))
    torch.cuda.synchronize()
    barrier(world)
    start, end = run(args.steps)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = reduce_max(start.elapsed_time(end) / args.steps, world, dev)
    h2d = xh.numel() * 2 + lh.numel() * 4 + bh.numel() * 4
    return {"value": T * world / (e2e_ms / 1e3), "unit": "tokens/s", "ms_per_step": e2e_ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": oh[0].numel() * 2,
            "pipelining": "inputs of step i+1 copied in and output of step i-1 copied out on two copy streams "
                          "while step i computes (the layer call replayed from a CUDA graph per buffer set); "
                          "timed from the first input copy to the last output copy"}


def load_peaks():
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        with open(pk) as f:
            return json.load(f), "measured"
    return {}, "fallback"


class Layer:
    """One expert layer's device inputs, pre-quantized weights, workspace and
    output, and the call that runs it."""

    def __init__(self, nv, dev, d, fc2_requant=None, fc2_combine=False):
        self.nv = nv
        self.d = d
        self.fc2_requant = fc2_requant
        self.fc2_combine = fc2_combine
        self.T = d["x"].shape[0]
        self.x = torch.from_numpy(d["x"].view(np.int16)).view(torch.bfloat16).to(dev)
        self.logits = torch.from_numpy(d["logits"]).to(dev)
        self.bias = torch.from_numpy(d["bias"]).to(dev)
        self.w1q = nv.quantize_grouped_weights(torch.from_numpy(d["w1"].view(np.int16)).view(torch.bfloat16).to(dev))
        self.w2q = nv.quantize_grouped_weights(torch.from_numpy(d["w2"].view(np.int16)).view(torch.bfloat16).to(dev))
        self.ws = torch.zeros(nv.lib().moe_expert_workspace(self.T, H, F, E, K_TOP), dtype=torch.uint8, device=dev)
        self.out = torch.empty((self.T, H), dtype=torch.bfloat16, device=dev)

    def __call__(self, evs=None):
        self.nv.moe_expert_forward(self.x, self.logits, self.bias, self.w1q, self.w2q, F, K_TOP, out=self.out,
                                   ws=self.ws, stage_events=evs, fc2_requant=self.fc2_requant,
                                   fc2_combine=self.fc2_combine)

    def check_error_word(self):
        err = self.ws[:4].view(torch.int32).item()
        if err != 0:
            raise RuntimeError(f"device error word {err:#x}")


def time_layer(layer, steps, warmup, flush, world, dev):
    """Mean step time and per-stage times (library stage events) of `steps`
    steps, L2 flushed before each step outside its events; also returns the
    host-time window of the timed loop."""
    nv = layer.nv
    for _ in range(max(warmup, 3)):
        layer()
    torch.cuda.synchronize()
    layer.check_error_word()
    nev = len(nv.STAGES) + 1
    events = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    torch.cuda.nvtx.range_push("timed")
    for i in range(steps):
        flush()
        layer(events[i])
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    t1 = time.monotonic()
    barrier(world)
    layer.check_error_word()
    step_ms = [ev[0].elapsed_time(ev[-1]) for ev in events]
    stage_ms = {s: [ev[j].elapsed_time(ev[j + 1]) for ev in events] for j, s in enumerate(nv.STAGES)}
    return statistics.fmean(step_ms), stage_ms, (t0, t1), min(step_ms)


def graph_leg(layer, steps, flush):
    """The same step captured once into a CUDA graph and replayed (L2 flushed
    before each replay, outside its events): the layer's eight launches as one
    graph launch, without the per-launch scheduling gaps of eager launches."""
    dev = layer.x.device
    layer()  # first calls made: attributes set and tensor-map encoders found before capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        layer()
    torch.cuda.current_stream(dev).wait_stream(side)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    layer.check_error_word()
    ts = []
    torch.cuda.synchronize()
    t0 = time.monotonic()
    for _ in range(steps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    t1 = time.monotonic()
    layer.check_error_word()
    ms = [a.elapsed_time(b) for a, b in ts]
    del g
    return {"ms_per_step": statistics.fmean(ms), "ms_per_step_min": min(ms),
            "tokens_per_s": layer.T / (statistics.fmean(ms) / 1e3), "steps": steps,
            "how": "one moe_expert_forward call captured in a CUDA graph, replayed; L2 flushed before each replay"}, (t0, t1)


def stage_rooflines(nv, T_, stage_ms, mean_ms, hbm_peak, bf16_peak):
    alg = algorithmic(T_, T_ * K_TOP)
    stages = {}
    for s in nv.STAGES:
        ms = statistics.fmean(stage_ms[s])
        bound, work = alg[s]
        if bound == "tensor":
            ach = work / (ms / 1e3) / 1e12
            peak = bf16_peak * FP4_OVER_BF16
            stages[s] = {"ms": ms, "share": ms / mean_ms, "bound": "tensor", "achieved": ach, "unit": "TFLOP/s",
                         "peak": peak, "frac": ach / peak, "frac_of_9pf": ach / 9000.0,
                         "frac_of_13_5pf": ach / 13500.0}
        else:
            ach = work / (ms / 1e3) / 1e9
            stages[s] = {"ms": ms, "share": ms / mean_ms, "bound": "hbm", "achieved": ach, "unit": "GB/s",
                         "peak": hbm_peak, "frac": ach / hbm_peak}
    gemm_ms = stages["fc1"]["ms"] + stages["fc2"]["ms"]
    gemm_flop = alg["fc1"][1] + alg["fc2"][1]
    gemms = {"ms": gemm_ms, "tflops": gemm_flop / (gemm_ms / 1e3) / 1e12,
             "frac_of_9pf": gemm_flop / (gemm_ms / 1e3) / 1e12 / 9000.0,
             "frac": gemm_flop / (gemm_ms / 1e3) / 1e12 / (bf16_peak * FP4_OVER_BF16)}
    return stages, gemms, alg


def sustained_leg(layer, local, seconds=2.5):
    """The layer back to back (no L2 flush) for about `seconds`, with SM clocks
    sampled inside that loop only: the rate a long run settles at under the
    power cap.  Stage events on every 16th step give the GEMMs' sustained rate."""
    nv = layer.nv
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(20):
        layer()
    b.record()
    torch.cuda.synchronize()
    n = max(int(seconds * 1e3 / (a.elapsed_time(b) / 20)), 100)
    nev = len(nv.STAGES) + 1
    sampled = {i: [torch.cuda.Event(enable_timing=True) for _ in range(nev)] for i in range(0, n, 16)}
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)
    torch.cuda.synchronize()
    t0 = time.monotonic()
    a.record()
    for i in range(n):
        layer(sampled.get(i))
    b.record()
    torch.cuda.synchronize()
    t1 = time.monotonic()
    clocks.stop()
    layer.check_error_word()
    ms = a.elapsed_time(b) / n
    clk = clocks.summary(t0, t1)
    fc = {s: statistics.fmean(ev[j].elapsed_time(ev[j + 1]) for ev in sampled.values())
          for j, s in enumerate(nv.STAGES) if s in ("fc1", "fc2")}
    R = layer.T * K_TOP
    gemm_flop = 2.0 * R * (2 * F) * H + 2.0 * R * H * F
    out = {"seconds": ms * n / 1e3, "steps": n, "ms_per_step": ms, "tokens_per_s": layer.T / (ms / 1e3),
           "fc1_ms": fc["fc1"], "fc2_ms": fc["fc2"],
           "gemm_tflops": gemm_flop / ((fc["fc1"] + fc["fc2"]) / 1e3) / 1e12, "clocks": clk}
    if clk:
        out["ms_x_median_sm_mhz"] = ms * clk["sm_mhz"]
    return out


def run_ours(args, rank, world, local):
    import nvfp4_quantized_moe_token_gb300 as nv
    dev = torch.device("cuda", local)
    peaks, peak_src = load_peaks()
    hbm_peak = peaks.get("hbm_gbs", 6800.0)
    bf16_peak = peaks.get("bf16_tflops", 1900.0)

    d = make_inputs()
    layer = Layer(nv, dev, d)
    flush = L2Flush(dev)
    clocks = ClockSampler(local) if not args.quick else None
    if clocks:
        clocks.start()
        time.sleep(0.3)
    # per-stage times from the library's stage events (eager launches), then the headline
    # step: the same call replayed from a CUDA graph (no stage events inside it)
    eager_ms, stage_ms, _, eager_min = time_layer(layer, args.steps, args.warmup, flush, world, dev)
    barrier(world)
    graph, window = graph_leg(layer, args.steps, flush)
    barrier(world)
    mean_ms, min_ms = graph["ms_per_step"], graph["ms_per_step_min"]
    mean_ms_all = reduce_max(mean_ms, world, dev)

    e2e = None
    if not (args.no_e2e or args.quick):
        e2e = run_e2e(args, nv, d, layer.w1q, layer.w2q, layer.ws, world, dev)
    if clocks:
        clocks.stop()
    clk = clocks.summary() if clocks else None
    if clk:
        inside = clocks.summary(*window)
        clk["timed_region"] = inside if inside else {"samples": 0, "note": "the timed loop ended between samples"}

    stages, gemms, alg = stage_rooflines(nv, T, stage_ms, eager_ms, hbm_peak, bf16_peak)
    dom = max(stages, key=lambda s: stages[s]["ms"])
    dm = stages[dom]
    roofline = {"kernel": dom, "bound": dm["bound"], "achieved": dm["achieved"], "peak": dm["peak"],
                "unit": dm["unit"], "frac": dm["frac"], "traffic": recorded_traffic(dom),
                "peak_source": f"{peak_src} ({'bf16 burst x 6 nominal FP4:BF16' if dm['bound'] == 'tensor' else 'copy GB/s'})",
                "work_per_launch": alg[dom][1]}

    res = {
        "metric": METRIC, "value": T * world / (mean_ms_all / 1e3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_ms_all, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e2m1 x e4m3 -> f32 acc, bf16 io", "data": "synthetic",
        "config": dict(CONFIG, parallelism=f"replicas x{world}"),
        "e2e": e2e, "roofline": roofline, "stages": stages, "gemms_fc1_fc2": gemms,
        "ms_per_step_min": min_ms,
        "step": "one moe_expert_forward call (route -> combine), replayed from a CUDA graph; L2 flushed before "
                "each step outside its events",
        "eager": {"ms_per_step": eager_ms, "ms_per_step_min": eager_min,
                  "tokens_per_s": T * world / (eager_ms / 1e3),
                  "how": "the same call launched eagerly with the library's stage events recorded between its "
                         "launches (the source of `stages`)"},
        "gpu_launches": 8 * args.steps,
        "clocks": clk,
    }
    return res, d, layer


def moe_8k_leg(nv, local, steps, warmup):
    """The 8192-token layer (router bias ~N(0, 1)), timed like the headline one."""
    dev = torch.device("cuda", local)
    peaks, _ = load_peaks()
    layer = Layer(nv, dev, workloads.moe_8k())
    flush = L2Flush(dev)
    eager_ms, stage_ms, _, _ = time_layer(layer, steps, warmup, flush, 1, dev)
    stages, gemms, _ = stage_rooflines(nv, layer.T, stage_ms, eager_ms, peaks.get("hbm_gbs", 6800.0),
                                       peaks.get("bf16_tflops", 1900.0))
    graph, _ = graph_leg(layer, steps, flush)
    del layer
    torch.cuda.empty_cache()
    return {"workload": "moe_expert_layer_8k (8192 tokens, router bias std 1, seed 2)",
            "ms_per_step": graph["ms_per_step"], "ms_per_step_min": graph["ms_per_step_min"],
            "tokens_per_s": 8192 / (graph["ms_per_step"] / 1e3), "steps": steps, "step": graph["how"],
            "eager_ms_per_step": eager_ms, "gemms_fc1_fc2": gemms, "stages": stages}


def fused_option_leg(nv, local, steps, warmup, combine=False):
    """The 32768-token layer with work moved into FC2, options that are off
    by default: the FC2 input requantized inside FC2 (moe_options.fc2_requant
    = MOE_REQUANT_IN_FC2) or, with combine, the router-weighted combine in
    FC2's epilogue (moe_options.fc2_combine).  The same timing as the
    headline, for comparison with the separate launches."""
    dev = torch.device("cuda", local)
    layer = Layer(nv, dev, make_inputs(), fc2_requant=None if combine else "in_fc2", fc2_combine=combine)
    flush = L2Flush(dev)
    eager_ms, stage_ms, _, _ = time_layer(layer, steps, warmup, flush, 1, dev)
    graph, _ = graph_leg(layer, steps, flush)
    del layer
    torch.cuda.empty_cache()
    st = {s: statistics.fmean(v) for s, v in stage_ms.items()}
    what = "combine in FC2's epilogue (GEMM mode 4)" if combine else "FC2 input requantized inside FC2 (GEMM mode 3)"
    return {"workload": "moe_expert_layer_32k, " + what,
            "ms_per_step": graph["ms_per_step"], "tokens_per_s": T / (graph["ms_per_step"] / 1e3),
            "eager_ms_per_step": eager_ms, "fc2_ms": st["fc2"], "stages_ms": st}


def _graph_per_launch(calls, replays, dev):
    """Device time per kernel of `calls` (callables that each enqueue one
    launch on the current stream), captured once into a CUDA graph and
    replayed back to back: the kernels' own rate, without the host-side
    cost of each Python call between them."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        for c in calls:
            c()
    torch.cuda.current_stream(dev).wait_stream(side)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(replays):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / (replays * len(calls))
    del g
    return ms


def quant_gbs(args, local, reps=50, four_over_six=None):
    """Quantizer throughput on the 16384 x 2048 per-token workload, over 4
    rotating copies of the input and outputs (256 MiB of input > L2, so
    every launch reads its rows from DRAM).  Three measurements: the
    launches captured in a CUDA graph and replayed back to back (the
    headline: the kernel's own rate); the same launches issued one Python
    call at a time (adds the host-side cost of each call wherever it exceeds
    the kernel's ~17 us); and single launches with the L2 flushed before
    each (adds the launch and event overhead of one small kernel).
    four_over_six 'mse' / 'mae' times the four-over-six quantizer on the
    same rows."""
    import nvfp4_quantized_moe_token_gb300 as nv
    dev = torch.device("cuda", local)
    xb = workloads.quant_rows()["x"]
    xs = [torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev) for _ in range(4)]
    qs = [nv.NVFP4Tensor.empty(16384, 2048, 16384, dev) for _ in range(4)]
    x, q = xs[0], qs[0]
    flush = L2Flush(dev)
    for _ in range(5):
        for i in range(4):
            nv.quantize_rows(xs[i], out=qs[i], four_over_six=four_over_six)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed_quant")
    groups = []
    for _ in range(max(reps // 4, 3)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(4):
            nv.quantize_rows(xs[i], out=qs[i], four_over_six=four_over_six)
        b.record()
        groups.append((a, b))
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    ms_calls = statistics.fmean(a.elapsed_time(b) for a, b in groups) / 4
    calls = [lambda i=i: nv.quantize_rows(xs[i], out=qs[i], four_over_six=four_over_six) for i in range(4)] * 4
    ms = _graph_per_launch(calls, max(reps // 16, 4), dev)
    ts = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        nv.quantize_rows(x, out=q, four_over_six=four_over_six)
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    ms_single = statistics.fmean(a.elapsed_time(b) for a, b in ts)
    nbytes = 16384 * (2048 * 2 + 1024 + 128 + 4)
    peaks = {}
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        with open(pk) as f:
            peaks = json.load(f)
    hbm = peaks.get("hbm_gbs", 6800.0)
    gbs = nbytes / (ms / 1e3) / 1e9
    out = {"workload": "quantize 16384 x 2048" + ("" if four_over_six is None else f", four-over-six ({four_over_six})"),
           "us": ms * 1e3, "gbs": gbs, "algorithmic_bytes": nbytes, "frac_of_hbm": gbs / hbm, "hbm_peak_gbs": hbm,
           "timing": "launches over 4 rotating input/output copies (256 MiB of input > L2) captured in a CUDA "
                     "graph and replayed back to back, per launch",
           "us_python_calls": ms_calls * 1e3, "frac_of_hbm_python_calls": nbytes / (ms_calls / 1e3) / 1e9 / hbm,
           "us_single_launch_l2_flushed": ms_single * 1e3,
           "frac_of_hbm_single_launch": nbytes / (ms_single / 1e3) / 1e9 / hbm}
    if four_over_six is None:
        out["traffic"] = recorded_traffic("quant")
    del xs, qs
    torch.cuda.empty_cache()
    return out


def dequant_gbs(args, local, reps=50):
    """DQ(Q(x)) throughput: the 16384 x 2048 workload quantized once, then
    dequantized to bf16 over 8 rotating input/output copies (656 MB per
    rotation > L2, so every launch reads its codes from DRAM): launches
    captured in a CUDA graph and replayed back to back (the headline), the
    same launches one Python call at a time, and single launches with the L2
    flushed before each."""
    import nvfp4_quantized_moe_token_gb300 as nv
    dev = torch.device("cuda", local)
    xb = workloads.quant_rows()["x"]
    x = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).to(dev)
    qs = [nv.quantize_rows(x) for _ in range(8)]
    ys = [torch.empty_like(x) for _ in range(8)]
    flush = L2Flush(dev)
    for _ in range(3):
        for i in range(8):
            nv.dequantize_rows(qs[i], out=ys[i])
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_push("timed_dequant")
    groups = []
    for _ in range(max(reps // 8, 3)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(8):
            nv.dequantize_rows(qs[i], out=ys[i])
        b.record()
        groups.append((a, b))
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_pop()
    ms_calls = statistics.fmean(a.elapsed_time(b) for a, b in groups) / 8
    calls = [lambda i=i: nv.dequantize_rows(qs[i], out=ys[i]) for i in range(8)] * 2
    ms = _graph_per_launch(calls, max(reps // 16, 4), dev)
    single = _timed(lambda: nv.dequantize_rows(qs[0], out=ys[0]), reps, flush)
    nbytes = 16384 * (1024 + 128 + 4 + 2048 * 2)  # codes, scales, row scale in; bf16 out
    hbm = 6800.0
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        with open(pk) as f:
            hbm = json.load(f).get("hbm_gbs", hbm)
    gbs = nbytes / (ms / 1e3) / 1e9
    del qs, ys
    torch.cuda.empty_cache()
    return {"workload": "dequantize (DQ(Q(x)) -> bf16) 16384 x 2048", "us": ms * 1e3, "gbs": gbs,
            "algorithmic_bytes": nbytes, "frac_of_hbm": gbs / hbm, "hbm_peak_gbs": hbm,
            "timing": "launches over 8 rotating copies captured in a CUDA graph and replayed back to back, per launch",
            "us_python_calls": ms_calls * 1e3, "us_single_launch_l2_flushed": single * 1e3}


def _timed(fn, reps, flush=None):
    ts = []
    for _ in range(reps):
        if flush is not None:
            flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        ts.append((a, b))
    torch.cuda.synchronize()
    return statistics.fmean(a.elapsed_time(b) for a, b in ts)


def linear_legs(local, bf16_peak, reps=20):
    """The dense W4A4 linear on the attention projections of the same model
    (32768 tokens; QKV 2048 -> 5120, o_proj 4096 -> 2048): per-token
    quantization of the activations plus the block-scaled GEMM, weights
    pre-quantized per tensor (L2 flushed per rep)."""
    import nvfp4_quantized_moe_token_gb300 as nv
    dev = torch.device("cuda", local)
    d = workloads.attn_proj()
    flush = L2Flush(dev)
    out = {}
    for name, xk, wk in (("qkv_proj", "x", "wqkv"), ("o_proj", "o", "wo")):
        x = torch.from_numpy(d[xk].view(np.int16)).view(torch.bfloat16).to(dev)
        w = torch.from_numpy(d[wk].view(np.int16)).view(torch.bfloat16).to(dev)
        M, K = x.shape
        N = w.shape[0]
        wq = nv.quantize_rows(w, per_tensor=True)
        xq = nv.quantize_rows(x)
        y = nv.linear(xq, wq)
        for _ in range(3):
            nv.quantize_rows(x, out=xq)
            nv.linear(xq, wq, out=y)
        torch.cuda.synchronize()
        q_ms = _timed(lambda: nv.quantize_rows(x, out=xq), reps, flush)
        g_ms = _timed(lambda: nv.linear(xq, wq, out=y), reps, flush)
        tf = 2.0 * M * N * K / (g_ms / 1e3) / 1e12
        peak = bf16_peak * FP4_OVER_BF16
        out[name] = {"m": M, "n": N, "k": K, "quantize_us": q_ms * 1e3, "gemm_us": g_ms * 1e3,
                     "step_us": (q_ms + g_ms) * 1e3, "gemm_tflops": tf, "gemm_frac": tf / peak,
                     "gemm_frac_of_9pf": tf / 9000.0, "quantize_gbs": M * (2 * K + K // 2 + K // 16 + 4) / (q_ms / 1e3) / 1e9}
        del x, w, xq, wq, y
    torch.cuda.empty_cache()
    return {"workload": "attention projections, 32768 tokens, per-token NVFP4 X, per-tensor NVFP4 W",
            "tokens_per_s_both": 32768 / ((out["qkv_proj"]["step_us"] + out["o_proj"]["step_us"]) / 1e6),
            "peak_tflops": bf16_peak * FP4_OVER_BF16, **out}


def weight_quantize_leg(local):
    """Per-tensor NVFP4 quantization of the 128 experts' FC1 and FC2 weights
    (off the timed path of the layer: static weights); bytes read + written."""
    import nvfp4_quantized_moe_token_gb300 as nv
    dev = torch.device("cuda", local)
    d = workloads.moe_32k()
    w1 = torch.from_numpy(d["w1"].view(np.int16)).view(torch.bfloat16).to(dev)
    w2 = torch.from_numpy(d["w2"].view(np.int16)).view(torch.bfloat16).to(dev)
    nv.quantize_grouped_weights(w1)
    nv.quantize_grouped_weights(w2)
    torch.cuda.synchronize()
    ms = _timed(lambda: (nv.quantize_grouped_weights(w1), nv.quantize_grouped_weights(w2)), 3)
    n = w1.numel() + w2.numel()
    nbytes = n * 2 * 2 + n // 2 + n // 16  # read twice (tensor amax, then encode), codes + scales written
    del w1, w2
    torch.cuda.empty_cache()
    return {"workload": "128 experts x (W1 1536 x 2048 + W2 2048 x 768), one per-tensor scale per expert matrix "
                        "(nvfp4_quantize_grouped: 3 launches per stack)",
            "ms": ms, "gbs": nbytes / (ms / 1e3) / 1e9}


def backward_leg(layer, local, reps=10):
    """The dequantized BF16 backward of FC1 on the headline layer's own
    operands: x^ = DQ(Q(x)) of the permuted quantized tokens written in the
    128-row-padded layout, w^ = DQ(Q(W1)) of the 128 experts, a synthetic
    gradient dY1 [Rp x 2F] (zero padding rows), then the grouped dgrad
    (dX = dY1 . w^_e) and wgrad (dW1_e = dY1_e^T . x^_e), L2 flushed before
    each launch.  Tensor-bound: FLOPs against the measured bf16 peak."""
    nv = layer.nv
    dev = torch.device("cuda", local)
    peaks, src = load_peaks()
    bf16_peak = peaks.get("bf16_tflops", 1900.0)
    lay = nv.moe_workspace_layout(layer.T, H, F, E, K_TOP)
    ws = layer.ws
    R = layer.T * K_TOP
    off = ws[lay["offsets"]:lay["offsets"] + 4 * (E + 1)].view(torch.int32)
    poff = ws[lay["padded_offsets"]:lay["padded_offsets"] + 4 * (E + 1)].view(torch.int32)
    Rp = int(poff[-1].item())
    a1 = nv.NVFP4Tensor(ws[lay["a1_codes"]:lay["a1_codes"] + R * H // 2].view(R, H // 2),
                        ws[lay["a1_sf"]:lay["a1_sf"] + Rp * H // 16],
                        ws[lay["a1_scale"]:lay["a1_scale"] + 4 * R].view(torch.float32), R, H)
    xh = torch.empty((Rp, H), dtype=torch.bfloat16, device=dev)
    nv.dequantize_rows(a1, group_offsets=off, padded_offsets=poff, out=xh, padded_rows=True)
    gw = torch.arange(0, (E + 1) * 2 * F, 2 * F, dtype=torch.int32, device=dev)
    wh = nv.dequantize_rows(layer.w1q, per_tensor=True, group_offsets=gw, padded_offsets=gw).view(E, 2 * F, H)
    # synthetic upstream gradient: data rows ~N(0, 1e-6), padding rows zero
    pad = torch.ones(Rp, dtype=torch.bool, device=dev)
    offs, poffs = off.long(), poff.long()
    e_of = torch.repeat_interleave(torch.arange(E, device=dev), offs[1:] - offs[:-1])
    prow = poffs[e_of] + (torch.arange(R, device=dev) - offs[e_of])
    pad[prow] = False
    dy = (torch.randn((Rp, 2 * F), device=dev) * 1e-3).to(torch.bfloat16)
    dy[pad] = 0
    dx = torch.empty((Rp, H), dtype=torch.bfloat16, device=dev)
    dw = torch.empty((E, 2 * F, H), dtype=torch.bfloat16, device=dev)
    err = torch.zeros(4, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    for _ in range(2):
        nv.grouped_dgrad_bf16(dy, wh, poff, out=dx, err=err)
        nv.grouped_wgrad_bf16(dy, xh, poff, out=dw, err=err)
    torch.cuda.synchronize()
    if int(err[0].item()) != 0:
        raise RuntimeError(f"backward GEMM error word {int(err[0].item()):#x}")
    dg_ms = _timed(lambda: nv.grouped_dgrad_bf16(dy, wh, poff, out=dx, err=err), reps, flush)
    wg_ms = _timed(lambda: nv.grouped_wgrad_bf16(dy, xh, poff, out=dw, err=err), reps, flush)
    dq_ms = _timed(lambda: nv.dequantize_rows(a1, group_offsets=off, padded_offsets=poff, out=xh, padded_rows=True),
                   reps, flush)
    flop = 2.0 * Rp * (2 * F) * H  # both products: padded rows included (their MMAs run)
    flop_valid = 2.0 * R * (2 * F) * H
    del xh, wh, dx, dw
    # FC2's backward on its own operands: d^ = DQ(Q(D)) of the requantized SwiGLU output (a2) in
    # the padded layout, w2^ = DQ(Q(W2)) per expert, a synthetic dY2 [Rp x H]
    a2 = nv.NVFP4Tensor(ws[lay["a2_codes"]:lay["a2_codes"] + R * F // 2].view(R, F // 2),
                        ws[lay["a2_sf"]:lay["a2_sf"] + Rp * ((F // 16 + 3) // 4 * 4)],
                        ws[lay["a2_scale"]:lay["a2_scale"] + 4 * R].view(torch.float32), R, F)
    dh = torch.empty((Rp, F), dtype=torch.bfloat16, device=dev)
    nv.dequantize_rows(a2, group_offsets=off, padded_offsets=poff, out=dh, padded_rows=True)
    gw2 = torch.arange(0, (E + 1) * H, H, dtype=torch.int32, device=dev)
    wh2 = nv.dequantize_rows(layer.w2q, per_tensor=True, group_offsets=gw2, padded_offsets=gw2).view(E, H, F)
    dy2 = (torch.randn((Rp, H), device=dev) * 1e-3).to(torch.bfloat16)
    dy2[pad] = 0
    dd = torch.empty((Rp, F), dtype=torch.bfloat16, device=dev)
    dw2 = torch.empty((E, H, F), dtype=torch.bfloat16, device=dev)
    nv.grouped_dgrad_bf16(dy2, wh2, poff, out=dd, err=err)
    nv.grouped_wgrad_bf16(dy2, dh, poff, out=dw2, err=err)
    torch.cuda.synchronize()
    if int(err[0].item()) != 0:
        raise RuntimeError(f"backward GEMM error word {int(err[0].item()):#x}")
    dg2_ms = _timed(lambda: nv.grouped_dgrad_bf16(dy2, wh2, poff, out=dd, err=err), reps, flush)
    wg2_ms = _timed(lambda: nv.grouped_wgrad_bf16(dy2, dh, poff, out=dw2, err=err), reps, flush)
    flop2 = 2.0 * Rp * H * F
    fc2 = {"workload": f"FC2 backward: dD [Rp x {F}] = dY2 [Rp x {H}] . w2^_e; dW2_e [{H} x {F}] = dY2_e^T . d^_e",
           "dgrad_us": dg2_ms * 1e3, "wgrad_us": wg2_ms * 1e3,
           "dgrad_tflops": flop2 / (dg2_ms / 1e3) / 1e12, "wgrad_tflops": flop2 / (wg2_ms / 1e3) / 1e12,
           "dgrad_frac": flop2 / (dg2_ms / 1e3) / 1e12 / bf16_peak,
           "wgrad_frac": flop2 / (wg2_ms / 1e3) / 1e12 / bf16_peak}
    del dh, wh2, dy2, dd, dw2
    out = {"workload": f"FC1 backward of the 32768-token layer: dX [Rp x {H}] = dY1 [Rp x {2 * F}] . w^_e; "
                       f"dW1_e [{2 * F} x {H}] = dY1_e^T . x^_e; Rp = {Rp} padded rows ({R} token-expert rows)",
           "dgrad_us": dg_ms * 1e3, "wgrad_us": wg_ms * 1e3, "dequant_x_padded_us": dq_ms * 1e3,
           "dgrad_tflops": flop / (dg_ms / 1e3) / 1e12, "wgrad_tflops": flop / (wg_ms / 1e3) / 1e12,
           "dgrad_frac": flop / (dg_ms / 1e3) / 1e12 / bf16_peak, "wgrad_frac": flop / (wg_ms / 1e3) / 1e12 / bf16_peak,
           "valid_rows_tflops_dgrad": flop_valid / (dg_ms / 1e3) / 1e12,
           "valid_rows_tflops_wgrad": flop_valid / (wg_ms / 1e3) / 1e12,
           "peak_tflops": bf16_peak, "peak_source": f"{src} bf16 burst (cuBLAS)", "fc2": fc2}
    del dy
    torch.cuda.empty_cache()
    return out


def library_fp4_reference(local, reps=20):
    """The library NVFP4 GEMM (torch._scaled_mm on float4_e2m1fn_x2 operands
    with E4M3 16-element block scales, bf16 out) on dense problems of the
    expert layer's two GEMM shapes and at 8192^3: a measured reference for
    the tensor-core ceiling, not part of the path.  None where torch lacks it."""
    dev = torch.device("cuda", local)
    if not hasattr(torch, "float4_e2m1fn_x2"):
        return None
    out = {}
    for name, (M, N, K) in {"fc1_shape_dense": (T * K_TOP, 2 * F, H), "fc2_shape_dense": (T * K_TOP, H, F),
                            "qkv_proj": (32768, 5120, 2048), "o_proj": (32768, 2048, 4096),
                            "square_8192": (8192, 8192, 8192)}.items():
        try:
            a = torch.randint(0, 256, (M, K // 2), dtype=torch.uint8, device=dev).view(torch.float4_e2m1fn_x2)
            b = torch.randint(0, 256, (N, K // 2), dtype=torch.uint8, device=dev).view(torch.float4_e2m1fn_x2)
            sa = torch.ones((M + 127) // 128 * 128 * ((K // 16 + 3) // 4 * 4), device=dev).to(torch.float8_e4m3fn)
            sb = torch.ones((N + 127) // 128 * 128 * ((K // 16 + 3) // 4 * 4), device=dev).to(torch.float8_e4m3fn)
            for _ in range(3):
                torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16)
            s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            s0.record()
            for _ in range(reps):
                torch._scaled_mm(a, b.t(), sa, sb, out_dtype=torch.bfloat16)
            s1.record()
            torch.cuda.synchronize()
            ms = s0.elapsed_time(s1) / reps
            out[name] = {"m": M, "n": N, "k": K, "us": ms * 1e3, "tflops": 2.0 * M * N * K / (ms / 1e3) / 1e12}
            del a, b, sa, sb
        except Exception as ex:  # reported, not retried
            out[name] = {"error": f"{type(ex).__name__}: {str(ex)[:200]}"}
    torch.cuda.empty_cache()
    return {"what": "torch._scaled_mm NVFP4 (cuBLASLt), dense, bf16 out, back-to-back (operands stay in L2 "
                    "only at 8192^3)", "results": out}


# ---------------------------------------------------------------- oracle timing

def oracle_setup(d):
    """Quantize and dequantize the static weights with the oracle (threads:
    the C calls release the GIL)."""
    import concurrent.futures as cf
    import oracle

    def one(e):
        q1 = oracle.quantize(d["w1"][e], per_tensor=True)
        q2 = oracle.quantize(d["w2"][e], per_tensor=True)
        return q1, q2, oracle.dequantize(*q1, per_tensor=True), oracle.dequantize(*q2, per_tensor=True)

    with cf.ThreadPoolExecutor(min(16, os.cpu_count() or 1)) as ex:
        r = list(ex.map(one, range(E)))
    return [x[0] for x in r], [x[1] for x in r], ([x[2] for x in r], [x[3] for x in r])


def oracle_sample_tokens(d, w1q, w2q, wdeq, start, n):
    import oracle
    sl = slice(start, start + n)
    oracle.moe_forward(d["x"][sl], d["logits"][sl], d["bias"], w1q, w2q, K_TOP, w_deq=wdeq)


def cpu_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        r = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for ln in r.stdout.splitlines():
            if ln.strip().startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith(("model name", "cpu part")):
                    return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def oracle_tokens_per_s(d, w1q, w2q, wdeq, threads, budget_s, sample):
    """Tokens/s of the oracle layer over `budget_s` seconds on `threads` host
    threads (one BLAS thread each), each running its own batches of `sample`
    consecutive tokens."""
    import concurrent.futures as cf
    t0 = time.perf_counter()

    def worker(w):
        n, i = 0, 0
        while time.perf_counter() - t0 < budget_s:
            start = ((w * 9973 + i * threads * 7) * sample) % (T - sample)
            oracle_sample_tokens(d, w1q, w2q, wdeq, start, sample)
            n += sample
            i += 1
        return n

    with cf.ThreadPoolExecutor(threads) as ex:
        n_tok = sum(ex.map(worker, range(threads)))
    dt = time.perf_counter() - t0
    return n_tok / dt, n_tok, dt


def cpu_baseline(d, budget_s=8.0, sample=64):
    """The oracle on the host's cores: once on one thread, once on every core
    (one oracle thread per core), BLAS pinned to one thread per caller."""
    w1q, w2q, wdeq = oracle_setup(d)
    n_cores = cpu_threads()
    v1, n1, dt1 = oracle_tokens_per_s(d, w1q, w2q, wdeq, 1, budget_s, sample)
    vn, nn, dtn = oracle_tokens_per_s(d, w1q, w2q, wdeq, n_cores, budget_s, sample)
    return {"value": vn, "unit": "tokens/s", "cores": n_cores, "kind": "oracle",
            "sample": f"{nn} tokens of the 32768-token layer in batches of {sample} consecutive tokens on "
                      f"{n_cores} threads, {dtn:.1f} s (full route/quantize/permute/FC1/SwiGLU/requant/FC2/"
                      f"combine per batch; fp64 GEMMs by numpy BLAS, one BLAS thread per oracle thread; weights "
                      f"quantized and dequantized once)",
            "single_thread": {"value": v1, "unit": "tokens/s", "cores": 1,
                              "sample": f"{n1} tokens in batches of {sample}, {dt1:.1f} s"},
            "cpu_model": cpu_model(), "blas_threads_per_worker": 1}


def cpu_configs():
    """The oracle, single-threaded, on the other workloads: the 64 x 256 x 512
    linear and the 16384 x 2048 quantization in full, the attention
    projections' quantization in full and their fp64 GEMM on a 256-row sample,
    and the 8192-token layer's routing and quantization in full."""
    import oracle
    out = {}
    lin = workloads.linear_small()
    t0 = time.perf_counter()
    oracle.linear(oracle.quantize(lin["x"]), oracle.quantize(lin["w"], per_tensor=True))
    out["linear_64x256x512"] = {"s": time.perf_counter() - t0, "scope": "full"}
    q = workloads.quant_rows()["x"]
    t0 = time.perf_counter()
    oracle.quantize(q)
    dt = time.perf_counter() - t0
    out["quantize_16384x2048"] = {"s": dt, "gbs": 16384 * (2048 * 2 + 1024 + 128 + 4) / dt / 1e9, "scope": "full"}
    del q
    ap = workloads.attn_proj()
    for name, xk, wk in (("qkv_proj", "x", "wqkv"), ("o_proj", "o", "wo")):
        t0 = time.perf_counter()
        xq = oracle.quantize(ap[xk])
        tq = time.perf_counter() - t0
        wq = oracle.quantize(ap[wk], per_tensor=True)
        rows = slice(0, 256)
        t0 = time.perf_counter()
        oracle.linear((xq[0][rows], xq[1][rows], xq[2][rows]), wq)
        tg = time.perf_counter() - t0
        M, K = ap[xk].shape
        N = ap[wk].shape[0]
        out[name] = {"quantize_s_full": tq, "gemm_s_256_rows": tg,
                     "gemm_s_full_extrapolated": tg * M / 256, "gflops": 2.0 * 256 * N * K / tg / 1e9}
    del ap
    m8 = workloads.moe_8k(with_weights=False)
    t0 = time.perf_counter()
    ids, _ = oracle.route(m8["logits"], m8["bias"], K_TOP)
    oracle.route_metadata(ids, E)
    tr = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle.quantize(m8["x"])
    out["moe_8k_route_and_quantize"] = {"route_s": tr, "quantize_s": time.perf_counter() - t0, "scope": "full"}
    return {"threads": 1, "results": out}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import concurrent.futures as cf
    d = make_inputs()
    w1q, w2q, wdeq = oracle_setup(d)
    n_cores = cpu_threads()
    sample = 8  # tokens per oracle thread per step: a step is n_cores x 8 tokens
    for i in range(args.warmup):
        oracle_sample_tokens(d, w1q, w2q, wdeq, i * sample, sample)
    t0 = time.perf_counter()
    with cf.ThreadPoolExecutor(n_cores) as ex:
        for i in range(args.steps):
            list(ex.map(lambda w: oracle_sample_tokens(d, w1q, w2q, wdeq,
                                                       ((i * n_cores + w) * sample * 13) % (T - sample), sample),
                        range(n_cores)))
    dt = time.perf_counter() - t0
    value = args.steps * n_cores * sample / dt
    res = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
           "data": "synthetic", "config": dict(CONFIG, parallelism="host cores"),
           "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": n_cores, "kind": "oracle",
                            "sample": f"each step: {n_cores} oracle threads (one BLAS thread each) x {sample} "
                                      f"tokens of the 32768-token layer (weights quantized once)",
                            "cpu_model": cpu_model()},
           "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(res))


def summary_of(res):
    """The figures a reader looks for first, last on the line (a truncated
    tail of the output still shows them)."""
    st = res["stages"]
    out = {"moe_32k_tokens_per_s": res["value"], "moe_32k_ms": res["ms_per_step"],
           "fc1_ms": st["fc1"]["ms"], "fc2_ms": st["fc2"]["ms"],
           "fc1_plus_fc2_ms": res["gemms_fc1_fc2"]["ms"],
           "fc1_plus_fc2_frac_of_9pf": res["gemms_fc1_fc2"]["frac_of_9pf"]}
    if res.get("e2e"):
        out["e2e_tokens_per_s"] = res["e2e"]["value"]
    if res.get("eager"):
        out["moe_32k_eager_tokens_per_s"] = res["eager"]["tokens_per_s"]
    if res.get("moe_8k"):
        out["moe_8k_tokens_per_s"] = res["moe_8k"]["tokens_per_s"]
        out["moe_8k_fc1_plus_fc2_frac_of_9pf"] = res["moe_8k"]["gemms_fc1_fc2"]["frac_of_9pf"]
    if res.get("requant_in_fc2"):
        out["moe_32k_requant_in_fc2_tokens_per_s"] = res["requant_in_fc2"]["tokens_per_s"]
    if res.get("combine_in_fc2"):
        out["moe_32k_combine_in_fc2_tokens_per_s"] = res["combine_in_fc2"]["tokens_per_s"]
    if res.get("sustained"):
        su = res["sustained"]
        out["sustained_tokens_per_s"] = su["tokens_per_s"]
        out["sustained_sm_mhz"] = (su.get("clocks") or {}).get("sm_mhz")
    if res.get("backward_fc1_bf16"):
        out["bwd_dgrad_frac_of_bf16"] = res["backward_fc1_bf16"]["dgrad_frac"]
        out["bwd_wgrad_frac_of_bf16"] = res["backward_fc1_bf16"]["wgrad_frac"]
    if res.get("quant"):
        out["quant_us"] = res["quant"]["us"]
        out["quant_frac_of_hbm"] = res["quant"]["frac_of_hbm"]
    if res.get("quant_four_over_six"):
        out["quant_46_frac_of_hbm"] = res["quant_four_over_six"]["frac_of_hbm"]
    if res.get("cpu_baseline"):
        out["cpu_oracle_tokens_per_s_all_cores"] = res["cpu_baseline"]["value"]
        out["cpu_oracle_tokens_per_s_1_thread"] = res["cpu_baseline"]["single_thread"]["value"]
    return out


def main():
    args = parse()
    rank, world, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import nvfp4_quantized_moe_token_gb300 as nv
    nv.lib()
    if args.only == "backward":
        if rank == 0:
            d = make_inputs() if args.tokens == 32768 else workloads.moe_8k()
            layer = Layer(nv, torch.device("cuda", local), d)
            layer()
            torch.cuda.synchronize()
            print(json.dumps({"backward_fc1_bf16": backward_leg(layer, local, reps=max(args.steps, 1))}))
        return
    if args.only in ("quant", "dequant"):
        if rank == 0:
            if args.only == "quant":
                out = {"quant": quant_gbs(args, local, reps=max(args.steps, 1)),
                       "quant_four_over_six": quant_gbs(args, local, reps=max(args.steps, 1), four_over_six="mse")}
            else:
                out = {"dequant": dequant_gbs(args, local, reps=max(args.steps, 1))}
            print(json.dumps(out))
        return
    res, d, layer = run_ours(args, rank, world, local)
    if rank == 0:
        if not args.quick:
            res["sustained"] = sustained_leg(layer, local)
            res["backward_fc1_bf16"] = backward_leg(layer, local)
            del layer
            torch.cuda.empty_cache()
            res["moe_8k"] = moe_8k_leg(nv, local, args.steps, args.warmup)
            res["requant_in_fc2"] = fused_option_leg(nv, local, args.steps, args.warmup)
            res["combine_in_fc2"] = fused_option_leg(nv, local, args.steps, args.warmup, combine=True)
            res["quant"] = quant_gbs(args, local)
            res["quant_four_over_six"] = quant_gbs(args, local, four_over_six="mse")
            res["dequant"] = dequant_gbs(args, local)
            res["linear_attention_projections"] = linear_legs(local, res["roofline"]["peak"] / FP4_OVER_BF16)
            res["weight_quantize"] = weight_quantize_leg(local)
            res["library_fp4_reference"] = library_fp4_reference(local)
        if not (args.no_cpu_baseline or args.quick):
            res["cpu_baseline"] = cpu_baseline(d)
            res["cpu_oracle_configs"] = cpu_configs()
        if not args.quick:
            res["summary"] = summary_of(res)
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
