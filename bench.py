#!/usr/bin/env python
"""Benchmark of the verify step (one JSON line on stdout).

A step is one spec_verify call over one batch of the workload.  The default
workload is the greedy blockwise-parallel verify of 64 sequences x 8 draft
positions over a 32000-token bf16 vocabulary; ``--workload`` picks another of
the seeded workloads (draft_verify_acceptance_gb300.workloads.WORKLOADS).

Device timing: the inputs are resident in HBM as R rotating copies whose total
exceeds twice the L2 size, so every step reads its logits from DRAM; K steps
are captured in CUDA graphs and timed with CUDA events on the launching
stream, bracketed by barrier + synchronize.  The metric is verified draft
positions per second (B*K per step, summed over ranks) over the max time of
all ranks.  ``e2e`` times the public call with pinned HOST tensors (copies
host->device, the kernel, device->host of the outputs, per step).

``--impl reference`` times the CPU oracle on the machine's host cores instead
(rank 0 only) on the same workload and metric.
"""
import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "greedy_bf16_B64_K8_V32000"
METRIC = "verified draft positions/sec (B*K/s)"
UNIT = "positions/s"
FALLBACK_HBM_GBS = 6800.0
REF_BUDGET_S = 150.0  # the reference arm's timed CPU work


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the per-workload table and the CPU baseline")
    ap.add_argument("--line", default=None,
                    help="time one contrastive-verify or rejection-cut workload alone "
                         "(--steps launches) and print its line")
    return ap.parse_args()


# --------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no collective on the data path)
# --------------------------------------------------------------------------
def dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    """The largest value of x over all ranks (timing is taken as the max)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_seed(base_seed, rank):
    """Each rank verifies its own independent batch (weak scaling)."""
    return base_seed + 1000 * rank


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self._stop = threading.Event()
        self._thr = None

    def _run(self):
        try:
            p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                                  "--format=csv,noheader,nounits", "-lms", "100"],
                                 stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            return
        try:
            for line in p.stdout:
                self.samples.append((time.perf_counter(), line.strip()))
                if self._stop.is_set():
                    break
        finally:
            p.kill()
            p.wait()

    def start(self):
        self._thr = threading.Thread(target=self._run, daemon=True)
        self._thr.start()
        time.sleep(0.3)

    def stop(self, t0, t1):
        self._stop.set()
        self._thr.join(timeout=3)
        rows = [s for (t, s) in self.samples if t0 <= t <= t1] or [s for _, s in self.samples[-3:]]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# measured peaks and committed ncu traffic
# --------------------------------------------------------------------------
def hbm_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# The sources each kernel is built from (a committed ncu figure stays valid
# while these hash the same).
KERNEL_SOURCES = {
    "greedy_kernel": ["verify_greedy.cu", "device_common.cuh", "launch.h"],
    "fused_sample_kernel": ["verify_sample_fused.cu", "sample_common.cuh", "device_common.cuh",
                            "launch.h"],
    "norm_stream_kernel": ["verify_sample_2p.cu", "sample_common.cuh", "device_common.cuh",
                           "launch.h"],
    "sample_kernel": ["verify_sample.cu", "sample_common.cuh", "device_common.cuh", "launch.h"],
    "cut_warp_kernel": ["rejection_cut.cu", "launch.h"],
    "scd_row_kernel": ["verify_scd.cu", "sample_common.cuh", "device_common.cuh", "launch.h"],
}


def strip_comments(src):
    """C/C++ source without its comments (string and character literals kept),
    so that editing a comment leaves a kernel's hash unchanged."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":  # a literal: copy it through, escapes included
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "".join(out)


def kernel_source_hash(kernel, read=None):
    """Hash of the sources a kernel is built from, comments and layout left
    out.  `read(name)` gives a file's text (default: the working tree)."""
    d = os.path.join(ROOT, "draft_verify_acceptance_gb300", "csrc")
    if read is None:
        def read(f):
            with open(os.path.join(d, f), encoding="utf-8") as fh:
                return fh.read()
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        code = " ".join(strip_comments(read(f)).split())  # whitespace runs as one space
        h.update(f.encode() + code.encode())
    return h.hexdigest()[:16]


def kernel_plan(inp):
    """(dominant kernel, kernel launches per verify call) for these inputs: the
    library's dispatch (src: launch_greedy / launch_sample) restated --
    greedy: one greedy_kernel; sampling with 16-byte aligned rows of at most
    4096 vectors: one fused_sample_kernel; longer aligned rows (up to the
    two-kernel sampler's limit): norm_stream_kernel then
    decide_sample_kernel; otherwise the streaming sample_kernel."""
    from draft_verify_acceptance_gb300 import workloads as W
    if inp.mode == W.MODE_GREEDY:
        return "greedy_kernel", 1
    esz = 2 if inp.dtype_name == "bf16" else 4
    if (inp.V * esz) % 16 != 0:
        return "sample_kernel", 1
    nvec = inp.V * esz // 16
    if nvec <= 4096:
        return "fused_sample_kernel", 1
    return "norm_stream_kernel", 2


def committed_traffic(workload, kernel):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, only
    if it was taken on that kernel's current sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("kernel") != kernel or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------
# native arm
# --------------------------------------------------------------------------
def device_time(binding, inp, steps, warmup, dev, l2_bytes, mode=None):
    """Prepare `steps` launches that rotate over R device copies of the inputs
    (R * bytes > 2x L2), warm up, and capture them in CUDA graphs.  Returns
    (R, algorithmic bytes per launch, stream, graphs to replay, two events,
    the output tensors).  `mode` overrides the inputs' mode (early exit)."""
    import torch
    mode = inp.mode if mode is None else mode
    nbytes = inp.algorithmic_bytes()
    R = max(2, math.ceil(2 * l2_bytes / max(nbytes, 1)) + 1)
    R = min(R, 64)
    copies = []
    for r in range(R):
        copies.append(tuple(None if t is None else t.to(dev) for t in
                            (inp.target, inp.draft, inp.tokens, inp.uniforms)))
    acc = torch.empty(inp.B, dtype=torch.int32, device=dev)
    out = torch.empty((inp.B, inp.K + 1), dtype=torch.int32, device=dev)
    dt = binding.DTYPE_BF16 if inp.target.dtype == torch.bfloat16 else binding.DTYPE_F32
    ws = torch.zeros(binding.workspace_size(inp.B, inp.K, inp.V, dt, inp.mode),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)

    def launch(r):
        c = copies[r % R]
        binding.verify(c[0], c[1], c[2], c[3], inp.temperature, mode, stream=stream,
                       workspace=ws, out=(acc, out))

    with torch.cuda.stream(stream):
        for w in range(max(warmup, 3)):
            launch(w)
    stream.synchronize()
    G = min(steps, 1000)
    graphs = []
    for n in sorted({G, steps % G} - {0}):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(n):
                launch(k)
        graphs.append((n, g))
    plan = [graphs[-1][1]] * (steps // G) if G else []
    if steps % G:
        plan.append([g for n, g in graphs if n == steps % G][0])
    # one untimed replay of each graph
    with torch.cuda.stream(stream):
        for _, g in graphs:
            g.replay()
    torch.cuda.synchronize(dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    return R, nbytes, stream, plan, e0, e1, (acc, out)


def run_native(args, rank, world, local):
    import torch
    from draft_verify_acceptance_gb300 import binding, workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2**20)
    inp = W.workload(args.workload, seed=shard_seed(0, rank))
    R, nbytes, stream, plan, e0, e1, acc_out = device_time(binding, inp, args.steps, args.warmup,
                                                           dev, l2)
    acc_out[0].fill_(-1)

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):  # graphs replay on the current stream
        e0.record(stream)
        for g in plan:
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    barrier(world)
    # the replayed graphs wrote real outputs (guards against timing an empty graph)
    n_host = acc_out[0].cpu()
    if not (int(n_host.min()) >= 0 and int(n_host.max()) <= inp.K):
        raise RuntimeError("timed launches did not produce valid outputs")
    clk = clocks.stop(t0, t1) if rank == 0 else None
    sec = e0.elapsed_time(e1) / 1e3
    sec_max = max_over_ranks(sec, world)

    positions = inp.B * inp.K
    value = positions * world * args.steps / sec_max
    per_launch = sec / args.steps
    peak, peak_kind = hbm_peak()
    achieved = nbytes / per_launch / 1e9

    # end to end through the public call with pinned host tensors
    e2e_steps = max(20, min(args.steps, 500))
    host = [None if t is None else t.pin_memory() for t in
            (inp.target, inp.draft, inp.tokens, inp.uniforms)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            binding.verify(*host, inp.temperature, inp.mode, stream=stream)
        barrier(world)
        h0 = time.perf_counter()
        for _ in range(e2e_steps):
            binding.verify(*host, inp.temperature, inp.mode, stream=stream)
        h1 = time.perf_counter()
    e2e_sec = max_over_ranks(h1 - h0, world)
    h2d = sum(t.numel() * t.element_size() for t in host if t is not None)
    d2h = inp.B * 4 + inp.B * (inp.K + 1) * 4

    extras = None
    cpu = None
    if rank == 0 and world == 1 and not args.no_extras:
        extras = per_workload_table(binding, args.workload, dev, l2, peak)
        cpu = cpu_baseline(inp)

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": sec_max * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded torch CPU generator; recipe in draft_verify_acceptance_gb300/workloads.py)",
        "config": {"workload": args.workload, "B": inp.B, "K": inp.K, "V": inp.V,
                   "logits_dtype": inp.dtype_name,
                   "mode": "greedy" if inp.mode == W.MODE_GREEDY else "sample",
                   "temperature": inp.temperature if inp.mode == W.MODE_SAMPLE else None,
                   "parallelism": f"replicas x{world}",
                   "l2": f"{R} rotating input copies of {nbytes / 1e6:.1f} MB (> 2x L2 of "
                         f"{l2 / 2**20:.0f} MiB)",
                   "timing": "CUDA graphs of <=1000 launches, CUDA events on the launch stream"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_kind": peak_kind,
                     "traffic": committed_traffic(args.workload, kernel_plan(inp)[0]),
                     "algorithmic_bytes_per_launch": nbytes,
                     "kernel": kernel_plan(inp)[0]},
        "e2e": {"value": positions * world * e2e_steps / e2e_sec, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "path": "binding.verify on pinned host tensors (H2D, kernel, D2H, sync)"},
        "gpu_launches": args.steps * kernel_plan(inp)[1],
        "clocks": clk,
        "cpu_baseline": cpu,
        "workloads": extras,
    }
    print(json.dumps(line))


def per_workload_table(binding, skip, dev, l2, peak, steps=3000):
    """Device throughput of every other workload (same timing method)."""
    import torch
    from draft_verify_acceptance_gb300 import workloads as W
    table = {}
    for name in W.WORKLOADS:
        if name == skip:
            continue
        inp = W.workload(name)
        R, nbytes, stream, plan, e0, e1, _ = device_time(binding, inp, steps, 5, dev, l2)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for g in plan:
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize(dev)
        sec = e0.elapsed_time(e1) / 1e3 / steps
        table[name] = {"us_per_step": sec * 1e6, "positions_per_s": inp.B * inp.K / sec,
                       "GB_per_s": nbytes / sec / 1e9, "frac_hbm": nbytes / sec / 1e9 / peak,
                       "algorithmic_bytes": nbytes}
        del plan
        torch.cuda.empty_cache()
        if inp.mode == W.MODE_SAMPLE and inp.K > 0:
            table[name + "+early_exit"] = early_exit_line(binding, inp, steps, dev, l2, peak, sec)
            table[name + "+draft_sample"] = draft_sample_line(binding, inp, steps, dev, l2, peak)
    for name, spec in W.SCD_WORKLOADS.items():
        table[name] = scd_line(binding, name, spec, steps, dev, l2, peak)
    for name, spec in W.REJECTION_WORKLOADS.items():
        table[name] = rejection_cut_line(binding, name, spec, steps, dev, l2, peak)
    return table


def scd_line(binding, name, spec, steps, dev, l2, peak):
    """Speculative contrastive decoding's verify step (bytes: every expert
    and amateur row read once, the tokens, the uniforms and the outputs),
    graph-replayed over rotating input copies > 2x L2 like the rest."""
    import torch
    from draft_verify_acceptance_gb300 import workloads as W
    spec = dict(spec)
    alpha = spec.pop("alpha")
    inp = W.make_scd_inputs(seed=0, name=name, **spec)
    B, K, V = inp.B, inp.K, inp.V
    es = inp.target.element_size()
    nbytes = 2 * B * (K + 1) * V * es + B * K * 4 + B * (K + 1) * 4 + B * 4 + B * (K + 1) * 4
    R = min(64, max(2, math.ceil(2 * l2 / max(nbytes, 1)) + 1))
    copies = [tuple(t.to(dev) for t in (inp.target, inp.draft, inp.tokens, inp.uniforms))
              for _ in range(R)]
    dt = binding.DTYPE_BF16 if inp.target.dtype == torch.bfloat16 else binding.DTYPE_F32
    ws = torch.zeros(binding.workspace_size(B, K, V, dt, binding.MODE_SAMPLE), dtype=torch.uint8,
                     device=dev)
    out = (torch.empty(B, dtype=torch.int32, device=dev),
           torch.empty((B, K + 1), dtype=torch.int32, device=dev))
    stream = torch.cuda.Stream(dev)

    def launch(k):
        c = copies[k % R]
        binding.verify_scd(c[0], c[1], c[2], c[3], inp.temperature, alpha, stream=stream,
                           workspace=ws, out=out)

    with torch.cuda.stream(stream):
        for r in range(3):
            launch(r)
        stream.synchronize()
        n = min(steps, 1000)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(n):
                launch(k)
        g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    sec = e0.elapsed_time(e1) / 1e3 / n
    mean_n = float(out[0].float().mean().item())
    del g, copies
    torch.cuda.empty_cache()
    return {"us_per_step": sec * 1e6, "positions_per_s": B * K / sec, "bytes": nbytes,
            "GB_per_s": nbytes / sec / 1e9, "frac_hbm": nbytes / sec / 1e9 / peak,
            "kernel": "scd_row_kernel", "mean_accepted_len": mean_n,
            "traffic": committed_traffic(inp.name, "scd_row_kernel")}


def rejection_cut_line(binding, name, spec, steps, dev, l2, peak):
    """Speculative Rejection's cut over G prompts of N scores (bytes: the
    scores read, the kept-index rows, r_cut and the counts written),
    graph-replayed over rotating score copies > 2x L2; the oracle's time on
    the same batch beside it."""
    import torch
    from draft_verify_acceptance_gb300 import workloads as W
    G, N, alpha = spec["G"], spec["N"], spec["alpha"]
    scores = W.make_scores(G, N, kind=spec["kind"], seed=0)
    nbytes = G * N * 4 * 2 + G * (8 + 4)
    R = min(64, max(2, math.ceil(2 * l2 / max(nbytes, 1)) + 1))
    copies = [scores.to(dev) for _ in range(R)]
    out = (torch.empty(G, dtype=torch.float64, device=dev),
           torch.empty(G, dtype=torch.int32, device=dev),
           torch.empty((G, N), dtype=torch.int32, device=dev))
    stream = torch.cuda.Stream(dev)
    with torch.cuda.stream(stream):
        for r in range(3):
            binding.rejection_cut(copies[r % R], alpha, stream=stream, out=out)
        stream.synchronize()
        n = min(steps, 1000)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(n):
                binding.rejection_cut(copies[k % R], alpha, stream=stream, out=out)
        g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    sec = e0.elapsed_time(e1) / 1e3 / n
    del g, copies
    torch.cuda.empty_cache()
    import oracle
    t0 = time.perf_counter()
    oracle.rejection_cut_ref(scores.numpy(), alpha)
    cpu_sec = time.perf_counter() - t0
    return {"us_per_step": sec * 1e6, "scores_per_s": G * N / sec, "bytes": nbytes,
            "GB_per_s": nbytes / sec / 1e9, "frac_hbm": nbytes / sec / 1e9 / peak,
            "kernel": "cut_warp_kernel" if N <= 1024 else "cut_block_kernel",
            "traffic": committed_traffic(name, "cut_warp_kernel") if N <= 1024 else None,
            "cpu_baseline": {"value": G * N / cpu_sec, "unit": "scores/s",
                             "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"the whole batch ({G} x {N}), once"}}


def draft_sample_line(binding, inp, steps, dev, l2, peak):
    """The drafter's sampling step over the workload's B*K draft rows (one
    uniform each), graph-replayed over rotating copies > 2x L2 like the rest."""
    import torch
    s = inp.draft.element_size()
    nbytes = inp.B * inp.K * inp.V * s + inp.B * inp.K * 4 * 3
    R = min(64, max(2, math.ceil(2 * l2 / max(nbytes, 1)) + 1))
    copies = [inp.draft.to(dev) for _ in range(R)]
    u = inp.uniforms[:, :inp.K].contiguous().to(dev)
    dt = binding.DTYPE_BF16 if inp.draft.dtype == torch.bfloat16 else binding.DTYPE_F32
    ws = torch.zeros(binding.workspace_size(inp.B * inp.K, 0, inp.V, dt, binding.MODE_SAMPLE),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    out = (torch.empty(u.shape, dtype=torch.int32, device=dev),
           torch.empty(u.shape, dtype=torch.float32, device=dev))
    with torch.cuda.stream(stream):
        for r in range(3):
            binding.draft_sample(copies[r % R], u, inp.temperature, stream=stream, workspace=ws,
                                 out=out)
        stream.synchronize()
        n = min(steps, 1000)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for k in range(n):
                binding.draft_sample(copies[k % R], u, inp.temperature, stream=stream, workspace=ws,
                                     out=out)
        g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    sec = e0.elapsed_time(e1) / 1e3 / n
    del g, copies
    torch.cuda.empty_cache()
    return {"us_per_step": sec * 1e6, "rows_per_s": inp.B * inp.K / sec, "bytes": nbytes,
            "GB_per_s": nbytes / sec / 1e9, "frac_hbm": nbytes / sec / 1e9 / peak}


def early_exit_line(binding, inp, steps, dev, l2, peak, parallel_sec):
    """The same workload in early-exit mode (position 0 first).  Bytes read:
    position 0's row pairs, plus every row when some sequence accepted x_0
    (then the full verify runs too); the outputs equal sampling mode's."""
    import torch
    R, nbytes, stream, plan, e0, e1, (acc, _) = device_time(
        binding, inp, steps, 5, dev, l2, mode=binding.MODE_SAMPLE_EARLY_EXIT)
    torch.cuda.synchronize(dev)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for g in plan:
            g.replay()
        e1.record(stream)
    torch.cuda.synchronize(dev)
    sec = e0.elapsed_time(e1) / 1e3 / steps
    s = inp.target.element_size()
    first = 2 * inp.B * inp.V * s + inp.B * 4 + inp.B * 4 + inp.B * (inp.K + 2) * 4
    full_ran = bool((acc > 0).any().item())  # the last replayed call's outputs
    read = first + (nbytes if full_ran else 0)
    del plan
    torch.cuda.empty_cache()
    return {"us_per_step": sec * 1e6, "positions_per_s": inp.B * inp.K / sec,
            "bytes_read": read, "GB_per_s": read / sec / 1e9, "frac_hbm": read / sec / 1e9 / peak,
            "full_verify_ran": full_ran, "speedup_vs_sampling_mode": parallel_sec / sec}


def cpu_baseline(inp, budget_s=10.0):
    """The oracle as it stands, on the host cores, over repetitions of the
    workload's batch until about `budget_s` seconds have passed."""
    import oracle
    from draft_verify_acceptance_gb300 import workloads as W
    t = W.as_numpy_logits(inp.target)
    d = W.as_numpy_logits(inp.draft)
    x = inp.tokens.numpy()
    u = None if inp.uniforms is None else inp.uniforms.numpy()
    B = inp.B
    # a bounded sample: the first b sequences, doubled until one call takes >= 0.5 s
    b = max(1, min(B, 4))
    while True:
        t0 = time.perf_counter()
        oracle.verify_ref(t[:b], None if d is None else d[:b], x[:b], None if u is None else u[:b],
                          inp.temperature, inp.mode)
        dt = time.perf_counter() - t0
        if dt >= 0.5 or b == B:
            break
        b = min(B, b * 2)
    reps, total, t0 = 0, 0.0, time.perf_counter()
    while total < budget_s:
        oracle.verify_ref(t[:b], None if d is None else d[:b], x[:b], None if u is None else u[:b],
                          inp.temperature, inp.mode)
        reps += 1
        total = time.perf_counter() - t0
    return {"value": b * inp.K * reps / total, "unit": UNIT, "cores": oracle.max_threads(),
            "kind": "oracle",
            "sample": f"first {b} of {B} sequences, {reps} repetitions, {total:.1f} s"}


# --------------------------------------------------------------------------
# reference arm: the CPU oracle on the host cores
# --------------------------------------------------------------------------
def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    from draft_verify_acceptance_gb300 import workloads as W
    inp = W.workload(args.workload)
    t = W.as_numpy_logits(inp.target)
    d = W.as_numpy_logits(inp.draft)
    x = inp.tokens.numpy()
    u = None if inp.uniforms is None else inp.uniforms.numpy()

    def step(b):
        oracle.verify_ref(t[:b], None if d is None else d[:b], x[:b],
                          None if u is None else u[:b], inp.temperature, inp.mode)

    # each step: a sample of the first b sequences, b as large as lets all
    # --steps steps finish within REF_BUDGET_S (b >= 1; with b = 1 and a very
    # large --steps the count is cut to what the budget holds, and the line
    # reports the steps actually timed)
    def step_time(bb, reps=3):
        t0 = time.perf_counter()
        for _ in range(reps):
            step(bb)
        return (time.perf_counter() - t0) / reps

    K = max(args.steps, 1)
    b, tb = 1, step_time(1)
    while b < inp.B:
        nb = min(inp.B, b * 2)
        tn = step_time(nb)
        if tn * K > REF_BUDGET_S:
            break
        b, tb = nb, tn
    steps = K if tb * K <= REF_BUDGET_S else max(1, int(REF_BUDGET_S / tb))
    for _ in range(max(args.warmup, 1)):
        step(b)
    t0 = time.perf_counter()
    for _ in range(steps):
        step(b)
    sec = time.perf_counter() - t0
    value = b * inp.K * steps / sec
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": steps, "warmup": args.warmup, "ms_per_step": sec * 1e3 / steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": args.workload, "B": inp.B, "K": inp.K,
                                        "V": inp.V},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": oracle.max_threads(),
                         "kind": "oracle", "sample": f"first {b} of {inp.B} sequences per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_line(args):
    """One line of the per-workload table on its own (for profiling runs)."""
    import torch
    from draft_verify_acceptance_gb300 import binding, workloads as W
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 126 * 2**20)
    peak, _ = hbm_peak()
    if args.line in W.SCD_WORKLOADS:
        res = scd_line(binding, args.line, W.SCD_WORKLOADS[args.line], args.steps, dev, l2, peak)
    elif args.line in W.REJECTION_WORKLOADS:
        res = rejection_cut_line(binding, args.line, W.REJECTION_WORKLOADS[args.line], args.steps,
                                 dev, l2, peak)
    else:
        raise SystemExit(f"unknown line {args.line!r}")
    print(json.dumps({"line": args.line, **res}))


def main():
    args = parse()
    if args.line:
        run_line(args)
        return
    rank, world, local = dist_init(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_native(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
