#!/usr/bin/env python
"""Benchmark of the verify step (one JSON line on stdout).

A step is one spec_verify call over one batch of the workload.  The default
workload is the largest one: the best-of-N-scale sampling verify of 1024
candidate sequences x 4 draft positions over a 32000-token bf16 vocabulary
(590 MB of logits per call); ``--workload`` picks another of the seeded
workloads (draft_verify_acceptance_gb300.workloads.WORKLOADS).  Every other
workload gets a complete line of its own under "workloads".

Device timing: the inputs are resident in HBM as R rotating copies whose total
exceeds twice the L2 size, so every step reads its logits from DRAM; K steps
are captured in CUDA graphs and timed with CUDA events on the launching
stream, bracketed by barrier + synchronize; one untimed replay is enqueued
just before the start event so the graphs' launch latency is not timed.  The
metric is verified draft positions per second (B*K per step, summed over
ranks) over the max time of all ranks.  ``e2e`` times the public call with pinned HOST tensors (copies
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

DEFAULT_WORKLOAD = "best_of_n_bf16_B1024_K4_V32000"
METRIC = "verified draft positions/sec (B*K/s)"
UNIT = "positions/s"
FALLBACK_HBM_GBS = 6800.0
REF_BUDGET_S = 150.0  # the reference arm's timed CPU work


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the per-workload table and the CPU baseline")
    ap.add_argument("--line", default=None,
                    help="time one contrastive-verify, rejection-cut, <workload>+draft_sample or "
                         "<workload>+early_exit line alone "
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
    "seq_sample_kernel": ["verify_sample_seq.cu", "sample_common.cuh", "device_common.cuh",
                          "launch.h"],
    "cut_warp_kernel": ["rejection_cut.cu", "launch.h"],
    "scd_row_kernel": ["verify_scd.cu", "sample_common.cuh", "device_common.cuh", "launch.h"],
    "row_sample_kernel": ["verify_draft_sample.cu", "sample_common.cuh", "device_common.cuh",
                          "launch.h"],
    "ee_cluster_kernel": ["verify_sample_ee.cu", "sample_common.cuh", "device_common.cuh",
                          "launch.h", "launch_ee.h"],
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
    greedy: one greedy_kernel; sampling with 16-byte aligned rows: at most
    one sequence per SM (152) whose 2K+1 rows fit 192 KiB: one
    seq_sample_kernel; else rows of at most 4096 vectors: one
    fused_sample_kernel; longer rows: norm_stream_kernel then
    decide_sample_kernel; unaligned rows: the streaming sample_kernel."""
    from draft_verify_acceptance_gb300 import workloads as W
    if inp.mode == W.MODE_GREEDY:
        return "greedy_kernel", 1
    esz = 2 if inp.dtype_name == "bf16" else 4
    if (inp.V * esz) % 16 != 0:
        return "sample_kernel", 1
    nvec = inp.V * esz // 16
    if inp.B <= 152 and (2 * inp.K + 1) * nvec * 16 <= 192 * 1024:
        return "seq_sample_kernel", 1
    if nvec <= 4096:
        return "fused_sample_kernel", 1
    return "norm_stream_kernel", 2


def committed_traffic(workload, kernel, key="dram_bytes_per_launch"):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, only
    if it was taken on that kernel's current sources (`key`
    "call_dram_bytes": all kernels of one verify call)."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("kernel") != kernel or e.get("source_hash") != kernel_source_hash(kernel):
        return None
    return e.get(key)


# --------------------------------------------------------------------------
# native arm
# --------------------------------------------------------------------------
def rotating_copies(nbytes, l2_bytes):
    """How many input copies a timed loop rotates over so that every launch
    reads its inputs from DRAM: their total exceeds twice the L2 size."""
    return min(64, max(2, math.ceil(2 * l2_bytes / max(nbytes, 1)) + 1))


class GraphTimer:
    """`steps` calls of `launch(k)` captured in CUDA graphs of at most 1000
    launches each, replayed on `stream` and timed there with CUDA events.

    Every run first enqueues one untimed replay, then the start event, the
    timed graphs and the stop event: the timed graphs are submitted while the
    GPU is still busy with the untimed replay, so the start event fires when
    that replay ends and the graphs' launch latency stays outside the
    measured interval, whatever `steps` is."""

    def __init__(self, launch, steps, warmup, stream, dev):
        import torch
        self.stream, self.dev, self.steps = stream, dev, steps
        with torch.cuda.stream(stream):
            for w in range(max(warmup, 3)):
                launch(w)
        stream.synchronize()
        G = min(steps, 1000)
        graphs = {}
        for n in sorted({G, steps % G} - {0}):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for k in range(n):
                    launch(k)
            graphs[n] = g
        self.graphs = graphs
        self.plan = [graphs[G]] * (steps // G) + ([graphs[steps % G]] if steps % G else [])
        self.warm = graphs[G]
        with torch.cuda.stream(stream):  # one untimed replay of each graph
            for g in graphs.values():
                g.replay()
        torch.cuda.synchronize(dev)
        self.e0 = torch.cuda.Event(enable_timing=True)
        self.e1 = torch.cuda.Event(enable_timing=True)

    def run(self, before_start=None):
        """Enqueue the untimed replay, `before_start()` (work that must run
        after it but outside the timed interval), the start event, the timed
        graphs and the stop event; the caller synchronizes."""
        import torch
        with torch.cuda.stream(self.stream):
            self.warm.replay()
            if before_start is not None:
                before_start()
            self.e0.record(self.stream)
            for g in self.plan:
                g.replay()
            self.e1.record(self.stream)

    def seconds(self):
        return self.e0.elapsed_time(self.e1) / 1e3

    def per_launch(self):
        import torch
        torch.cuda.synchronize(self.dev)
        self.run()
        torch.cuda.synchronize(self.dev)
        return self.seconds() / self.steps


def device_setup(binding, inp, dev, l2_bytes, mode=None):
    """R rotating device copies of the inputs (R * bytes > 2x L2), the outputs,
    a zero-filled workspace, a stream, and launch(k): one verify call on copy
    k mod R.  `mode` overrides the inputs' mode (early exit)."""
    import torch
    mode = inp.mode if mode is None else mode
    R = rotating_copies(inp.algorithmic_bytes(), l2_bytes)
    copies = [tuple(None if t is None else t.to(dev) for t in
                    (inp.target, inp.draft, inp.tokens, inp.uniforms)) for _ in range(R)]
    acc = torch.empty(inp.B, dtype=torch.int32, device=dev)
    out = torch.empty((inp.B, inp.K + 1), dtype=torch.int32, device=dev)
    dt = binding.DTYPE_BF16 if inp.target.dtype == torch.bfloat16 else binding.DTYPE_F32
    ws = torch.zeros(binding.workspace_size(inp.B, inp.K, inp.V, dt, mode), dtype=torch.uint8,
                     device=dev)
    stream = torch.cuda.Stream(dev)

    def launch(k):
        c = copies[k % R]
        binding.verify(c[0], c[1], c[2], c[3], inp.temperature, mode, stream=stream,
                       workspace=ws, out=(acc, out))

    return R, stream, launch, (acc, out)


def roofline(inp, nbytes, sec_per_call, peak, peak_kind, workload):
    kernel, launches = kernel_plan(inp)
    achieved = nbytes / sec_per_call / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_kind": peak_kind,
            "traffic": committed_traffic(workload, kernel),
            "call_traffic": committed_traffic(workload, kernel, key="call_dram_bytes"),
            "algorithmic_bytes_per_launch": nbytes, "kernel": kernel,
            "kernels_per_call": launches}


def e2e_record(binding, inp, stream, world, steps):
    """The public call on pinned HOST tensors: every step copies the inputs
    host -> device, verifies, and copies the outputs back (the binding
    synchronizes the stream before returning)."""
    import torch
    host = [None if t is None else t.pin_memory() for t in
            (inp.target, inp.draft, inp.tokens, inp.uniforms)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            binding.verify(*host, inp.temperature, inp.mode, stream=stream)
        barrier(world)
        h0 = time.perf_counter()
        for _ in range(steps):
            binding.verify(*host, inp.temperature, inp.mode, stream=stream)
        h1 = time.perf_counter()
    sec = max_over_ranks(h1 - h0, world)
    h2d = sum(t.numel() * t.element_size() for t in host if t is not None)
    d2h = inp.B * 4 + inp.B * (inp.K + 1) * 4
    return {"value": inp.B * inp.K * world * steps / sec, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "path": "binding.verify on pinned host tensors (H2D, kernel, D2H, sync)"}


def parity_record(binding, inp, dev):
    """One spec_verify_ex call on the whole batch against the oracle on the
    same input bytes: how many sequences are bit-equal, how many each
    boundary category excludes (the oracle's flags in double: the ratio
    band, the CDF band, a residual mass below the band; and the kernel's own
    flags), the largest error of p_i(x_i) and q_i(x_i), the mean accepted
    length and the empirical acceptance rate of each draft position."""
    import numpy as np
    import torch
    import oracle
    from draft_verify_acceptance_gb300 import workloads as W
    mv = lambda t: None if t is None else t.to(dev)
    res = binding.verify_ex(mv(inp.target), mv(inp.draft), mv(inp.tokens), mv(inp.uniforms),
                            inp.temperature, inp.mode)
    torch.cuda.synchronize(dev)
    ref = oracle.verify_ref(W.as_numpy_logits(inp.target), W.as_numpy_logits(inp.draft),
                            inp.tokens.numpy(), None if inp.uniforms is None else inp.uniforms.numpy(),
                            inp.temperature, inp.mode, want_debug=True)
    n = res["accepted_len"].cpu().numpy()
    out = res["out_tokens"].cpu().numpy()
    fl = ref["flags"]
    ok = fl == 0
    equal = (n == ref["accepted_len"]) & (out == ref["out_tokens"]).all(1)
    rec = {"sequences": int(inp.B), "compared": int(ok.sum()),
           "bit_equal": int((equal & ok).sum()), "mismatched": int((~equal & ok).sum()),
           "flagged": {"ratio_band": int(((fl & oracle.FLAG_RATIO) != 0).sum()),
                       "cdf_band": int(((fl & oracle.FLAG_CDF) != 0).sum()),
                       "tiny_residual": int(((fl & oracle.FLAG_TINY_RESIDUAL) != 0).sum()),
                       "any": int((~ok).sum()),
                       "flagged_but_equal": int((equal & ~ok).sum())},
           "kernel_flagged": int((res["flags"].cpu().numpy() != 0).sum()),
           "status": int(res["status"].item()), "oracle_status": int(ref["status"])}
    if inp.mode == W.MODE_SAMPLE and inp.K > 0:
        rec["p_at_max_abs_err"] = float(np.abs(res["p_at"].cpu().numpy() - ref["p_at"]).max())
        rec["q_at_max_abs_err"] = float(np.abs(res["q_at"].cpu().numpy() - ref["q_at"]).max())
        rec["tolerance"] = 2e-3 if inp.dtype_name == "bf16" else 1e-5
    per_pos = []
    for i in range(inp.K):
        reached = int((n >= i).sum())
        per_pos.append(round(float((n > i).sum()) / reached, 4) if reached else None)
    acc = {"mean_accepted_len": float(n.mean()) if n.size else 0.0, "per_position": per_pos}
    return rec, acc


def cpu_baselines(inp, budget_s):
    """The oracle as it stands on all host cores and on one core."""
    import oracle
    allc = cpu_baseline(inp, budget_s)
    nmax = oracle.max_threads()
    oracle.set_threads(1)
    try:
        one = cpu_baseline(inp, budget_s)
    finally:
        oracle.set_threads(nmax)
    allc["single_core"] = {"value": one["value"], "cores": 1, "sample": one["sample"]}
    return allc


def run_native(args, rank, world, local):
    import torch
    from draft_verify_acceptance_gb300 import binding, workloads as W

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2**20)
    inp = W.workload(args.workload, seed=shard_seed(0, rank))
    nbytes = inp.algorithmic_bytes()
    R, stream, launch, (acc, out) = device_setup(binding, inp, dev, l2)
    timer = GraphTimer(launch, args.steps, args.warmup, stream, dev)

    clocks = ClockSampler(local)
    if rank == 0:
        clocks.start()
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    # the outputs are cleared after the untimed replay, so the check below
    # sees what the timed graphs wrote
    timer.run(before_start=lambda: acc.fill_(-1))
    torch.cuda.synchronize(dev)
    t1 = time.perf_counter()
    barrier(world)
    n_host = acc.cpu()
    if not (int(n_host.min()) >= 0 and int(n_host.max()) <= inp.K):
        raise RuntimeError("timed launches did not produce valid outputs")
    clk = clocks.stop(t0, t1) if rank == 0 else None
    sec = timer.seconds()
    sec_max = max_over_ranks(sec, world)
    del timer, launch
    torch.cuda.empty_cache()

    positions = inp.B * inp.K
    value = positions * world * args.steps / sec_max
    peak, peak_kind = hbm_peak()
    e2e = e2e_record(binding, inp, stream, world, max(20, min(args.steps, 200)))

    extras = cpu = parity = accept = None
    if rank == 0 and world == 1 and not args.no_extras:
        parity, accept = parity_record(binding, inp, dev)
        cpu = cpu_baselines(inp, 5.0)
        extras = per_workload_table(binding, args.workload, dev, l2, peak, peak_kind)

    if rank != 0:
        return
    kernel, launches = kernel_plan(inp)
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
                   "timing": "CUDA graphs of <=1000 launches after one untimed replay, "
                             "CUDA events on the launch stream"},
        "roofline": roofline(inp, nbytes, sec_max / args.steps, peak, peak_kind, args.workload),
        "e2e": e2e,
        "gpu_launches": args.steps * launches,
        "clocks": clk,
        "cpu_baseline": cpu,
        "parity": parity,
        "acceptance": accept,
        "workloads": extras,
    }
    print(json.dumps(line))


def workload_record(binding, inp, dev, l2, peak, peak_kind, steps=500, cpu_budget=3.0):
    """The complete line of one seeded workload: device time per call
    (graph-replayed, inputs rotating over copies > 2x L2), its roofline, the
    end-to-end figure, the oracle at all cores and at one core, and the
    parity and acceptance record."""
    import torch
    R, stream, launch, _ = device_setup(binding, inp, dev, l2)
    sec = GraphTimer(launch, steps, 5, stream, dev).per_launch()
    del launch
    torch.cuda.empty_cache()
    nbytes = inp.algorithmic_bytes()
    rec = {"us_per_step": sec * 1e6, "positions_per_s": inp.B * inp.K / sec,
           "roofline": roofline(inp, nbytes, sec, peak, peak_kind, inp.name),
           "e2e": e2e_record(binding, inp, stream, 1, 20)}
    rec["parity"], rec["acceptance"] = parity_record(binding, inp, dev)
    rec["cpu_baseline"] = cpu_baselines(inp, cpu_budget)
    return rec, sec


def per_workload_table(binding, skip, dev, l2, peak, peak_kind, steps=500):
    """A complete line for every other workload, and the variant lines
    (early exit, draft sampler, contrastive verify, rejection cut)."""
    import torch
    from draft_verify_acceptance_gb300 import workloads as W
    table = {}
    for name in W.WORKLOADS:
        inp = W.workload(name)
        if name != skip:
            table[name], sec = workload_record(binding, inp, dev, l2, peak, peak_kind, steps)
        else:
            R, stream, launch, _ = device_setup(binding, inp, dev, l2)
            sec = GraphTimer(launch, steps, 5, stream, dev).per_launch()
            del launch
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
    graph-replayed over rotating input copies > 2x L2 like the rest; the
    oracle's time on a sample of the batch beside it."""
    import numpy as np
    import torch
    import oracle
    from draft_verify_acceptance_gb300 import workloads as W
    spec = dict(spec)
    alpha = spec.pop("alpha")
    inp = W.make_scd_inputs(seed=0, name=name, **spec)
    B, K, V = inp.B, inp.K, inp.V
    es = inp.target.element_size()
    nbytes = 2 * B * (K + 1) * V * es + B * K * 4 + B * (K + 1) * 4 + B * 4 + B * (K + 1) * 4
    R = rotating_copies(nbytes, l2)
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

    sec = GraphTimer(launch, steps, 3, stream, dev).per_launch()
    mean_n = float(out[0].float().mean().item())
    del launch, copies
    torch.cuda.empty_cache()
    # parity of the last call's batch against the oracle, and the oracle's time
    t = W.as_numpy_logits(inp.target)
    a = W.as_numpy_logits(inp.draft)
    c0 = time.perf_counter()
    ref = oracle.scd_verify_ref(t, a, inp.tokens.numpy(), inp.uniforms.numpy(), inp.temperature,
                                alpha, want_debug=True)
    cpu_sec = time.perf_counter() - c0
    ok = ref["flags"] == 0
    n = out[0].cpu().numpy()
    o = out[1].cpu().numpy()
    equal = (n == ref["accepted_len"]) & (o == ref["out_tokens"]).all(1)
    achieved = nbytes / sec / 1e9
    return {"us_per_step": sec * 1e6, "positions_per_s": B * K / sec,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "algorithmic_bytes_per_launch": nbytes,
                         "kernel": "scd_row_kernel",
                         "traffic": committed_traffic(inp.name, "scd_row_kernel")},
            "mean_accepted_len": mean_n,
            "parity": {"sequences": B, "compared": int(ok.sum()),
                       "bit_equal": int((equal & ok).sum()),
                       "mismatched": int((~equal & ok).sum()), "flagged": int((~ok).sum())},
            "cpu_baseline": {"value": B * K / cpu_sec, "unit": UNIT,
                             "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"the whole batch ({B} sequences), once"}}


def rejection_cut_line(binding, name, spec, steps, dev, l2, peak):
    """Speculative Rejection's cut over G prompts of N scores (bytes: the
    scores read, the kept-index rows, r_cut and the counts written),
    graph-replayed over rotating score copies > 2x L2; the oracle's time on
    the same batch beside it."""
    import numpy as np
    import torch
    import oracle
    from draft_verify_acceptance_gb300 import workloads as W
    G, N, alpha = spec["G"], spec["N"], spec["alpha"]
    scores = W.make_scores(G, N, kind=spec["kind"], seed=0)
    nbytes = G * N * 4 * 2 + G * (8 + 4)
    R = rotating_copies(nbytes, l2)
    copies = [scores.to(dev) for _ in range(R)]
    out = (torch.empty(G, dtype=torch.float64, device=dev),
           torch.empty(G, dtype=torch.int32, device=dev),
           torch.empty((G, N), dtype=torch.int32, device=dev))
    stream = torch.cuda.Stream(dev)

    def launch(k):
        binding.rejection_cut(copies[k % R], alpha, stream=stream, out=out)

    sec = GraphTimer(launch, steps, 3, stream, dev).per_launch()
    del launch, copies
    torch.cuda.empty_cache()
    t0 = time.perf_counter()
    ref = oracle.rejection_cut_ref(scores.numpy(), alpha)
    cpu_sec = time.perf_counter() - t0
    same = (np.array_equal(out[0].cpu().numpy(), ref["r_cut"])
            and np.array_equal(out[1].cpu().numpy(), ref["n_accepted"])
            and np.array_equal(out[2].cpu().numpy(), ref["accepted"]))
    kernel = "cut_warp_kernel" if N <= 1024 else "cut_block_kernel"
    achieved = nbytes / sec / 1e9
    return {"us_per_step": sec * 1e6, "scores_per_s": G * N / sec,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "algorithmic_bytes_per_launch": nbytes,
                         "kernel": kernel,
                         "traffic": committed_traffic(name, kernel)},
            "parity": {"prompts": G, "bit_equal": bool(same)},
            "cpu_baseline": {"value": G * N / cpu_sec, "unit": "scores/s",
                             "cores": oracle.max_threads(), "kind": "oracle",
                             "sample": f"the whole batch ({G} x {N}), once"}}


def draft_sample_line(binding, inp, steps, dev, l2, peak):
    """The drafter's sampling step over the workload's B*K draft rows (one
    uniform each), graph-replayed over rotating copies > 2x L2 like the rest."""
    import torch
    s = inp.draft.element_size()
    nbytes = inp.B * inp.K * inp.V * s + inp.B * inp.K * 4 * 3
    R = rotating_copies(nbytes, l2)
    copies = [inp.draft.to(dev) for _ in range(R)]
    u = inp.uniforms[:, :inp.K].contiguous().to(dev)
    dt = binding.DTYPE_BF16 if inp.draft.dtype == torch.bfloat16 else binding.DTYPE_F32
    ws = torch.zeros(binding.workspace_size(inp.B * inp.K, 0, inp.V, dt, binding.MODE_SAMPLE),
                     dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    out = (torch.empty(u.shape, dtype=torch.int32, device=dev),
           torch.empty(u.shape, dtype=torch.float32, device=dev))

    def launch(k):
        binding.draft_sample(copies[k % R], u, inp.temperature, stream=stream, workspace=ws,
                             out=out)

    sec = GraphTimer(launch, steps, 3, stream, dev).per_launch()
    del launch, copies
    torch.cuda.empty_cache()
    achieved = nbytes / sec / 1e9
    row_bytes = inp.V * s
    kernel = "row_sample_kernel" if row_bytes % 16 == 0 and row_bytes <= 8 * 96 * 1024 else None
    return {"us_per_step": sec * 1e6, "rows_per_s": inp.B * inp.K / sec, "bytes": nbytes,
            "GB_per_s": achieved, "frac_hbm": achieved / peak,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "algorithmic_bytes_per_launch": nbytes,
                         "kernel": kernel,
                         "traffic": committed_traffic(inp.name + "+draft_sample", kernel)
                         if kernel else None}}


def ee_cluster_size(nvec):
    """The early-exit kernel's cluster size for rows of nvec 16-byte vectors
    (src: ee_cluster, verify_sample_ee.cu restated): the smallest C in
    {1, 2, 4, 8} whose two slices and lane checkpoints fit 200 KiB; 0 if none."""
    for C in (1, 2, 4, 8):
        nvs = (nvec + C - 1) // C
        steps = ((nvs + 15) // 16 + 31) // 32
        if 2 * nvs * 16 + (steps + 3) // 4 * 16 * 32 * 8 <= 200 * 1024:
            return C
    return 0


def early_exit_schedule(inp, sm_count=152):
    """The library's early-exit dispatch restated (src: launch_sample):
    "small_batch" (one CTA per sequence, every row read), "cluster" (one
    cluster per sequence walking the positions), or "two_phase"."""
    nvec = inp.V * inp.target.element_size() // 16
    if inp.B <= sm_count and (2 * inp.K + 1) * nvec * 16 <= 192 * 1024:
        return "small_batch"
    return "cluster" if ee_cluster_size(nvec) > 0 else "two_phase"


def early_exit_line(binding, inp, steps, dev, l2, peak, parallel_sec):
    """The same workload in early-exit mode; the outputs equal sampling
    mode's.  Bytes read, by schedule: the small-batch kernel reads every
    row; the cluster kernel the row pairs of positions 0..n of each sequence
    (the bonus row instead of a pair at n = K); the two-phase schedule
    position 0's row pairs, plus every row when some sequence accepted x_0."""
    import torch
    R, stream, launch, (acc, _) = device_setup(binding, inp, dev, l2,
                                               mode=binding.MODE_SAMPLE_EARLY_EXIT)
    sec = GraphTimer(launch, steps, 5, stream, dev).per_launch()
    s = inp.target.element_size()
    small = inp.B * inp.K * 4 + inp.B * 4 + inp.B * (inp.K + 2) * 4  # tokens, u, outputs
    n = acc.cpu().long()  # the last replayed call's outputs
    schedule = early_exit_schedule(inp, torch.cuda.get_device_properties(dev).multi_processor_count)
    if schedule == "small_batch":
        read = inp.algorithmic_bytes()
        full_ran = True
    elif schedule == "cluster":
        rows = torch.where(n < inp.K, 2 * (n + 1), 2 * inp.K + 1)
        read = int(rows.sum().item()) * inp.V * s + small
        full_ran = False
    else:
        full_ran = bool((n > 0).any().item())
        read = 2 * inp.B * inp.V * s + small + (inp.algorithmic_bytes() if full_ran else 0)
    del launch
    torch.cuda.empty_cache()
    kernel = "ee_cluster_kernel" if schedule == "cluster" else None
    return {"us_per_step": sec * 1e6, "positions_per_s": inp.B * inp.K / sec, "schedule": schedule,
            "bytes_read": read, "GB_per_s": read / sec / 1e9, "frac_hbm": read / sec / 1e9 / peak,
            "full_verify_ran": full_ran, "speedup_vs_sampling_mode": parallel_sec / sec,
            "roofline": {"bound": "hbm", "achieved": read / sec / 1e9, "peak": peak, "unit": "GB/s",
                         "frac": read / sec / 1e9 / peak, "algorithmic_bytes_per_launch": read,
                         "kernel": kernel,
                         "traffic": committed_traffic(inp.name + "+early_exit", kernel)
                         if kernel else None}}


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
    # a bounded sample: the first b sequences, doubled until one call takes
    # >= budget_s / 20
    b = max(1, min(B, 4))
    while True:
        t0 = time.perf_counter()
        oracle.verify_ref(t[:b], None if d is None else d[:b], x[:b], None if u is None else u[:b],
                          inp.temperature, inp.mode)
        dt = time.perf_counter() - t0
        if dt >= budget_s / 20 or b == B:
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
    elif args.line.endswith("+draft_sample") and args.line[:-len("+draft_sample")] in W.WORKLOADS:
        inp = W.workload(args.line[:-len("+draft_sample")])
        res = draft_sample_line(binding, inp, args.steps, dev, l2, peak)
    elif args.line.endswith("+early_exit") and args.line[:-len("+early_exit")] in W.WORKLOADS:
        inp = W.workload(args.line[:-len("+early_exit")])
        R, stream, launch, _ = device_setup(binding, inp, dev, l2)
        sec = GraphTimer(launch, args.steps, 5, stream, dev).per_launch()
        del launch
        res = early_exit_line(binding, inp, args.steps, dev, l2, peak, sec)
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
