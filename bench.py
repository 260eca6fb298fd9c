"""Benchmark of the GB300 FlashAttention-2 forward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload page|tiny|slice|varlen|sweep_d128_n8192|...]

One step is one forward pass (one kernel launch) over the whole batch of the
workload: by default the page workload B16 N4096 H16 d128, bf16 inputs in
[batch, seq, heads, d_head] layout drawn N(0,1) from a fixed seed.  Inputs
(805 MB) and the output (268 MB) are larger than L2, so no flush is needed
between steps.

value      TFLOP/s = 4*B*H*N^2*d / (device time per step), inputs resident in HBM,
           summed over ranks (each rank runs its own replica of the workload;
           the forward has no exchange step, so scaling is weak).
e2e        the same metric through the public call with host buffers: each step
           copies q, k, v from pinned host memory, runs the forward and copies
           O and LSE back, all inside the timed region; the copies of
           neighbouring steps overlap the compute (two copy streams, two device
           buffer sets), as a serving loop would run them.
roofline   the kernel's achieved TFLOP/s (algorithmic FLOPs / launch time,
           CUDA events on the launch stream) against the measured bf16 peak.
cpu_baseline  the fp64 CPU oracle (test infrastructure) timed on a bounded
           sample of the same workload on this host's cores (rank 0, N=1).

--impl reference times that oracle as the reference arm (the pages ship no
implementation; the oracle is the reference), printing the same JSON line.
--fp8 times the e4m3 forward (fa_fwd_fp8, or fa_fwd_fp8_varlen on the packed
workload) on the workload quantised once
beforehand (block scales; the quantisation is not timed), against the fp8
dense peak taken as twice the measured bf16 one (the nominal ratio).
--bwd times the backward pass instead (fa_bwd / fa_bwd_varlen, d = 64 or 128: preprocessing, key-block kernel,
dQ conversion), FLOPs counted as 2.5x the forward's (five matrix products
against two).  Rank 0 prints one JSON line on stdout.
"""
from __future__ import annotations

import argparse
import copy
import ctypes
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

METRIC = "attention fwd TFLOP/s (bf16, B16 N4096 H16 d128) and % of GB300 bf16 peak"
UNIT = "TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")
KERNEL_SOURCES = ("attention_forward_fa2_gb300/csrc/fa_fwd_kernel.cuh",
                  "attention_forward_fa2_gb300/csrc/ptx.cuh")


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def code_text(src: str) -> str:
    """C/C++ source without its comments, whitespace runs collapsed: the part
    of a source file that decides the compiled code (string and character
    literals are kept as they are)."""
    out, i, n = [], 0, len(src)
    while i < n:
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif src[i] in "\"'":
            q, j = src[i], i + 1
            while j < n and src[j] != q:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(src[i])
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash() -> str:
    """Hash of the forward kernel's code (comments and layout excluded), the
    key under which profiles/traffic.json stores the measured DRAM bytes."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_text(f.read()).encode("utf-8"))
        h.update(b"\0")
    return h.hexdigest()[:16]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def load_traffic(workload: str):
    """Per-launch DRAM bytes from a committed ncu summary, if it was taken on
    the current kernel source for this workload."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    entry = t.get(workload)
    if not entry or entry.get("kernel_source_hash") != kernel_source_hash():
        return None
    return entry.get("bytes_per_launch")


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu = gpu  # nvidia-smi -i accepts an index or a UUID
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        sm, smax, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
                power.append(float(parts[3]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        loaded = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w_max": max(power) if power else None}


# -------------------------------------------------------------- distributed
def dist_setup(n_gpus: int, backend: str = "nccl"):
    """(rank, local rank, world size) from the launcher's environment; joins
    the process group when there is more than one rank.  The benchmark's
    ranks use NCCL, one GPU each; "gloo" serves the CPU tests of this logic."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if n_gpus > 1 and world != n_gpus:
        raise SystemExit("--gpus %d needs torchrun with %d processes (WORLD_SIZE=%d)" % (n_gpus, n_gpus, world))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        import torch
        if backend == "nccl":
            torch.cuda.set_device(local)
            dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        else:
            dist.init_process_group(backend)
    return rank, local, world


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest of the ranks' values (every rank gets it): a job is as
    slow as its slowest rank."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------- oracle timing
class OracleSample:
    """A bounded sample of workload `w` for the fp64 oracle: one batch,
    min(threads, H) heads, the full key length, and as many query rows as fit
    `budget_s` seconds on `threads` host threads (calibrated once)."""

    def __init__(self, w, budget_s: float, threads: int):
        import oracle
        from attention_forward_fa2_gb300 import inputs as I
        self.oracle = oracle
        oracle.set_num_threads(threads)
        self.threads = threads
        H = max(1, min(threads, w.H))
        Nk = max(w.lengths) if w.varlen else w.Nk
        d = w.d
        q, k, v = I.make_dense(1, 8, Nk, H, d, seed=w.seed + 1000)
        self.kb, self.vb = I.bf16_bits(k), I.bf16_bits(v)
        t0 = time.perf_counter()
        oracle.attn_dense(I.bf16_bits(q), self.kb, self.vb)
        t_cal = max(time.perf_counter() - t0, 1e-4)
        nq_max = max(w.lengths) if w.varlen else w.Nq
        nq = int(max(1, min(nq_max, 8 * budget_s / t_cal)))
        q, _, _ = I.make_dense(1, nq, 1, H, d, seed=w.seed + 2000)
        self.qb = I.bf16_bits(q)
        self.flops = 4.0 * H * nq * Nk * d
        self.desc = ("fp64 oracle (S and P materialised) on 1 batch x %d heads x %d queries x %d keys, "
                     "d=%d, a bounded sample of the %s workload; %d threads" % (H, nq, Nk, d, w.name, threads))

    def run(self) -> float:
        t0 = time.perf_counter()
        self.oracle.attn_dense(self.qb, self.kb, self.vb)
        return time.perf_counter() - t0


class OracleFull:
    """The fp64 oracle over the whole workload once (every batch and head, the
    full query and key lengths): the CPU baseline of the page workload."""

    def __init__(self, w, threads: int, causal: bool = False):
        import oracle
        from attention_forward_fa2_gb300 import inputs as I
        self.oracle = oracle
        oracle.set_num_threads(threads)
        self.w, self.causal = w, causal
        q, k, v, cu_q, cu_k = I.make(w)
        self.qb, self.kb, self.vb = I.bf16_bits(q), I.bf16_bits(k), I.bf16_bits(v)
        self.cu = (cu_q.numpy(), cu_k.numpy()) if w.varlen else None
        self.flops = w.flops(causal=causal)
        self.desc = ("fp64 oracle (S and P materialised) on the whole %s workload (%s%s), timed once; "
                     "%d threads" % (w.name, w.note, ", causal" if causal else "", threads))

    def run(self) -> float:
        t0 = time.perf_counter()
        if self.cu is not None:
            self.oracle.attn_varlen(self.qb, self.kb, self.vb, self.cu[0], self.cu[1], max(self.w.lengths),
                                    causal=self.causal)
        else:
            self.oracle.attn_dense(self.qb, self.kb, self.vb, causal=self.causal)
        return time.perf_counter() - t0


def cpu_baseline(args, w):
    """The oracle timed on this host's cores: the whole workload once for the
    page workload (about a minute on 16 cores), a bounded sample otherwise or
    with --cpu-baseline sample."""
    mode = args.cpu_baseline
    if mode == "auto":
        mode = "full" if w.name == "page" else "sample"
    cores = host_cores()
    if mode == "full":
        ref = OracleFull(w, cores, causal=args.causal)
        dt = ref.run()
        return {"value": ref.flops / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample": ref.desc, "coverage": "full workload", "seconds": dt}
    sample = OracleSample(w, args.cpu_seconds, cores)
    dt = sample.run()
    return {"value": sample.flops / dt / 1e12, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": sample.desc, "coverage": "sample", "seconds": dt}


# --------------------------------------------------------------------- arms
def run_reference(args, w):
    rank, world = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    cores = host_cores()
    budget = max(0.5, min(5.0, 120.0 / max(1, args.steps + args.warmup)))
    sample = OracleSample(w, budget, cores)
    for _ in range(args.warmup):
        sample.run()
    times = [sample.run() for _ in range(args.steps)]
    total = sum(times)
    value = sample.flops * len(times) / total / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1), generated on the host)",
        "config": workload_config(w, getattr(args, "causal", False)),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample.desc},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    return 0


E2E_COPIES = ("every step copies its inputs in and its results out; the copies of neighbouring steps "
              "overlap its compute (two copy streams, two device buffer sets)")


def pipelined_e2e(torch, dev, stream, sets, host_in, host_out, run, steps, world):
    """Milliseconds per end-to-end step with the copies of neighbouring steps
    overlapped: step i's inputs go host -> device on one copy stream while
    step i-1 computes on `stream` and step i-2's results go device -> host on
    a second copy stream.  Two device buffer sets alternate; events order each
    set's reuse (inputs after the compute two steps back has read them,
    outputs after their copy out).  sets[s] = (device inputs, device outputs),
    host_in the pinned inputs (every step copies all of them), host_out[s] the
    pinned outputs of set s, run(s) launches one step on `stream` for set s."""
    cs_in, cs_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def one(i):
        s = i % 2
        with torch.cuda.stream(cs_in):
            if i >= 2:
                cs_in.wait_event(ev_comp[s])
            for d_, h_ in zip(sets[s][0], host_in):
                d_.copy_(h_, non_blocking=True)
            ev_in[s].record(cs_in)
        stream.wait_event(ev_in[s])
        if i >= 2:
            stream.wait_event(ev_out[s])
        run(s)
        ev_comp[s].record(stream)
        with torch.cuda.stream(cs_out):
            cs_out.wait_event(ev_comp[s])
            for h_, d_ in zip(host_out[s], sets[s][1]):
                h_.copy_(d_, non_blocking=True)
            ev_out[s].record(cs_out)

    for i in range(2):
        one(i)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    cs_in.wait_event(e0)
    for i in range(2, 2 + steps):
        one(i)
    e1.record(cs_out)  # the last copy out is the last work of the region
    torch.cuda.synchronize(dev)
    barrier(world)
    return e0.elapsed_time(e1) / steps


def copy_gbs(torch, dev, dsts, srcs):
    """GB/s of copying srcs into dsts (one copy each, on a side stream), best of three."""
    cs = torch.cuda.Stream(device=dev)
    nbytes = sum(t.numel() * t.element_size() for t in srcs)
    best = float("inf")
    for _ in range(3):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(cs):
            a.record(cs)
            for d_, s_ in zip(dsts, srcs):
                d_.copy_(s_, non_blocking=True)
            b.record(cs)
        torch.cuda.synchronize(dev)
        best = min(best, a.elapsed_time(b))
    return nbytes / (best * 1e-3) / 1e9 if best > 0 else None


def per_step_stats(marks):
    """Median, minimum and maximum of the per-step device times (ms) from
    events recorded between the timed steps (empty for a graph replay)."""
    if len(marks) < 2:
        return None
    t = sorted(a.elapsed_time(b) for a, b in zip(marks[:-1], marks[1:]))
    return {"median": statistics.median(t), "min": t[0], "max": t[-1]}


def workload_config(w, causal=False):
    """The workload a line measures (the same dict on both arms)."""
    cfg = {"workload": "%s: %s" % (w.name, w.note or ""), "B": w.B, "H": w.H, "d": w.d,
           "layout": "[batch, seq, heads, d_head] bf16", "causal": bool(causal),
           "l2": "inputs and output larger than L2 (no flush needed)",
           "parallelism": "replicas (one full workload per GPU, no collective)"}
    if w.varlen:
        cfg["sequences"] = len(w.lengths)
        cfg["total_tokens"] = sum(w.lengths)
        cfg["max_seqlen"] = max(w.lengths)
    else:
        cfg["Nq"] = w.Nq
        cfg["Nk"] = w.Nk
    return cfg


def kernel_info(w, args, kernel_cfg):
    """How our arm ran the workload: entry point, launch mode, tile config."""
    k = {"launch": "cuda graph replay" if args.graph else "stream launches", "form": "fa_fwd (bf16)"}
    if kernel_cfg:
        k["config"] = kernel_cfg
    if args.split:
        k["form"] = "key-split (fa_fwd_splitkv)"
    if getattr(args, "fp8", False):
        k["form"] = "fp8 e4m3, block-quantised (fa_fwd_fp8%s)" % ("_varlen" if w.varlen else "")
    return k


def run_ours(args, w):
    import torch
    import attention_forward_fa2_gb300 as fa
    from attention_forward_fa2_gb300 import build as fabuild
    from attention_forward_fa2_gb300 import inputs as I

    rank, local, world = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    fabuild.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)

    q, k, v, cu_q, cu_k = I.make(w)
    maxlen = max(w.lengths) if w.varlen else None
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    dcu = cu_q.to(dev) if w.varlen else None
    o = torch.empty_like(dq)
    Nq = maxlen if w.varlen else w.Nq
    lse = torch.empty((w.B, w.H, Nq), dtype=torch.float32, device=dev)

    t8 = None
    if args.fp8:
        if w.d != 128 or args.split:
            raise SystemExit("--fp8 takes d = 128 workloads without --split")
        t8 = (fa.quantize_fp8_varlen(dq, dk, dv, dcu, dcu, maxlen, maxlen) if w.varlen
              else fa.quantize_fp8(dq, dk, dv))
        torch.cuda.synchronize(dev)

    def step_on(bq, bk, bv, bcu, bt8, bo, bl):
        if args.fp8:
            (fa.forward_fp8_varlen if w.varlen else fa.forward_fp8)(bt8, causal=args.causal, out=bo, lse=bl)
            return
        if args.split:
            fa.forward_splitkv(bq, bk, bv, out=bo, lse=bl, causal=args.causal, workspace=ws)
        elif w.varlen:
            fa.forward(bq, bk, bv, cu_seqlens=bcu, max_seqlen=maxlen, out=bo, lse=bl, causal=args.causal)
        else:
            fa.forward_qk(bq, bk, bv, out=bo, lse=bl, causal=args.causal)

    def step():
        step_on(dq, dk, dv, dcu, t8, o, lse)

    ws = None
    if args.split:
        if w.varlen:
            raise SystemExit("--split takes dense workloads only")
        n_split = fa.splitkv_num_splits(w.B, w.Nq, w.Nk, w.H, w.d)
        ws = torch.empty(fa.splitkv_workspace_bytes(w.B, w.Nq, w.H, w.d, n_split), dtype=torch.uint8,
                         device=dev)
    if args.autotune:
        if w.varlen:
            fa.autotune(dq, dk, dv, cu_seqlens=dcu, max_seqlen=maxlen)
        else:
            fa.autotune(dq, dk, dv)
    kernel_cfg = fa.get_config(w.d, maxlen if w.varlen else w.Nk, w.varlen)

    # ---------------------------------------------------------- device timing
    for _ in range(args.warmup):
        step()
    graph = None
    if args.graph:
        # Replay the timed launches from a CUDA graph: removes host launch
        # overhead, which dominates for problems of a few microseconds.
        torch.cuda.synchronize(dev)
        gs = torch.cuda.Stream(device=dev)
        gs.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(gs):
            with torch.cuda.graph(graph, stream=gs):
                for _ in range(args.steps):
                    step()
        torch.cuda.synchronize(dev)
    rc, info = fa.check_status()
    if rc != fa.FA_OK:
        raise SystemExit("device error during warm-up: %s %s" % (fa.strerror(rc), info))
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    sampler = ClockSampler("GPU-%s" % uuid if uuid is not None else str(local))
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    marks = [] if graph is not None else [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    e0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i_ in range(args.steps):
            marks[i_].record(stream)
            step()
        marks[-1].record(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    step_stats = per_step_stats(marks)
    rc, info = fa.check_status()
    if rc != fa.FA_OK:
        raise SystemExit("device error in the timed region: %s %s" % (fa.strerror(rc), info))
    ms_max = max_over_ranks(ms, world)
    flops = w.flops(causal=args.causal)
    value = world * flops / (ms_max * 1e-3) / 1e12
    kernel_tflops = flops / (ms * 1e-3) / 1e12  # one launch per step, this rank

    # ------------------------------------------------------------ sustained
    # The same step back to back for a few seconds: the clocks settle under
    # the power limit, so this is compared with the sustained GEMM peak.
    sustained = None
    if args.sustained_seconds > 0 and graph is None:
        n_sus = max(args.steps, int(math.ceil(args.sustained_seconds * 1e3 / ms)))
        sampler2 = ClockSampler("GPU-%s" % uuid if uuid is not None else str(local))
        sampler2.start()
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        s0.record(stream)
        for _ in range(n_sus):
            step()
        s1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
        clk_sus = sampler2.stop()
        ms_sus = max_over_ranks(s0.elapsed_time(s1) / n_sus, world)
        sustained = {"value": world * flops / (ms_sus * 1e-3) / 1e12, "unit": UNIT, "ms_per_step": ms_sus,
                     "steps": n_sus, "seconds": ms_sus * n_sus / 1e3, "clocks": clk_sus}
        rc, info = fa.check_status()
        if rc != fa.FA_OK:
            raise SystemExit("device error in the sustained region: %s %s" % (fa.strerror(rc), info))

    # -------------------------------------------------------- end to end
    e2e_steps = max(3, min(args.steps, 20))
    # Every step copies its inputs from pinned host memory (the e4m3 codes for
    # --fp8; their block scales stay resident) and its O and LSE back.
    if args.fp8:
        q, k, v = t8.q8.cpu(), t8.k8.cpu(), t8.vt8.cpu()
    host_in = [t.pin_memory() for t in (q, k, v)] + ([cu_q.pin_memory()] if w.varlen else [])

    def device_set(first):
        if first:
            ins = [t8.q8, t8.k8, t8.vt8] if args.fp8 else [dq, dk, dv]
            bt8, bo, bl = t8, o, lse
        else:
            ins = [torch.empty_like(t) for t in ((t8.q8, t8.k8, t8.vt8) if args.fp8 else (dq, dk, dv))]
            bt8 = None
            if args.fp8:
                # The same block scales with this set's code buffers.
                bt8 = copy.copy(t8)
                bt8.q8, bt8.k8, bt8.vt8 = ins
            bo, bl = torch.empty_like(o), torch.empty_like(lse)
        if w.varlen:
            ins = ins + [dcu if first else torch.empty_like(dcu)]
            if bt8 is not None and not first:
                bt8.cu_seqlens_q = bt8.cu_seqlens_k = ins[3]
        return ins, [bo, bl], bt8

    sets = [device_set(True), device_set(False)]
    host_out = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (o, lse)] for _ in range(2)]

    def run_set(si):
        ins, (bo, bl), bt8 = sets[si]
        step_on(ins[0], ins[1], ins[2], ins[3] if w.varlen else None, bt8, bo, bl)

    e2e_ms = max_over_ranks(pipelined_e2e(torch, dev, stream, [(s_[0], s_[1]) for s_ in sets], host_in, host_out,
                                          run_set, e2e_steps, world), world)
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = o.numel() * o.element_size() + lse.numel() * lse.element_size()
    # The host link measured in the same run: one step's input bytes host ->
    # device and its output bytes device -> host, alone (best of three).
    h2d_gbs = copy_gbs(torch, dev, sets[1][0], host_in)
    d2h_gbs = copy_gbs(torch, dev, host_out[0], sets[0][1])
    rc, info = fa.check_status()
    if rc != fa.FA_OK:
        raise SystemExit("device error in the e2e region: %s %s" % (fa.strerror(rc), info))

    if rank != 0:
        return 0
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_note = "%s bf16 dense burst (MEASURED_PEAKS.json)" % src if src == "measured" else "fallback 1.9 PFLOP/s bf16"
    if args.fp8:
        peak *= 2.0
        peak_note = "fp8 dense = 2 x " + peak_note + " (nominal fp8/bf16 ratio 4.5/2.25)"
    traffic = load_traffic(w.name + ("_fp8" if args.fp8 else "") + ("_causal" if args.causal else ""))
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "step_ms": step_stats, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3 (fp32 accumulate)" if args.fp8 else "bf16",
        "data": "synthetic (seeded N(0,1), generated on the host)",
        "config": workload_config(w, args.causal),
        "kernel": kernel_info(w, args, None if args.fp8 else kernel_cfg),
        "pct_of_peak": 100.0 * kernel_tflops / peak,
        "roofline": {"bound": "tensor", "achieved": kernel_tflops, "peak": peak, "unit": UNIT,
                     "frac": kernel_tflops / peak, "traffic": traffic,
                     "peak_source": peak_note,
                     "kernel": ("fa_fwd_kernel<128,128,4,fp8%s>" % (",varlen" if w.varlen else "")) if args.fp8
                     else "fa_fwd_kernel<%d,128,*>" % w.d,
                     "algorithmic_flops_per_launch": flops},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "steps": e2e_steps, "copies": E2E_COPIES,
                "h2d_gbs": h2d_gbs, "d2h_gbs": d2h_gbs,
                "copy_bound_ms": 1e3 * h2d / (h2d_gbs * 1e9) if h2d_gbs else None},
        "gpu_launches": args.steps * (2 if args.split else 1),
        "clocks": clocks,
    }
    if sustained is not None:
        sus_peak = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
        if args.fp8:
            sus_peak *= 2.0
        sustained["peak"] = sus_peak
        sustained["frac"] = sustained["value"] / world / sus_peak
        sustained["peak_source"] = ("%s bf16 dense sustained (MEASURED_PEAKS.json)%s"
                                    % (src, ", x2 for fp8" if args.fp8 else ""))
        line["sustained"] = sustained
    if world == 1 and args.cpu_baseline != "none":
        line["cpu_baseline"] = cpu_baseline(args, w)
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


BWD_METRIC = "attention bwd TFLOP/s (bf16, 2.5x forward FLOPs) and % of GB300 bf16 peak"


def run_bwd(args, w):
    """Backward pass over the (dense, d = 128) workload: device time per step
    with inputs resident, and the same through the public call with host
    buffers (q, k, v, o, lse, dO in; dq, dk, dv out)."""
    import torch
    import attention_forward_fa2_gb300 as fa
    from attention_forward_fa2_gb300 import build as fabuild
    from attention_forward_fa2_gb300 import inputs as I

    rank, local, world = dist_setup(args.gpus)
    torch.cuda.set_device(local)
    fabuild.build()
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    q, k, v, cu_q, cu_k = I.make(w)
    dout = I.randn_bf16(tuple(q.shape), torch.Generator().manual_seed(w.seed + 1000))
    dq, dk, dv, ddo = q.to(dev), k.to(dev), v.to(dev), dout.to(dev)
    if w.varlen:
        maxlen = max(w.lengths)
        dcq, dck = cu_q.to(dev), cu_k.to(dev)
        o, lse = fa.forward_qk(dq, dk, dv, None, dcq, dck, maxlen, maxlen, causal=args.causal)
        ws = torch.empty(fa.bwd_workspace_bytes(w.B, maxlen, w.H, w.d), dtype=torch.uint8, device=dev)
    else:
        o, lse = fa.forward_qk(dq, dk, dv, causal=args.causal)
        ws = torch.empty(fa.bwd_workspace_bytes(w.B, w.Nq, w.H, w.d), dtype=torch.uint8, device=dev)
    gq, gk, gv = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)

    def backward_on(bq, bk, bv, bo, bl, bdo, rq, rk, rv):
        if w.varlen:
            fa.backward_varlen(bq, bk, bv, bo, bl, bdo, dcq, dck, maxlen, maxlen, causal=args.causal, workspace=ws,
                               dq=rq, dk=rk, dv=rv)
        else:
            fa.backward(bq, bk, bv, bo, bl, bdo, causal=args.causal, workspace=ws, dq=rq, dk=rk, dv=rv)

    def step():
        backward_on(dq, dk, dv, o, lse, ddo, gq, gk, gv)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    rc, info = fa.check_status()
    if rc != fa.FA_OK:
        raise SystemExit("device error during warm-up: %s %s" % (fa.strerror(rc), info))
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    sampler = ClockSampler("GPU-%s" % uuid if uuid is not None else str(local))
    sampler.start()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    e0.record(stream)
    for i_ in range(args.steps):
        marks[i_].record(stream)
        step()
    marks[-1].record(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    ms = e0.elapsed_time(e1) / args.steps
    step_stats = per_step_stats(marks)
    rc, info = fa.check_status()
    if rc != fa.FA_OK:
        raise SystemExit("device error in the timed region: %s %s" % (fa.strerror(rc), info))
    ms_max = max_over_ranks(ms, world)
    flops = 2.5 * w.flops(causal=args.causal)
    value = world * flops / (ms_max * 1e-3) / 1e12
    step_tflops = flops / (ms * 1e-3) / 1e12

    e2e_steps = max(3, min(args.steps, 10))
    hosts = [t.pin_memory() for t in (q, k, v, o.cpu(), lse.cpu(), dout)]
    sets = [([dq, dk, dv, o, lse, ddo], [gq, gk, gv]),
            ([torch.empty_like(t) for t in (dq, dk, dv, o, lse, ddo)], [torch.empty_like(t) for t in (gq, gk, gv)])]
    outs = [[torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (gq, gk, gv)] for _ in range(2)]

    def run_set(si):
        (bq, bk, bv, bo, bl, bdo), (rq, rk, rv) = sets[si]
        backward_on(bq, bk, bv, bo, bl, bdo, rq, rk, rv)

    e2e_ms = max_over_ranks(pipelined_e2e(torch, dev, stream, sets, hosts, outs, run_set, e2e_steps, world), world)
    if rank != 0:
        return 0
    peaks, src = load_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    line = {
        "metric": BWD_METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "step_ms": step_stats, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) q, k, v, dO; o and lse from the forward)",
        "config": workload_config(w, args.causal),
        "kernel": {"launch": "stream launches", "form": "backward (fa_bwd%s)" % ("_varlen" if w.varlen else "")},
        "pct_of_peak": 100.0 * step_tflops / peak,
        "roofline": {"bound": "tensor", "achieved": step_tflops, "peak": peak, "unit": UNIT,
                     "frac": step_tflops / peak, "traffic": None,
                     "peak_source": "%s bf16 dense burst (MEASURED_PEAKS.json)" % src
                     if src == "measured" else "fallback 1.9 PFLOP/s bf16",
                     "kernel": "fa_bwd step (prep + fa_bwd_kernel<%d> + dq conversion); achieved is "
                               "per step, a lower bound for the key-block kernel" % w.d,
                     "algorithmic_flops_per_launch": flops},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in hosts),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in outs[0]),
                "ms_per_step": e2e_ms, "steps": e2e_steps, "copies": E2E_COPIES},
        "gpu_launches": args.steps * 3,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


PHASE_NAMES = {
    "mma": (0, ("wait_q", "wait_kv", "wait_p", "wait_o_empty", "issue", "steps", "units")),
    "load": (8, ("wait_q_empty", "wait_kv_empty", "issue", "ring_slots")),
    "softmax_tile0": (16, ("wait_s", "store_publish", "steps", "max_recomputed", "final", "load_s", "exp")),
    "softmax_tile1": (24, ("wait_s", "store_publish", "steps", "max_recomputed", "final", "load_s", "exp")),
    "epilogue": (32, ("wait_l_and_o", "read_o", "staging_wait", "store", "tiles")),
}


# Event trace of the instrumented build: TRACE_SHAPE = (units, steps, events)
# words after the per-CTA phase words, and the index of each event (the
# TraceEvent enumeration of the kernel source; "...0" events of tile 1 are the
# tile-0 index + 1).
TRACE_SHAPE = (3, 40, 32)
TRACE_EVENTS = {
    "mma_kv": 0, "mma_p0": 1, "mma_pv0": 3, "mma_s0": 5, "mma_o_empty": 7, "soft_s0": 8,
    "soft_p0": 10, "soft_load0": 12, "soft_exp0": 13, "epi_o0": 14, "load_kv": 16, "load_q": 17,
    "mma_q": 18, "mma_q_empty": 19, "mma_wait_q": 20, "mma_wait_kv": 21, "mma_step_end": 22,
    "mma_decoded": 23, "soft_warp_p": 24,
}


def trace_summary(tr):
    """Median hand-off latencies (cycles) from the event trace of CTA 0's first
    unit, and the timeline of each unit boundary: tr[unit, step, event]
    clock64 stamps (0 = not recorded)."""
    import numpy as np
    E = TRACE_EVENTS
    u = tr[0]
    nsteps = tr.shape[1]
    med = lambda a: round(float(np.median(a)), 1) if len(a) else None
    res = {}
    steps = [j for j in range(1, nsteps - 1) if u[j, E["mma_kv"]] > 0 and u[j + 1, E["mma_kv"]] > 0]
    for t in (0, 1):
        s_issue = [u[j, E["mma_s0"] + t] for j in steps]
        s_seen = [u[j, E["soft_s0"] + t] for j in steps]
        p_pub = [u[j, E["soft_p0"] + t] for j in steps]
        p_seen = [u[j + 1, E["mma_p0"] + t] for j in steps]  # P(j) is consumed at step j + 1
        ok = [i for i in range(len(steps)) if min(s_issue[i], s_seen[i], p_pub[i], p_seen[i]) > 0]
        res["tile%d_S_issued_to_softmax_sees_S" % t] = med([s_seen[i] - s_issue[i] for i in ok])
        res["tile%d_softmax_S_to_P_published" % t] = med([p_pub[i] - s_seen[i] for i in ok])
        res["tile%d_P_published_to_mma_sees_P" % t] = med([p_seen[i] - p_pub[i] for i in ok])
        res["tile%d_cycle" % t] = med([u[j + 1, E["mma_s0"] + t] - u[j, E["mma_s0"] + t] for j in steps
                                       if u[j + 1, E["mma_s0"] + t] > 0 and u[j, E["mma_s0"] + t] > 0])
    res["tile0_softmax_load"] = med([u[j, E["soft_load0"]] - u[j, E["soft_s0"]] for j in steps
                                     if u[j, E["soft_load0"]] > 0 and u[j, E["soft_s0"]] > 0])
    res["tile0_softmax_exp"] = med([u[j, E["soft_exp0"]] - u[j, E["soft_load0"]] for j in steps
                                    if u[j, E["soft_exp0"]] > 0 and u[j, E["soft_load0"]] > 0])
    res["mma_pv0_issue"] = med([u[j, E["mma_pv0"]] - u[j, E["mma_p0"]] for j in steps
                                if u[j, E["mma_pv0"]] > 0 and u[j, E["mma_p0"]] > 0])
    res["mma_s0_issue_after_pv0"] = med([u[j, E["mma_s0"]] - u[j, E["mma_pv0"]] for j in steps
                                         if u[j, E["mma_s0"]] > 0 and u[j, E["mma_pv0"]] > 0])
    # Spread of the P(j) publication over the four warps of each tile: the
    # MMA thread sees P when the last of them has arrived.
    wp = E["soft_warp_p"]
    for t in (0, 1):
        spread = [max(u[j, wp + 4 * t:wp + 4 * t + 4]) - min(u[j, wp + 4 * t:wp + 4 * t + 4]) for j in steps
                  if min(u[j, wp + 4 * t:wp + 4 * t + 4]) > 0]
        last_warp = [int(np.argmax(u[j, wp + 4 * t:wp + 4 * t + 4])) for j in steps
                     if min(u[j, wp + 4 * t:wp + 4 * t + 4]) > 0]
        res["tile%d_P_warp_spread" % t] = med(spread)
        res["tile%d_P_last_warp_counts" % t] = [last_warp.count(i) for i in range(4)] if last_warp else None
    res["raw_unit0_first_steps"] = [[int(x) for x in u[j]] for j in range(0, min(4, nsteps))]
    # Unit boundaries (unit n -> n + 1), relative to the MMA thread's last P V
    # issue of tile 0 in unit n (cycles).  The epilogue's events of a unit sit
    # in its step rows 0 (O final seen), 1 (O read, O-empty signalled) and 2
    # (staging free).
    for n in range(tr.shape[0] - 1):
        u, v = tr[n], tr[n + 1]
        pv0 = u[:, E["mma_pv0"]]
        if not (pv0 > 0).any() or v[0, E["mma_kv"]] <= 0:
            continue
        last = max(j for j in range(nsteps) if pv0[j] > 0)
        t0 = pv0[last]
        rel = lambda x: int(x - t0) if x > 0 else None
        eo = E["epi_o0"]
        res["boundary_%d_%d" % (n, n + 1)] = {
            "epi_tile0_O_final_seen": rel(u[0, eo]), "epi_tile0_staging_free": rel(u[2, eo]),
            "epi_tile0_O_read": rel(u[1, eo]), "epi_tile1_O_final_seen": rel(u[0, eo + 1]),
            "epi_tile1_staging_free": rel(u[2, eo + 1]), "epi_tile1_O_read": rel(u[1, eo + 1]),
            "mma_next_decoded": rel(v[0, E["mma_decoded"]]), "mma_next_Q_wait": rel(v[0, E["mma_wait_q"]]),
            "mma_next_Q_seen": rel(v[0, E["mma_q"]]), "mma_next_kv0": rel(v[0, E["mma_kv"]]),
            "mma_next_S0_issued": rel(v[0, E["mma_s0"]]), "mma_next_S1_issued": rel(v[0, E["mma_s0"] + 1]),
            "mma_next_P0_seen": rel(v[1, E["mma_p0"]]), "mma_next_O_empty_seen": rel(v[1, E["mma_o_empty"]]),
            "mma_next_PV1_issued": rel(v[1, E["mma_pv0"] + 1]),
            "soft_last_P0": rel(u[last - 1, E["soft_p0"]]) if last >= 1 else None,
            "soft_next_S0_seen": rel(v[0, E["soft_s0"]]), "soft_next_P0_published": rel(v[0, E["soft_p0"]]),
            "mma_Q_empty_committed": rel(max(u[:, E["mma_q_empty"]])),
            "load_last_slot_issued": rel(u[last, E["load_kv"]]),
            "load_next_Q_issued": rel(v[0, E["load_q"]]), "load_next_kv0_issued": rel(v[0, E["load_kv"]]),
            "load_next_kv1_issued": rel(v[1, E["load_kv"]])}
    return res


def run_phase(args, w):
    """--phase: one forward of the workload through the phase-clock build of
    the library (libfa_gb300_phase.so); prints where each role of a CTA spends
    its cycles, averaged over the CTAs.  The instrumented kernel is slightly
    slower than the product one, so this line is a diagnostic, not a bench
    value."""
    import torch
    import attention_forward_fa2_gb300 as fa
    from attention_forward_fa2_gb300 import build as fabuild
    from attention_forward_fa2_gb300 import inputs as I

    fabuild.build(phase=True)
    L = fa.load_library(fa.PHASE_LIB_PATH)
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    q, k, v, cu_q, cu_k = I.make(w)
    dq, dk, dv = q.to(dev), k.to(dev), v.to(dev)
    maxlen = max(w.lengths) if w.varlen else w.Nq
    dcu = cu_q.to(dev).contiguous() if w.varlen else None
    o = torch.empty_like(dq)
    lse = torch.empty((w.B, w.H, maxlen), dtype=torch.float32, device=dev)
    # One record per CTA of the grid (one CTA per work item of 256 query rows).
    items = w.B * w.H * ((maxlen + 255) // 256)
    trace_words = TRACE_SHAPE[0] * TRACE_SHAPE[1] * TRACE_SHAPE[2]  # event trace of CTA 0
    buf = torch.zeros(items * 48 + trace_words, dtype=torch.int64, device=dev)
    words = L.fa_set_phase_buffer(buf.data_ptr(), buf.numel())
    if words <= 0:
        raise SystemExit("fa_set_phase_buffer failed: %d" % words)
    stream = torch.cuda.current_stream(dev).cuda_stream
    cu = dcu.data_ptr() if dcu is not None else None
    t8 = None
    if args.fp8:
        if w.varlen:
            raise SystemExit("--phase --fp8 covers the dense workloads")
        t8 = fa.quantize_fp8(dq, dk, dv)  # codes and scales (the quantiser is not instrumented)
        torch.cuda.synchronize(dev)
    for _ in range(args.warmup + 1):
        if t8 is not None:
            rc = L.fa_fwd_fp8(t8.q8.data_ptr(), t8.k8.data_ptr(), t8.vt8.data_ptr(), t8.q_scale.data_ptr(),
                              t8.k_scale.data_ptr(), t8.v_scale.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B,
                              w.Nq, w.Nk, w.H, w.H, w.d, 1.0 / math.sqrt(w.d), 1 if args.causal else 0, stream)
        else:
            rc = L.fa_fwd_ex(dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), o.data_ptr(), lse.data_ptr(), w.B,
                             maxlen, maxlen if w.varlen else w.Nk, w.H, w.H, w.d, 1.0 / math.sqrt(w.d), cu, cu,
                             fa.FA_FLAG_CAUSAL if args.causal else 0, stream)
        if rc != 0:
            raise SystemExit("forward failed: %d" % rc)
    info = (ctypes.c_int * 3)()
    rc = L.fa_check_status(stream, info)
    L.fa_set_phase_buffer(None, 0)
    if rc != 0:
        raise SystemExit("device status %d" % rc)
    allw = buf.cpu().numpy()
    # The trace follows the words of the grid (one CTA per item for packed
    # batches, else min(items, SMs) CTAs).
    nsm = torch.cuda.get_device_properties(dev).multi_processor_count
    launched = items if w.varlen else min(items, nsm)
    ph = allw[:launched * words].reshape(-1, words).astype("float64")
    ph = ph[ph[:, 41] > 0]
    grid = int(ph.shape[0])
    tr = allw[launched * words:launched * words + trace_words].reshape(TRACE_SHAPE).astype("float64")
    trace = trace_summary(tr)
    if args.trace_out:
        with open(args.trace_out, "w") as f:
            json.dump(tr.astype("int64").tolist(), f)
    out = {}
    for role, (base, names) in PHASE_NAMES.items():
        out[role] = {n: round(float(ph[:, base + i].mean()), 1) for i, n in enumerate(names)}
    ns = float((ph[:, 41] - ph[:, 40]).mean())
    cycles = sum(out["mma"][n] for n in ("wait_q", "wait_kv", "wait_p", "wait_o_empty", "issue"))
    steps = max(out["mma"]["steps"], 1.0)
    per_step = {"mma_" + n: round(out["mma"][n] / steps, 1) for n in ("wait_q", "wait_kv", "wait_p",
                                                                      "wait_o_empty", "issue")}
    for t in ("softmax_tile0", "softmax_tile1"):
        st = max(out[t]["steps"], 1.0)
        for n in ("wait_s", "load_s", "exp", "store_publish"):
            per_step[t + "_" + n] = round(out[t][n] / st, 1)
    line = {"phase_clocks": out, "per_key_value_step_cycles": per_step, "ctas": grid, "trace": trace,
            "cta_ns": round(ns, 1), "mma_role_cycles": round(cycles, 1),
            "clock_ghz_estimate": round(cycles / ns, 3) if ns > 0 else None,
            "workload": w.name, "causal": bool(args.causal), "fp8": bool(args.fp8),
            "note": "instrumented build (FA_PHASE_CLOCKS=1), last of %d launches; not a bench value"
                    % (args.warmup + 1)}
    print(json.dumps(line))
    return 0


def main(argv=None):
    from attention_forward_fa2_gb300 import inputs as I
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="page", choices=sorted(I.WORKLOADS))
    ap.add_argument("--autotune", action="store_true", help="tune the kernel config first")
    ap.add_argument("--graph", action="store_true",
                    help="replay the timed launches from a CUDA graph (small problems)")
    ap.add_argument("--split", action="store_true",
                    help="key-split form (short query sets); launches also count the merge kernel")
    ap.add_argument("--causal", action="store_true",
                    help="causal mask (FLOPs count the visible query/key pairs only)")
    ap.add_argument("--bwd", action="store_true", help="time the backward pass instead")
    ap.add_argument("--fp8", action="store_true", help="time the e4m3 forward instead")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="oracle sample budget")
    ap.add_argument("--cpu-baseline", choices=("auto", "full", "sample", "none"), default="auto",
                    help="oracle timing: the whole workload once (default for the page workload), "
                         "a bounded sample (default otherwise), or none")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="same as --cpu-baseline none")
    ap.add_argument("--sustained-seconds", type=float, default=3.0,
                    help="length of the back-to-back window for the sustained figure (0: skip)")
    ap.add_argument("--phase", action="store_true",
                    help="diagnostic: per-role phase clocks of one forward (instrumented build)")
    ap.add_argument("--trace-out", default=None,
                    help="with --phase: write the raw event trace [unit][step][event] (JSON) to this file")
    args = ap.parse_args(argv)
    if args.no_cpu_baseline:
        args.cpu_baseline = "none"
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    w = I.WORKLOADS[args.workload]
    if args.impl == "reference":
        return run_reference(args, w)
    if args.phase:
        return run_phase(args, w)
    if args.bwd:
        return run_bwd(args, w)
    return run_ours(args, w)


if __name__ == "__main__":
    sys.exit(main())
