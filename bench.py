#!/usr/bin/env python
"""Benchmark of the gpt-oss MoE MLP block (libmoe_b300) on B300 GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

A step is one moe_forward over one batch of T synthetic tokens: router, top-4,
selected softmax, permutation, grouped gate_up GEMM with clamped SwiGLU, grouped
down GEMM with the weighted combine in its epilogue.  The default workload is
the gpt-oss-20b MoE layer at decode (T = 32, d = W = 2880, E = 32, top-4).
Inputs are resident in HBM when the timed region starts; L2 is flushed (a
256 MB write, then a 256 MB read) before every timed step.  Prints ONE JSON
line (rank 0).  Its "workloads" key adds device-timed results for the other
gpt-oss layer shapes (20b prefill, 120b prefill, 120b skewed at T = 16384 and
T = 64) unless --workloads-only-main is given.

Under torchrun (N > 1) every rank runs an independent replica of the layer on
its own GPU (the layer needs no exchange between GPUs); `value` is the tokens
of all ranks over the slowest rank's time.  `--gpus N` without torchrun's
environment starts N such ranks itself.

--impl reference times the CPU oracle (fp64 numpy, the checker of this
library) on a bounded token sample of the same workload; only rank 0 works.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import socket
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from sparse_moe_transformer_selected_b300 import inputs as gen  # noqa: E402

METRIC = "MoE-layer tokens/s at 20b/120b shapes; % of HBM or tensor-pipe roofline"
# trace-event intervals of one moe_forward (include/moe.h, moe_set_trace_events);
# the combine runs in the down kernel's epilogue, so the last interval is empty
STAGES = ["router_topk", "route_scan", "route_scatter", "gate_up", "down_combine", "_end"]
FUSE_SCAN_TILES = 8          # router tiles of 32 tokens up to which top-k runs the scan
OTHER_WORKLOADS = ["gptoss20b_prefill", "gptoss120b_prefill", "gptoss120b_skew16k",
                   "gptoss120b_skew64"]
# steps shorter than this are timed against the burst peaks
SUSTAINED_AFTER_MS = 1000.0


def kernels_per_step(T: int, d: int, E: int, block_scaled: bool) -> int:
    """Kernels one moe_forward launches: router logits, router top-k, then
    gate_up and down with the combine (the block-scaled design runs the three
    in one kernel); plus the scan and the scatter when T has more than 8
    router tiles (else the last top-k CTA runs them), and the scatter whenever
    the TMEM design needs its gathered f16 rows.  Above 8 router tiles with d a
    multiple of 64 (and E <= 256) the logits run on the tensor cores, after a
    kernel that splits the router weights into bf16 terms."""
    tiles = (T + 31) // 32
    experts = 1 if block_scaled else 2
    if tiles > FUSE_SCAN_TILES:
        tc_split = 1 if (d % 64 == 0 and 1 <= E <= 256) else 0
        return 4 + experts + tc_split
    return 2 + experts + (0 if block_scaled else 1)


KERNEL_SOURCES = {
    "router_topk": "router_topk.cu", "route_scan": "permute.cu", "route_scatter": "permute.cu",
    "gate_up": "expert_gemm_tmem.cu", "down_combine": "expert_gemm_tmem.cu",
}
# the block-scaled design (E4M3-term activations) runs gate_up, down and the
# combine as one kernel, timed as the stage "experts"
MX_SOURCES = {"experts": "expert_gemm_mx.cu"}
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


def kernel_source(kernel: str, mx: bool) -> str:
    return (MX_SOURCES if mx else KERNEL_SOURCES).get(kernel, KERNEL_SOURCES.get(kernel, ""))


def env_rank():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)),
            int(os.environ.get("WORLD_SIZE", 1)))


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------ clocks --

class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"moe_bench_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# ----------------------------------------------------- algorithmic work --

def stage_work(wl: gen.Workload, counts: np.ndarray):
    """Algorithmic bytes and flops of each kernel for one step (ideal traffic:
    every operand read once, every result written once)."""
    T, d, W, E, k = wl.T, wl.d, wl.W, wl.E, wl.k
    R = T * k
    active = int((counts > 0).sum())
    gu_bytes_expert = 2 * W * d // 2 + 2 * W * d // 32 + 2 * W * 2          # codes, scales, bias
    dn_bytes_expert = d * W // 2 + d * W // 32 + d * 2
    out = {
        "router_topk": {"flops": 2 * T * d * E, "bytes": T * d * 2 + E * d * 4 + E * 4 + R * 12},
        "route_scan": {"flops": 0, "bytes": 8 * E * ((T + 31) // 32) + 8 * (E + 1)},
        "route_scatter": {"flops": 0, "bytes": R * d * 2 + T * d * 2 + R * 20},
        "gate_up": {"flops": 2 * R * d * 2 * W,
                    "bytes": active * gu_bytes_expert + R * d * 2 + R * W * 4,
                    "unit": f"{active} active experts x {gu_bytes_expert} B + x_perm + h"},
        # y written once and read back once by the combine, out written once
        "down_combine": {"flops": 2 * R * W * d + 2 * R * d,
                         "bytes": active * dn_bytes_expert + R * W * 4 + 2 * R * d * 4 + T * d * 2,
                         "unit": f"{active} active experts x {dn_bytes_expert} B + h + y + out"},
        "_active": active,
    }
    out["experts"] = {
        "flops": out["gate_up"]["flops"] + out["down_combine"]["flops"],
        "bytes": active * (gu_bytes_expert + dn_bytes_expert) + T * d * 2 + T * d * 2,
        "unit": f"{active} active experts x {gu_bytes_expert + dn_bytes_expert} B + x terms + out "
                "(h and y are produced and consumed inside the kernel)"}
    return out


def kernel_traffic(kernel: str, workload: str, mx: bool = False):
    """DRAM bytes per launch from a committed ncu capture, if the kernel's source
    is unchanged since (profiles/dram_traffic.txt: kernel workload sha bytes)."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    src = os.path.join(ROOT, "sparse_moe_transformer_selected_b300", "csrc", kernel_source(kernel, mx))
    if not os.path.exists(path) or not os.path.exists(src):
        return None
    sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    with open(path) as f:
        for line in f:
            p = line.split()
            if len(p) == 4 and not line.startswith("#") and p[0] == kernel and p[1] == workload \
                    and p[2] == sha:
                return float(p[3])
    return None


def roofline(wl, counts, stage_ms, step_ms, mx, peaks, peak_src, mma_peaks=None):
    """The dominant kernel against its roofline: HBM bytes when its flop/byte is
    under the ridge point, else tensor flops against the dense peak of the MMA
    kind it issues (kind::f16: bf16's; burst for steps under a second)."""
    work = stage_work(wl, counts)
    top = max((s for s in stage_ms if s in work), key=lambda s_: stage_ms[s_])
    wk = work[top]
    intensity = wk["flops"] / max(1, wk["bytes"])
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    sec = stage_ms[top] * 1e-3
    if intensity < ridge or wk["flops"] == 0:
        roof = {"bound": "hbm", "achieved": wk["bytes"] / sec / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s"}
        note = f"HBM copy bandwidth ({peak_src})"
    else:
        sustained = step_ms >= SUSTAINED_AFTER_MS
        pk = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
        roof = {"bound": "tensor", "achieved": wk["flops"] / sec / 1e12, "peak": pk,
                "unit": "TFLOP/s"}
        note = (f"dense bf16 / kind::f16 {'sustained' if sustained else 'burst'} ({peak_src})")
    roof["frac"] = roof["achieved"] / roof["peak"]
    if roof["bound"] == "tensor" and not mx and mma_peaks and mma_peaks.get("f16_tmem_a_n128"):
        # the rate of the instruction form the TMEM design issues (kind::f16,
        # A in tensor memory; its chunks are up to 192 tokens, and N = 128 and
        # N = 256 measure the same rate) on this GPU: down issues two MMAs
        # (h hi, h lo) per K step, gate_up one
        issued = roof["achieved"] * (2.0 if top == "down_combine" else 1.0)
        roof["form_peak_tflops"] = mma_peaks["f16_tmem_a_n128"]
        roof["frac_of_form_peak"] = issued / mma_peaks["f16_tmem_a_n128"]
    roof["traffic"] = kernel_traffic(top, wl.name, mx)
    roof["kernel_source"] = kernel_source(top, mx)
    roof["kernel"] = top
    roof["peak_source"] = note
    roof["algorithmic"] = {"bytes": wk["bytes"], "flops": wk["flops"], "per": wk.get("unit", "")}
    if roof["bound"] == "hbm":
        roof["frac_of_8tbs"] = roof["achieved"] / 8000.0
    return roof, work["_active"]


# ---------------------------------------------------------- replicas --

def max_over_ranks(values, world: int, device="cpu"):
    """Per-rank timings -> their maximum over all ranks (every rank gets it).

    The layer needs no exchange between GPUs, so N > 1 runs N independent
    replicas; the job is as fast as its slowest rank.
    """
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_tokens_per_s(tokens_per_rank: int, world: int, ms_slowest: float) -> float:
    """Tokens of all ranks over the slowest rank's step time (weak scaling)."""
    return tokens_per_rank * world / (ms_slowest * 1e-3)


def free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launcher_command(argv, n: int, port: int):
    """The torchrun command that runs this script as n ranks on one node."""
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
            "--master-addr", "127.0.0.1", "--master-port", str(port),
            os.path.abspath(__file__), *argv]


# ------------------------------------------------------------- CPU arm --

def oracle_sample(inp, n_tokens: int, seed: int = 99, workers: int = 1):
    from oracle import moe_oracle as O
    rng = np.random.Generator(np.random.PCG64(seed))
    tokens = np.sort(rng.choice(inp.wl.T, size=min(n_tokens, inp.wl.T), replace=False))
    t0 = time.perf_counter()
    O.moe_forward_inputs(inp, tokens=tokens, workers=workers)
    return len(tokens), time.perf_counter() - t0


def host_cores() -> int:
    return os.cpu_count() or 1


def default_sample(wl: gen.Workload) -> int:
    # the oracle dequantises each touched expert (~1.7 s of one core at
    # d = W = 2880, spread over the cores by its expert threads), so a few
    # tokens per core take 10-30 s; small layers run whole
    return wl.T if wl.d * wl.W <= 512 * 512 else min(wl.T, 2 * host_cores())


def cpu_baseline_entry(value, n_tokens, wl, seconds, cores):
    return {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n_tokens} seeded tokens of the {wl.name} layer per timed sample "
                      f"(routing of all {wl.T} tokens + expert FFN of the sample), "
                      f"{seconds:.1f} s, experts on {cores} threads"}


def run_reference(args, wl):
    rank, _, world = env_rank()
    if rank != 0:
        return
    inp = gen.make_inputs(wl)
    cores = host_cores()
    # size each step so the whole run stays within about 150 s of CPU time
    _, t1 = oracle_sample(inp, 1, seed=7, workers=cores)
    budget = 150.0 / (args.steps + args.warmup)
    n = args.cpu_sample or max(1, min(default_sample(wl), int(budget / max(t1, 1e-3))))
    for _ in range(max(0, args.warmup - 1)):
        oracle_sample(inp, n, seed=7, workers=cores)
    times, toks = [], 0
    for s in range(args.steps):
        nt, dt = oracle_sample(inp, n, seed=100 + s, workers=cores)
        times.append(dt)
        toks += nt
    total = sum(times)
    value = toks / total
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * total / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(wl, world),
        "cpu_baseline": cpu_baseline_entry(value, n, wl, total, cores),
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_block(wl, world):
    return {"workload": wl.name, "T": wl.T, "d_model": wl.d, "expert_width": wl.W,
            "experts": wl.E, "top_k": wl.k, "weights": "MXFP4 (E2M1 x 32 + E8M0)",
            "router_bias": wl.router_bias,
            "l2": "flushed before every timed step (256 MB write, then 256 MB read)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}


# ------------------------------------------------------------- GPU arm --

def measure(wl, steps, warmup, world, flush_l2, with_e2e):
    """Device-timed steps of one workload on this rank's GPU, the per-stage
    breakdown, and (with_e2e) the end-to-end timings through the public call."""
    import torch
    from sparse_moe_transformer_selected_b300 import moe
    from sparse_moe_transformer_selected_b300.device import DeviceMoE

    inp = gen.make_inputs(wl)
    dev = DeviceMoE.upload(inp)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        dev.forward()
    torch.cuda.synchronize()
    counts = np.diff(dev.region("offsets").cpu().numpy())

    # device-timed steps, each preceded by an L2 flush; one event pair around
    # each moe_forward (nothing recorded between its kernels, so consecutive
    # kernels overlap their launches as they do for a user)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    for s in range(steps):
        flush_l2()
        ev[s][0].record(stream)
        dev.forward()
        ev[s][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ms = statistics.fmean(a_.elapsed_time(b_) for a_, b_ in ev)

    # per-stage breakdown, in separate steps with CUDA events recorded by the
    # library between its stages (on the stream the kernels run on)
    tev = [[torch.cuda.Event(enable_timing=True) for _ in range(7)] for _ in range(steps)]
    for row in tev:                                 # materialise the event handles
        for e in row:
            e.record(stream)
    torch.cuda.synchronize()
    for s in range(steps):
        flush_l2()
        moe.moe_set_trace_events(tev[s])
        dev.forward()
    moe.moe_set_trace_events(None)
    torch.cuda.synchronize()
    stage_ms = {name: statistics.fmean(r[i].elapsed_time(r[i + 1]) for r in tev)
                for i, name in enumerate(STAGES)}
    fmt, _ = dev.hidden_format()
    if fmt == moe.HIDDEN_E4M3_TERMS:
        # one expert kernel between trace events 3 and 4
        stage_ms["experts"] = stage_ms.pop("gate_up") + stage_ms.pop("down_combine")
    res = {"ms": ms, "stage_ms": stage_ms, "counts": counts,
           "mx": fmt == moe.HIDDEN_E4M3_TERMS, "dev": dev}
    if with_e2e:
        # end to end through the public call: each step copies x from pinned
        # host memory, calls moe_forward (argument checks, design choice, TMA
        # descriptors from the cache, 5-6 launches) and copies out back
        x_host = dev.x.cpu().pin_memory()
        out_host = torch.empty_like(dev.out, device="cpu").pin_memory()

        # the host side warms up more slowly than the device: in the first
        # benchmark process on a freshly started box this loop measured up to
        # 40% slower than in a second process, so the untimed steps here run
        # for at least half a second of wall time (and `warmup` steps)
        def e2e_steps(run):
            ts = []
            t_end = time.perf_counter() + 0.5
            n_warm = 0
            while n_warm < warmup or time.perf_counter() < t_end:
                dev.x.copy_(x_host, non_blocking=True)
                run()
                out_host.copy_(dev.out, non_blocking=True)
                stream.synchronize()
                n_warm += 1
            for s in range(steps):
                flush_l2()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                dev.x.copy_(x_host, non_blocking=True)
                run()
                out_host.copy_(dev.out, non_blocking=True)
                b.record(stream)
                b.synchronize()
                ts.append(a.elapsed_time(b))
            return statistics.fmean(ts)

        res["e2e_ms"] = e2e_steps(dev.forward)
        graph = dev.capture_graph()                 # the same call replayed from a CUDA graph
        res["e2e_graph_ms"] = e2e_steps(graph.replay)
        res["h2d"] = int(dev.x.numel() * 2)
        res["d2h"] = int(dev.out.numel() * 2)
    moe.moe_poll_status(dev.workspace)
    return res


def run_ours(args, wl):
    import torch
    import torch.distributed as dist
    from sparse_moe_transformer_selected_b300 import moe

    rank, local_rank, world = env_rank()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (B300)")
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    moe.load()                                     # fails loudly if the library is missing

    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    drain = torch.ones(64 << 20, dtype=torch.float32, device="cuda")   # 256 MB

    def flush_l2():
        # write a buffer twice the size of L2, then read another one: the read
        # evicts the dirty lines of the write, so their write-back to HBM does
        # not run inside the next timed step
        flush.fill_(1)
        drain.sum()

    # the dense rate of each MMA kind the GEMMs issue, with their own instruction
    # forms (moe_mma_peak): the denominators a block-scaled kernel is held to
    status_ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    mma_peaks = {kind: round(moe.moe_mma_peak(kind, 20000, status_ws), 1)
                 for kind in ("f16", "mxf8f6f4", "f16_tmem_a_n128", "f16_tmem_a_n256")}
    moe.moe_poll_status(status_ws)

    with ClockSampler(local_rank) as clk:
        main = measure(wl, args.steps, args.warmup, world, flush_l2, with_e2e=True)
    ms, e2e, e2e_graph = max_over_ranks([main["ms"], main["e2e_ms"], main["e2e_graph_ms"]], world,
                                        device="cuda")
    peaks, peak_src = load_peaks()
    roof, active = roofline(wl, main["counts"], main["stage_ms"], ms, main["mx"], peaks, peak_src,
                            mma_peaks)
    inp_main = None if args.no_cpu_baseline or world > 1 else gen.make_inputs(wl)
    del main["dev"]

    others = {}
    if not args.main_only:
        for name in OTHER_WORKLOADS:
            if name == wl.name:
                continue
            owl = gen.WORKLOADS[name]
            r = measure(owl, args.other_steps, 3, world, flush_l2, with_e2e=False)
            del r["dev"]
            oms = max_over_ranks([r["ms"]], world, device="cuda")[0]
            oroof, oact = roofline(owl, r["counts"], r["stage_ms"], oms, r["mx"], peaks, peak_src,
                                   mma_peaks)
            others[name] = {
                "tokens_per_s": whole_job_tokens_per_s(owl.T, world, oms), "ms_per_step": oms,
                "steps": args.other_steps, "design": "block-scaled" if r["mx"] else "tmem f16",
                "roofline": {k_: oroof[k_] for k_ in ("bound", "kernel", "achieved", "unit",
                                                      "peak", "frac", "peak_source",
                                                      "form_peak_tflops", "frac_of_form_peak",
                                                      "traffic", "frac_of_8tbs")
                             if k_ in oroof},
                "stages_ms": {k_: round(v, 5) for k_, v in r["stage_ms"].items() if k_ != "_end"},
                "active_experts": oact}
            torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    mx = main["mx"]
    line = {
        "metric": METRIC, "value": whole_job_tokens_per_s(wl.T, world, ms), "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": ("e2m1 x e4m3 block-scaled MMA, fp32 accumulation" if mx
                  else "f16 x f16 MMA on exactly dequantised MXFP4, fp32 accumulation"),
        "data": "synthetic (seeded PCG64: x~N(0,1) bf16, random MXFP4 experts)",
        "config": config_block(wl, world),
        "clocks": clk.summary(),
        "e2e": {"value": whole_job_tokens_per_s(wl.T, world, e2e), "unit": "tokens/s",
                "h2d_bytes_per_step": main["h2d"], "d2h_bytes_per_step": main["d2h"],
                "call": "moe_forward through the C ABI every step",
                "graph_replay_value": whole_job_tokens_per_s(wl.T, world, e2e_graph)},
        "gpu_launches": kernels_per_step(wl.T, wl.d, wl.E, mx) * args.steps,
        "roofline": roof,
        "stages_ms": {k_: round(v, 5) for k_, v in main["stage_ms"].items() if k_ != "_end"},
        "active_experts": active,
        "mma_peaks_tflops": {**mma_peaks, "how": "moe_mma_peak: back-to-back K-steps of each "
                                                 "instruction form (f16 and mxf8f6f4: 128x256 from "
                                                 "shared memory; f16_tmem_a: A in tensor memory), "
                                                 "one CTA per SM, CUDA events (this run)"},
    }
    if others:
        line["workloads"] = others
    if inp_main is not None:
        cores = host_cores()
        n = args.cpu_sample or default_sample(wl)
        nt, dt = oracle_sample(inp_main, n, workers=cores)
        line["cpu_baseline"] = cpu_baseline_entry(nt / dt, nt, wl, dt, cores)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="gptoss20b_decode",
                    choices=sorted({**gen.WORKLOADS, **gen.STRESS_WORKLOADS}))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-sample", type=int, default=0, help="oracle tokens per CPU sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--main-only", action="store_true",
                    help="skip the device-timed results of the other gpt-oss layer shapes")
    ap.add_argument("--other-steps", type=int, default=5, help="timed steps per other workload")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)      # at least 3 untimed warm-up steps
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # not started by torchrun: start the N ranks here (one per GPU)
        raise SystemExit(subprocess.call(launcher_command(sys.argv[1:], args.gpus, free_port())))
    wl = {**gen.WORKLOADS, **gen.STRESS_WORKLOADS}[args.workload]
    if args.impl == "reference":
        run_reference(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
