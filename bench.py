"""Benchmark of the verification hot path (attention + greedy acceptance).

One step = spec_verify_attn + spec_accept_greedy over one batch of a named
synthetic workload (default: the largest one, the ragged GQA 8B-target bf16
shape -- batch 32, 32 q / 8 kv heads, head_dim 128, contexts uniform in
[1024, 8192], k = 4, page size 16, vocab 128256).  The two calls are
independent, so the acceptance runs on a second stream beside the attention
(forked and joined every step; --no-overlap: one stream, in order).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   # the float64 CPU oracle, same metric

Prints one JSON line.  `value` is verified draft tokens per second (B*k per
step / device step time, inputs resident in HBM); `e2e` is the same metric
through the public API with the per-step inputs copied from pinned host
memory and the results read back inside the timed region; `roofline` relates
the attention call's algorithmic bytes to its measured time and to the
measured HBM copy bandwidth; `accepted_tok_s` is the goodput (tokens the
step gains, sum of accepted_len + 1, per second); `timing` adds the same
steps timed by one event pair and the median of 200 individually timed
steps; `cpu_baseline` is the float64 oracle on all host cores (and on one).
With N > 1 (torchrun) every rank runs its own
replica on its own GPU (the path has no cross-GPU exchange); the slowest
rank's time counts and `value` sums all ranks' tokens.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_verification_attn_gb300.workload import (  # noqa: E402
    WORKLOADS, algorithmic_bytes, make_inputs)

DEFAULT_WORKLOAD = "gqa8b_ragged_bf16"
METRIC = "verified draft tokens/sec"
UNIT = "tokens/s"
L2_BYTES = 129 * 2**20
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when world == 1)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(units_per_rank: int, rank_seconds: float, world: int, device=None):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    slowest = reduce_max(rank_seconds, world, device)
    return units_per_rank * world / slowest, slowest


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# sources whose change makes the committed attention / acceptance counters stale:
# the kernels of the step and the device helpers they include (the ABI's other
# entry points and their kernels do not run in the step)
STEP_SOURCES = ("attn_tc.cu", "attn_tc2.cu", "attn_mma.cu", "attn_simt.cu", "attn_small.cu",
                "accept.cu", "common.cuh")


def kernel_source_hash() -> str:
    """Hash of the step's kernel sources with comments and blank lines removed
    (a comment edit does not change the kernels the counters describe)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_attn_gb300", "csrc")
    for name in STEP_SOURCES:
        with open(os.path.join(csrc, name)) as fh:
            text = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
        lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
        h.update("\n".join(ln for ln in lines if ln).encode())
    return h.hexdigest()[:16]


def profiled_traffic(workload: str):
    """DRAM bytes per attention launch from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "verify_attn_%s.md" % workload)
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*([0-9.eE+]+)", text)
    h = re.search(r"kernel_sources_sha256_16:\s*([0-9a-f]+)", text)
    if not m or not h or h.group(1) != kernel_source_hash():
        return None
    return float(m.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.samples = []
        if self.proc is None:
            return False
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 9:
                self.samples.append(parts)
        return False

    def summary(self):
        if not getattr(self, "samples", None):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(s[1]) for s in self.samples if s[1].replace(".", "").isdigit()]
        smax = [float(s[2]) for s in self.samples if s[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for s in self.samples for i in range(4)
                          if s[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(self.samples)}


# ---------------------------------------------------------------- CPU oracle timing

def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:
        return max(1, os.cpu_count() or 1)


def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else platform)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform
    return platform.machine()


def _oracle_rows_threaded(oracle, inp, rows, threads):
    """The oracle's attention rows over chunks on `threads` host threads (the
    oracle is a C library called through ctypes, which releases the GIL)."""
    from concurrent.futures import ThreadPoolExecutor
    s = inp.spec
    args = (inp.q, s.q_dtype, inp.k_cache, inp.v_cache, s.kv_dtype, inp.k_scale, inp.v_scale,
            inp.block_table, inp.ctx_lens, inp.scale)
    if threads <= 1:
        oracle.attn_rows(*args, rows)
        return
    chunks = [np.ascontiguousarray(c) for c in np.array_split(rows, min(len(rows), 8 * threads))
              if len(c)]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda c: oracle.attn_rows(*args, c), chunks))


def _oracle_accept_threaded(oracle, inp, threads):
    from concurrent.futures import ThreadPoolExecutor
    s = inp.spec
    if threads <= 1 or s.batch < 2:
        oracle.accept_greedy(inp.logits, s.logits_dtype, inp.draft_tokens)
        return
    parts = [(b0, b1) for b0, b1 in zip(*[np.linspace(0, s.batch, min(s.batch, threads) + 1,
                                                       dtype=int)[j:] for j in (0, 1)])
             if b1 > b0]
    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(lambda r: oracle.accept_greedy(np.ascontiguousarray(inp.logits[r[0]:r[1]]),
                                                   s.logits_dtype,
                                                   np.ascontiguousarray(inp.draft_tokens[r[0]:r[1]])),
                    parts))


def oracle_step_time(inp, threads: int, budget_s: float, seed: int = 0):
    """Time the float64 oracle on one step of the workload, on `threads` host
    threads: every attention row when that fits `budget_s`, else a random
    sample of the rows scaled to the whole step; plus the acceptance over all
    sequences.  Returns (seconds per full step, description, scale factor)."""
    import oracle
    s = inp.spec
    B, k, Hq = s.batch, s.num_draft, s.num_q_heads
    rows_total = B * k * Hq
    rng = np.random.default_rng(seed)
    all_rows = np.stack(np.meshgrid(np.arange(B), np.arange(k), np.arange(Hq), indexing="ij"),
                        -1).reshape(-1, 3).astype(np.int32)
    # calibrate on a few rows per thread, then fill the time budget
    probe = all_rows[rng.choice(rows_total, size=min(4 * threads, rows_total), replace=False)]
    t0 = time.perf_counter()
    _oracle_rows_threaded(oracle, inp, probe, threads)
    per_row = max((time.perf_counter() - t0) / len(probe), 1e-7)
    n = int(min(rows_total, max(len(probe), budget_s * 0.8 / per_row)))
    rows = all_rows if n == rows_total else all_rows[np.sort(rng.choice(rows_total, size=n,
                                                                        replace=False))]
    t0 = time.perf_counter()
    _oracle_rows_threaded(oracle, inp, rows, threads)
    t_attn = (time.perf_counter() - t0) * rows_total / n
    t0 = time.perf_counter()
    _oracle_accept_threaded(oracle, inp, threads)
    t_acc = time.perf_counter() - t0
    who = "%d thread%s (C float64 oracle)" % (threads, "" if threads == 1 else "s")
    if n == rows_total:
        desc = "the whole step: all %d attention rows (b, i, h) and the acceptance of all %d " \
               "sequences, on %s" % (rows_total, B, who)
    else:
        desc = ("%d of %d attention rows (b, i, h) timed and scaled by %.2fx, plus the "
                "acceptance of all %d sequences, on %s" % (n, rows_total, rows_total / n, B, who))
    return t_attn + t_acc, desc, rows_total / n


def cpu_baseline(inp, budget_s: float):
    """The oracle as it stands on the host cores: all cores (the reported
    value) and one core, each on a bounded sample of one step."""
    s = inp.spec
    units = s.batch * s.num_draft
    threads = host_threads()
    t_all, desc_all, _ = oracle_step_time(inp, threads, budget_s, seed=0)
    t_one, desc_one, _ = oracle_step_time(inp, 1, budget_s, seed=1)
    return {"value": units / t_all, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": desc_all, "cpu": cpu_model(), "cpu_count": os.cpu_count(),
            "single_core": {"value": units / t_one, "unit": UNIT, "cores": 1,
                            "sample": desc_one}}


def run_reference(args, inp, world, rank):
    """--impl reference: the oracle as it stands on the host cores (all of
    them), whole steps when the run fits a few minutes, else a bounded sample
    of each step scaled to the whole step (the factor is in the line)."""
    if rank != 0:
        return
    s = inp.spec
    units = s.batch * s.num_draft
    threads = host_threads()
    # about two and a half minutes of oracle time for the whole run
    per_step_budget = 150.0 / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        oracle_step_time(inp, threads, per_step_budget, seed=1000)
    times, desc, factors = [], "", []
    for st in range(args.steps):
        t, desc, f = oracle_step_time(inp, threads, per_step_budget, seed=st)
        times.append(t)
        factors.append(f)
    t_step = float(np.mean(times))
    value = units / t_step
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": t_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(inp, "host memory (CPU oracle)"),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "each step: " + desc, "cpu": cpu_model(),
                         "cpu_count": os.cpu_count()},
        "extrapolation": float(np.mean(factors)),
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def workload_config(inp, l2_note):
    s = inp.spec
    ctx = s.ctx if isinstance(s.ctx, int) else [int(inp.ctx_lens.min()), int(inp.ctx_lens.max())]
    return {"workload": s.name, "batch": s.batch, "q_heads": s.num_q_heads,
            "kv_heads": s.num_kv_heads, "head_dim": s.head_dim, "ctx": ctx,
            "num_draft": s.num_draft, "page_size": s.page_size, "vocab": s.vocab,
            "kv_dtype": s.kv_dtype, "seed": inp.seed, "l2": l2_note,
            "queue": "prefilled (spin kernel while the host enqueues the timed steps)",
            "parallelism": "replicas"}


# ---------------------------------------------------------------- GPU run

def run_gpu(args, inp, world, rank, local):
    import torch
    import torch.distributed as dist
    from speculative_decoding_verification_attn_gb300 import binding

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    binding.load()
    s = inp.spec
    k, scale = s.num_draft, inp.scale
    nbytes = algorithmic_bytes(inp)
    units = s.batch * k

    base = binding.inputs_to_torch(inp, device)
    rejection = args.accept == "rejection"
    if rejection:
        # lossless speculative sampling: seeded target and drafter logits of
        # the workload's shape, drafts drawn from the drafter's distribution
        from speculative_decoding_verification_attn_gb300.workload import make_rejection_inputs
        rej = make_rejection_inputs(s.batch, k, s.vocab, s.logits_dtype, seed=inp.seed)
        to_dev = lambda a: (torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
                            if s.logits_dtype == "bf16" else torch.from_numpy(a)).to(device)
        base["logits"] = to_dev(rej.target_logits)
        base["draft_logits"] = to_dev(rej.draft_logits)
        base["draft_tokens"] = torch.from_numpy(rej.draft_tokens).to(device)
        nbytes = dict(nbytes)
        extra = base["draft_logits"].numel() * base["draft_logits"].element_size()
        nbytes["accept"] += extra
        nbytes["total"] += extra
    # rotate over enough input copies that one step's inputs are out of L2
    # by the time they are used again
    n_sets = max(2, math.ceil(2.5 * L2_BYTES / nbytes["total"]))
    sets = [base] + [{n: v.clone() for n, v in base.items()} for _ in range(n_sets - 1)]
    outs = [binding.alloc_outputs(inp, device) for _ in range(n_sets)]
    stream = torch.cuda.current_stream()

    def accept(t, o, j):
        if rejection:
            binding.spec_accept_rejection(t["logits"], t["draft_logits"], t["draft_tokens"], k, 1.0,
                                          rej.seed + j, o["accepted_len"], o["next_token"])
        else:
            binding.spec_accept_greedy(t["logits"], t["draft_tokens"], k, o["accepted_len"],
                                       o["next_token"])

    # The two calls of a step are independent (acceptance reads only the
    # logits and the drafts), so by default the acceptance runs on a second
    # stream forked before the attention call and joined after it, and takes
    # the SMs the attention's tail leaves free; --no-overlap runs the two in
    # order on one stream.
    side = torch.cuda.Stream(device)
    fork_ev = [torch.cuda.Event() for _ in range(2)]
    join_ev = [torch.cuda.Event() for _ in range(2)]

    def compute(t, o, j):
        if args.overlap:
            fork_ev[j & 1].record(stream)
            side.wait_event(fork_ev[j & 1])
        binding.spec_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                 t["ctx_lens"], k, scale, o["out"], o["lse"],
                                 t.get("k_scale"), t.get("v_scale"))
        if args.overlap:
            with torch.cuda.stream(side):
                accept(t, o, j)
            join_ev[j & 1].record(side)
            stream.wait_event(join_ev[j & 1])
        else:
            accept(t, o, j)

    def step(j):
        compute(sets[j % n_sets], outs[j % n_sets], j)

    for j in range(max(args.warmup, 3)):
        step(j)
    torch.cuda.synchronize()

    # attention / acceptance / step times from events on the launching stream
    def held(n):
        # hold the stream with a spin kernel while the host enqueues the
        # timed steps, so no interval includes host submission time (the e2e
        # figure below keeps the host in the loop)
        if hasattr(torch.cuda, "_sleep"):
            torch.cuda._sleep(int(min(2e8, 1e5 * n)))

    reps = max(200, args.steps)
    rev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(reps)]
    with ClockSampler(local) as clk:
        # keep the GPU under the same load for ~1 s so the sampler sees it
        t_pad = time.perf_counter()
        j = 0
        while time.perf_counter() - t_pad < 1.0:
            step(j)
            j += 1
            if j % 64 == 0:
                torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        # the timed region: exactly K steps between one pair of events
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        held(args.steps)
        e0.record(stream)
        for j in range(args.steps):
            step(j)
        e1.record(stream)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        # a second timed region for the per-call breakdown: REPS steps with an
        # event pair around each call (the events between the two calls cost
        # the step a few microseconds, so this region does not give `value`)
        held(reps)
        for j in range(reps):
            t, o = sets[j % n_sets], outs[j % n_sets]
            rev[j][0].record(stream)
            binding.spec_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                     t["ctx_lens"], k, scale, o["out"], o["lse"],
                                     t.get("k_scale"), t.get("v_scale"))
            rev[j][1].record(stream)
            accept(t, o, j)
            rev[j][2].record(stream)
        torch.cuda.synchronize()
        # a third and fourth region: the attention calls alone, then the
        # acceptance calls alone, K each back to back between one event pair
        # (each kernel's average launch duration in a stream of its own
        # launches, for the roofline; the per-call events above block the
        # launch overlap of consecutive kernels and add their own cost)
        a0, a1, c0, c1 = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        held(2 * args.steps)
        a0.record(stream)
        for j in range(args.steps):
            t, o = sets[j % n_sets], outs[j % n_sets]
            binding.spec_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["block_table"],
                                     t["ctx_lens"], k, scale, o["out"], o["lse"],
                                     t.get("k_scale"), t.get("v_scale"))
        a1.record(stream)
        c0.record(stream)
        for j in range(args.steps):
            t, o = sets[j % n_sets], outs[j % n_sets]
            accept(t, o, j)
        c1.record(stream)
        torch.cuda.synchronize()
    clocks = clk.summary()
    value, slowest_step_s = aggregate(units, e0.elapsed_time(e1) / 1e3 / args.steps, world,
                                      device)
    ms_per_step = slowest_step_s * 1e3
    rep_step = np.array([e[0].elapsed_time(e[2]) for e in rev])
    rep_attn = np.array([e[0].elapsed_time(e[1]) for e in rev])
    rep_acc = np.array([e[1].elapsed_time(e[2]) for e in rev])
    attn_ms = a0.elapsed_time(a1) / args.steps
    acc_ms = c0.elapsed_time(c1) / args.steps
    # goodput: tokens the step gains, sum over sequences of accepted_len + 1
    # (every input set holds the same values, so any set's results serve)
    gained = int((outs[0]["accepted_len"].long() + 1).sum().item())
    accepted_tok_s = gained * world / slowest_step_s
    timing = {"step": ("acceptance on a second stream forked before the attention call and "
                       "joined after it" if args.overlap else
                       "attention then acceptance on one stream"),
              "timed_region": "K steps between one event pair (value, ms_per_step)",
              "breakdown_region": "%d steps, an event pair around each call" % reps,
              "kernel_regions": "K attention calls, then K acceptance calls, back to back "
                                "between one event pair each (roofline attn_ms / accept_ms)",
              "reps": reps, "step_median_ms": float(np.median(rep_step)),
              "step_mean_ms": float(rep_step.mean()),
              "attn_median_ms": float(np.median(rep_attn)),
              "attn_mean_ms": float(rep_attn.mean()),
              "accept_median_ms": float(np.median(rep_acc)),
              "accept_mean_ms": float(rep_acc.mean()),
              "attn_back_to_back_ms": attn_ms, "accept_back_to_back_ms": acc_ms}

    # end to end through the public API: every step's inputs copied from
    # pinned host memory and its results read back, inside the timed region.
    # A step's inputs (and its results) are packed into one buffer, so one
    # host->device and one device->host copy per step, and the copies run on
    # streams of their own: step j+1's inputs upload while step j computes,
    # over the rotating input sets (the KV cache stays resident, as it does in
    # a serving engine between steps).
    host_names = ["q", "logits", "draft_tokens", "block_table", "ctx_lens"]
    host = binding.inputs_to_torch(inp, pin=True)
    if rejection:
        host_names.append("draft_logits")
        host = dict(host)
        for n in ("logits", "draft_logits", "draft_tokens"):
            host[n] = base[n].cpu().pin_memory()
    h_in = {n: host[n] for n in host_names}
    h2d = sum(v.numel() * v.element_size() for v in h_in.values())
    d2h = sum(v.numel() * v.element_size() for v in outs[0].values())

    def layout(tensors):
        offs, off = {}, 0
        for n, v in tensors.items():
            offs[n] = off
            off += -(-(v.numel() * v.element_size()) // 256) * 256
        return offs, off

    def views(buf, offs, like):
        return {n: buf[offs[n]:offs[n] + v.numel() * v.element_size()].view(v.dtype).view(v.shape)
                for n, v in like.items()}

    in_offs, in_bytes = layout(h_in)
    out_offs, out_bytes = layout(outs[0])
    h_in_pack = torch.empty(in_bytes, dtype=torch.uint8, pin_memory=True)
    for n, v in views(h_in_pack, in_offs, h_in).items():
        v.copy_(h_in[n])
    h_out_pack = torch.empty(out_bytes, dtype=torch.uint8, pin_memory=True)
    d_in = [torch.empty(in_bytes, dtype=torch.uint8, device=device) for _ in range(n_sets)]
    d_out = [torch.empty(out_bytes, dtype=torch.uint8, device=device) for _ in range(n_sets)]
    e_sets = [dict(sets[i], **views(d_in[i], in_offs, h_in)) for i in range(n_sets)]
    e_outs = [views(d_out[i], out_offs, outs[0]) for i in range(n_sets)]
    h2d_s, d2h_s = torch.cuda.Stream(device), torch.cuda.Stream(device)
    # per input set: its upload, the compute of its last step (inputs
    # consumed) and the read-back of that step (outputs free).  Created once:
    # a wait takes the event's most recent record, so re-recording is safe.
    ev_in = [torch.cuda.Event() for _ in range(n_sets)]
    ev_done = [torch.cuda.Event() for _ in range(n_sets)]
    ev_read = [torch.cuda.Event() for _ in range(n_sets)]

    def e2e_run(n_steps, start_event=None):
        used = [False] * n_sets
        if start_event is not None:
            h2d_s.wait_event(start_event)
        for j in range(n_steps):
            i = j % n_sets
            with torch.cuda.stream(h2d_s):
                if used[i]:
                    h2d_s.wait_event(ev_done[i])
                d_in[i].copy_(h_in_pack, non_blocking=True)
                ev_in[i].record(h2d_s)
            stream.wait_event(ev_in[i])
            if used[i]:
                stream.wait_event(ev_read[i])
            compute(e_sets[i], e_outs[i], j)
            ev_done[i].record(stream)
            with torch.cuda.stream(d2h_s):
                d2h_s.wait_event(ev_done[i])
                h_out_pack.copy_(d_out[i], non_blocking=True)
                ev_read[i].record(d2h_s)
            used[i] = True
        return ev_read[(n_steps - 1) % n_sets]

    e2e_run(max(args.warmup, 3))
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    last = e2e_run(args.steps, e0)
    stream.wait_event(last)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_value, _ = aggregate(units, e0.elapsed_time(e1) / 1e3 / args.steps, world, device)
    # the read-back results are those of the device-resident run on the same inputs
    got = views(h_out_pack, out_offs, outs[0])
    ref = outs[(args.steps - 1) % n_sets]
    if not rejection and not all(torch.equal(got[n], ref[n].cpu())
                                 for n in ("accepted_len", "next_token")):
        raise SystemExit("end-to-end results differ from the device-resident run")

    peak, peak_kind = measured_peaks()
    achieved = nbytes["attn"] / (attn_ms / 1e3) / 1e9
    traffic = profiled_traffic(s.name)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if s.q_dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) q/K/V, N(0,2) logits; no datasets or weights)",
        "config": workload_config(inp, "inputs > L2: %d rotating copies of %.0f MB" %
                                  (n_sets, nbytes["total"] / 1e6)),
        "accepted_tok_s": accepted_tok_s,
        "accepted_tokens_per_step": gained,
        "timing": timing,
        "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps * (launches_per_step(
            inp, torch.cuda.get_device_properties(device).multi_processor_count) +
            (1 if rejection else 0)),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "kernel": "spec_verify_attn (attention + split-KV combine), K calls back "
                               "to back between one event pair",
                     "peak_source": peak_kind, "attn_ms": attn_ms, "accept_ms": acc_ms,
                     "attn_bytes": nbytes["attn"], "step_bytes": nbytes["total"],
                     "accept_GBps": nbytes["accept"] / (acc_ms / 1e3) / 1e9,
                     "step_frac": nbytes["total"] / (ms_per_step / 1e3) / 1e9 / peak},
        "clocks": clocks,
    }
    if rejection:
        line["config"]["accept"] = "rejection sampling (T = 1, SplitMix64 draws, fresh seed per step)"
    if args.num_ctas or args.split_weight:
        line["config"]["num_ctas"] = args.num_ctas
        line["config"]["split_weight"] = args.split_weight
    if args.small_cluster:
        line["config"]["small_cluster"] = args.small_cluster
    if rank == 0 and not args.no_cpu_baseline and not rejection:
        line["cpu_baseline"] = cpu_baseline(inp, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_codec(args, inp):
    """The delta + run-length page codec on the workload's INT8 cache: every
    (page, kv-head) block of K and V encoded and decoded, each timed with CUDA
    events over --steps launches; the round trip is checked first.  Reports
    the decode rate (INT8 bytes produced per second) with the decode's bytes
    moved against the HBM roofline, the encode rate, and the coded size
    relative to the INT8 pages -- the bytes a decode-in-load attention would
    read instead of the INT8 pages."""
    import torch
    from speculative_decoding_verification_attn_gb300 import binding
    s = inp.spec
    if s.kv_dtype != "i8":
        raise SystemExit("--codec needs an INT8-cache workload (e.g. int8kv_70b_layer)")
    binding.load()
    P, D = s.page_size, s.head_dim
    codes = torch.cat([torch.from_numpy(np.ascontiguousarray(c).reshape(-1, P, D))
                       for c in (inp.k_cache, inp.v_cache)]).cuda()
    nblk, n = codes.shape[0], P * D
    pairs = torch.empty((nblk, 2 * n), dtype=torch.uint8, device="cuda")
    npairs = torch.empty(nblk, dtype=torch.int32, device="cuda")
    out = torch.empty_like(codes)
    binding.spec_codec_encode(codes, pairs, npairs)
    binding.spec_codec_decode(pairs, npairs, out)
    torch.cuda.synchronize()
    if not torch.equal(out, codes) or binding.spec_device_error() != 0:
        raise SystemExit("codec round trip failed")
    coded = int(npairs.sum().item()) * 2 + 4 * nblk

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(args.steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.steps / 1e3

    enc_s = timed(lambda: binding.spec_codec_encode(codes, pairs, npairs))
    dec_s = timed(lambda: binding.spec_codec_decode(pairs, npairs, out))
    peak, peak_kind = measured_peaks()
    moved = coded + nblk * n
    line = {"metric": "INT8 page decode rate", "value": nblk * n / dec_s / 1e9, "unit": "GB/s",
            "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "higher_is_better": True,
            "dtype": "u8", "data": "synthetic (the workload generator's INT8 cache)",
            "config": {"workload": s.name + " K and V caches", "blocks": nblk, "page_size": P,
                       "head_dim": D, "int8_bytes": nblk * n,
                       "l2": "coded pages %d MB, decoded %d MB per launch" % (coded >> 20,
                                                                             (nblk * n) >> 20)},
            "coded_over_int8": coded / (nblk * n),
            "encode_ms": enc_s * 1e3, "decode_ms": dec_s * 1e3,
            "encode_GBps": nblk * n / enc_s / 1e9,
            "roofline": {"bound": "hbm", "achieved": moved / dec_s / 1e9, "peak": peak,
                         "unit": "GB/s", "frac": moved / dec_s / 1e9 / peak,
                         "traffic": None, "kernel": "codec_decode_kernel",
                         "peak_source": peak_kind}}
    print(json.dumps(line), flush=True)


def launches_per_step(inp, num_sms: int) -> int:
    """Kernels one step launches (mirrors the library's automatic choice): for
    a bf16 cache (head_dim 128, page size 16..256, up to 128 query rows per
    kv-head) the 128-key tcgen05 kernel and its combine, except that with <=
    16 rows, more (sequence, kv-head) segments than SMs and a block table
    shorter than 3072 keys the warp-MMA kernel, which merges its split-KV
    partials itself; an INT8 cache the 64-key tcgen05 kernel and its combine;
    other shapes the single-pass SIMT kernel when a whole sequence fits its
    shared memory (one launch), else the chunked SIMT kernel and its combine;
    plus the acceptance kernel."""
    s = inp.spec
    G = s.num_q_heads // s.num_kv_heads
    rows = s.num_draft * G
    tc_shape = (s.q_dtype == "bf16" and s.kv_dtype in ("bf16", "i8") and s.head_dim == 128
                and 16 <= s.page_size <= 256 and s.page_size & (s.page_size - 1) == 0)
    many_short = (s.batch * s.num_kv_heads > num_sms
                  and inp.block_table.shape[1] * s.page_size < 3072)
    if tc_shape and s.kv_dtype == "bf16" and rows <= 16 and many_short:
        return 1 + 1
    if tc_shape and rows <= 128:
        return 2 + 1
    lcap = inp.block_table.shape[1] * s.page_size
    rg = min(rows, 64)
    floats = lcap * (s.head_dim + 4) + lcap * s.head_dim + (rg * lcap + 3) // 4 * 4 + \
        rg * s.head_dim + 4 * 512 + rg
    single = lcap <= 4096 and floats * 4 + (lcap // s.page_size + 2) * 4 <= 200 * 1024
    return (1 if single else 2) + 1


def workload_spec(args):
    """The named workload, with the sweep overrides applied."""
    import dataclasses
    spec = WORKLOADS[args.workload]
    if args.ctx is not None:
        spec = dataclasses.replace(spec, ctx=int(args.ctx), name="%s@ctx%d" % (spec.name, args.ctx))
    return spec


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--accept", choices=["greedy", "rejection"], default="greedy",
                    help="acceptance rule of the step (greedy: the headline configuration)")
    ap.add_argument("--codec", action="store_true",
                    help="time the delta + run-length page codec on the workload's INT8 cache "
                         "instead of the step")
    ap.add_argument("--ctx", type=int, default=None,
                    help="sweeps: every sequence's cached context set to this length")
    ap.add_argument("--num-ctas", type=int, default=0,
                    help="sweeps: persistent CTAs of the tensor-core kernels (0 = one per SM)")
    ap.add_argument("--split-weight", type=int, default=0,
                    help="sweeps: SPEC_OPT_SPLIT_WEIGHT (0 = the kernels' default)")
    ap.add_argument("--small-cluster", type=int, default=0,
                    help="sweeps: SPEC_OPT_SMALL_CLUSTER, CTAs per unit of the single-pass "
                         "kernel (0 = automatic, 1 = no cluster)")
    ap.add_argument("--no-overlap", dest="overlap", action="store_false",
                    help="run a step's acceptance after its attention on one stream (default: "
                         "on a second stream beside it)")
    args = ap.parse_args(argv)

    world, rank, local = dist_env()
    if args.impl == "reference":
        if rank == 0:
            run_reference(args, make_inputs(workload_spec(args), args.seed, canary=False), world,
                          rank)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    import __graft_entry__
    __graft_entry__.build()
    inp = make_inputs(workload_spec(args), args.seed, canary=False)
    if args.num_ctas or args.split_weight or args.small_cluster:
        from speculative_decoding_verification_attn_gb300 import binding
        binding.spec_set_option(binding.SPEC_OPT_NUM_CTAS, args.num_ctas)
        binding.spec_set_option(binding.SPEC_OPT_SPLIT_WEIGHT, args.split_weight)
        binding.spec_set_option(binding.SPEC_OPT_SMALL_CLUSTER, args.small_cluster)
    if args.codec:
        if rank == 0:
            run_codec(args, inp)
        return
    run_gpu(args, inp, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
