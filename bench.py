"""Benchmark of the vocab-wide sampling pass (libdsample) -- prints ONE JSON line on rank 0.

Default workload: the throughput configuration -- 64 requests, C = 8 rows, ragged
T ~ U{100..400} positions (P = 15510, 124080 cells), V = 1025, bf16 c and u,
guidance 2, temperature 0.9, top ratio 0.1, seed 2. One step = one ds_sample call
over the whole batch (iteration counter = step index mod 32). Inputs are 510 MB,
far above the 129 MB L2, so no flush is needed between steps.

Besides the contract's keys the line carries, for the headline and (under `also`)
for every other configuration: the roofline of the call, the CPU oracle timed on
a bounded sample of the same workload on this host, and parity statistics of the
GPU output against the oracle on that sample (computed outside the timed region).
`ms_per_call` adds the median and minimum of 64 single calls, each between its own
pair of events, timed after the contract's region.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload cfg3|cfg5|cfg4|cfg1|cfg2] [--no-extra]

With --gpus N > 1 outside torchrun the script starts N ranks itself (one process
per GPU, torch.distributed.run on 127.0.0.1). Under torchrun every rank runs its
own full batch (weak scaling: cells are independent, no collective on the data
path); the timed region is bracketed by barriers and the max over ranks is
reported. --launch-selftest runs the same launch, timing and reporting path on
CPU ranks (gloo) with a sleep for a step, to check the multi-rank plumbing
without a GPU; its line says so.
"""
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

import numpy as np  # noqa: E402
import torch  # noqa: E402

FALLBACK_HBM_GBS = 6800.0
# The sources that define each workload's kernels and their launch plan: its
# committed DRAM figure stays valid while their code is unchanged.
KERNEL_SOURCES = {
    "cfg3": ["ds_device.cuh", "ds_sample_common.cuh", "ds_warp_common.cuh", "k_sample_warp.cu"],
    "cfg5": ["ds_device.cuh", "ds_sample_common.cuh", "k_sample_stream.cu", "k_sample_cluster.cu"],
    "cfg4": ["ds_device.cuh", "k_greedy.cu"],
}


# ------------------------------------------------------------------------------------- helpers
def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        for key in ("hbm_gbs", "hbm_GBs", "hbm_copy_gbs"):
            if key in d and d[key]:
                return float(d[key]), "measured"
    except (OSError, ValueError):
        pass
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(workload):
    """Hash of the code of a workload's kernel sources: line comments and trailing blanks are
    dropped, so that an edited comment does not retire the committed traffic figures."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[workload]:
        with open(os.path.join(ROOT, "vocab_wide_logit_gb300", "csrc", name), encoding="utf-8") as f:
            for line in f:
                code = line.split("//", 1)[0].rstrip()
                if code:
                    h.update(code.encode("utf-8") + b"\n")
    return h.hexdigest()[:16]


def committed_traffic(workload):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernels."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(workload)
    if not e or e.get("kernel_source_hash") != kernel_source_hash(workload):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], 0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = max(mx, float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def make_workload(name):
    from vocab_wide_logit_gb300 import workloads as wl
    if name == "cfg4":
        return wl.config4()
    return wl.SAMPLE_CONFIGS[name]()


class SampleRunner:
    def __init__(self, inp, dev):
        import vocab_wide_logit_gb300 as pkg
        self.pkg = pkg
        self.inp = inp
        self.rid = torch.from_numpy(inp.request_ids).to(dev)
        self.sl = torch.from_numpy(inp.seq_lens.astype(np.int32)).to(dev)
        self.g = torch.from_numpy(inp.guidance).to(dev)
        self.tau = torch.from_numpy(inp.temperature).to(dev)
        self.c = inp.c_logits.to(dev)
        self.u = inp.u_logits.to(dev) if inp.u_logits is not None else None
        self.tok = torch.empty((inp.C, inp.P), dtype=torch.int32, device=dev)
        self.lp = torch.empty((inp.C, inp.P), dtype=torch.float32, device=dev)

    def step(self, i):
        self.pkg.ds_sample(self.rid, self.c, self.u, self.sl, self.g, self.tau, self.inp.top_ratio,
                           self.inp.seed, i % 32, self.tok, self.lp)

    units = property(lambda self: self.inp.cells)
    bytes_per_step = property(lambda self: self.inp.algorithmic_bytes())


class GreedyRunner:
    """Rotates 4 input buffers (4 x 127 MB > L2) so that no call is served from L2."""

    def __init__(self, g, dev, n_buf=4):
        import vocab_wide_logit_gb300 as pkg
        self.pkg = pkg
        self.g = g
        base = g.logits.to(dev)
        self.bufs = [base] + [base.roll(j + 1, dims=0).contiguous() for j in range(n_buf - 1)]
        self.mx = torch.empty(g.n, dtype=torch.float32, device=dev)
        self.lse = torch.empty(g.n, dtype=torch.float32, device=dev)
        self.am = torch.empty(g.n, dtype=torch.int32, device=dev)

    def step(self, i):
        self.pkg.ds_greedy_lse(self.bufs[i % len(self.bufs)], self.mx, self.lse, self.am)

    units = property(lambda self: self.g.n)
    bytes_per_step = property(lambda self: self.g.algorithmic_bytes())


class DeviceTimer:
    """CUDA events on the current stream (the stream every launch goes to)."""

    def start(self):
        torch.cuda.synchronize()
        self.e0 = torch.cuda.Event(enable_timing=True)
        self.e1 = torch.cuda.Event(enable_timing=True)
        self.e0.record(torch.cuda.current_stream())

    def stop(self):
        self.e1.record(torch.cuda.current_stream())
        torch.cuda.synchronize()
        return self.e0.elapsed_time(self.e1)


class HostTimer:
    """Wall clock, for the CPU (gloo) test of the multi-rank logic."""

    def start(self):
        self.t0 = time.perf_counter()

    def stop(self):
        return (time.perf_counter() - self.t0) * 1e3


def max_over_ranks(ms, world, device):
    """Largest per-rank time of the timed region (rank clocks are independent)."""
    if world <= 1:
        return ms
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def time_steps(runner, steps, warmup, world, timer=None, device="cuda", counter=None):
    """W untimed steps, then exactly K timed steps bracketed by a barrier and a device
    synchronisation on both sides; returns ms per step, the max over ranks. With a launch
    counter (the library's ds_launch_count), the kernels launched inside the timed region
    are left in runner.timed_launches."""
    timer = timer or DeviceTimer()
    for i in range(warmup):
        runner.step(i)
    if device == "cuda":
        torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    c0 = counter() if counter else 0
    timer.start()
    for i in range(steps):
        runner.step(warmup + i)
    ms = timer.stop()
    if counter:
        runner.timed_launches = counter() - c0
    ms = max_over_ranks(ms, world, device)
    if world > 1:
        torch.distributed.barrier()
    return ms / steps


class PerRequestRunner:
    """Config 3 through ds_sample_ex: per-request top ratios drawn from {0.05, 0.1, 0.2} and
    per-request iteration counters (the sampling buffers of a SampleRunner)."""

    def __init__(self, base, dev):
        self.b = base
        rng = np.random.Generator(np.random.PCG64(12))
        B = base.inp.B
        self.ratios = torch.from_numpy(rng.choice(np.array([0.05, 0.1, 0.2], np.float32), size=B)).to(dev)
        self.iters = torch.from_numpy(rng.integers(0, 1 << 20, size=B).astype(np.int32)).to(dev)

    def step(self, i):
        b = self.b
        b.pkg.ds_sample(b.rid, b.c, b.u, b.sl, b.g, b.tau, b.inp.top_ratio, b.inp.seed, 0, b.tok, b.lp,
                        top_ratios=self.ratios, iterations=self.iters)

    units = property(lambda self: self.b.inp.cells)
    bytes_per_step = property(lambda self: self.b.inp.algorithmic_bytes())


class RevealRunner:
    """Confidence ranking and reveal on one config-3 sampling step: every request commits a tenth
    of its C x T cells (score = the step's logprob)."""

    def __init__(self, base, dev):
        b = base
        b.step(0)
        torch.cuda.synchronize()
        self.b = b
        self.scores = b.lp.clone()
        self.tokens = b.tok.clone()
        counts = np.ceil(0.1 * b.inp.C * b.inp.seq_lens.astype(np.float64)).astype(np.int32)
        self.counts = torch.from_numpy(counts).to(dev)
        self.canvas = torch.full((b.inp.C, b.inp.P), -1, dtype=torch.int32, device=dev)
        self.revealed = torch.empty((b.inp.C, b.inp.P), dtype=torch.uint8, device=dev)
        self.n_rev = int(counts.sum())

    def step(self, i):
        self.b.pkg.ds_reveal(self.scores, self.tokens, self.b.sl, self.counts, self.canvas, self.revealed)

    units = property(lambda self: self.b.inp.cells)
    # scores read, revealed tokens read and written to the canvas, one flag byte per cell
    bytes_per_step = property(lambda self: 5 * self.b.inp.cells + 8 * self.n_rev)


class LogSoftmaxRunner:
    """Dense log-softmax of the config-4 rows (rotating input buffers), fp32 or bf16 out."""

    def __init__(self, greedy, dtype):
        self.g = greedy
        n, V = greedy.g.n, greedy.g.V
        self.out = torch.empty((n, V), dtype=dtype, device=greedy.mx.device)
        self.osize = 4 if dtype == torch.float32 else 2

    def step(self, i):
        g = self.g
        g.pkg.ds_log_softmax(g.bufs[i % len(g.bufs)], self.out, g.mx, g.lse, g.am)

    units = property(lambda self: self.g.g.n)
    bytes_per_step = property(lambda self: self.g.g.n * ((2 + self.osize) * self.g.g.V + 12))


class MergeRunner:
    """Merge of vocabulary-shard triples: 16384 tokens x 8 shards (max, lse, global argmax bits)."""

    def __init__(self, pkg, dev, n=16384, shards=8):
        self.pkg = pkg
        rng = np.random.Generator(np.random.PCG64(13))
        t = np.empty((n, shards, 3), np.float32)
        t[..., 0] = rng.normal(0.0, 4.0, size=(n, shards))
        t[..., 1] = t[..., 0] + np.log(rng.uniform(1.0, 3e4, size=(n, shards)))
        t[..., 2] = rng.integers(0, 248320, size=(n, shards)).astype(np.int32).view(np.float32)
        self.t = torch.from_numpy(t).to(dev)
        self.mx = torch.empty(n, dtype=torch.float32, device=dev)
        self.lse = torch.empty(n, dtype=torch.float32, device=dev)
        self.am = torch.empty(n, dtype=torch.int32, device=dev)
        self.n, self.shards = n, shards

    def step(self, i):
        self.pkg.ds_merge_triples(self.t, self.mx, self.lse, self.am)

    units = property(lambda self: self.n)
    bytes_per_step = property(lambda self: self.n * (12 * self.shards + 12))


def next_row_entry(runner, steps, warmup, workload, note):
    """Device time and HBM roofline of one next-row entry point (same timing rules as the main line),
    and the per-call device time from a CUDA-graph replay (latency-bound calls are otherwise timed at
    the host's issue rate)."""
    ms = time_steps(runner, steps, warmup, 1)
    peak, src = hbm_peak()
    gbs = runner.bytes_per_step / (ms / 1e3) / 1e9
    return {"workload": workload, "ms_per_call": round(ms, 5), "ms_per_call_graph": graph_call_ms(runner),
            "units_per_s": round(runner.units / (ms / 1e3), 1),
            "algorithmic_bytes_per_call": runner.bytes_per_step, "achieved_gbs": round(gbs, 1),
            "frac": round(gbs / peak, 4), "peak": peak, "peak_source": src, "note": note}


def graph_call_ms(runner, calls=20, reps=5):
    """Device time per call with the host out of the way: `calls` calls captured in one CUDA graph
    and replayed (each call's launches and their programmatic dependencies become graph nodes), so
    a latency-bound call is not timed at the rate the host can issue it. Median over replays."""
    st = torch.cuda.Stream()
    runner.step(0)  # launch settings are looked up and kept before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g, stream=st):
            for i in range(calls):
                runner.step(i)
    except RuntimeError as e:  # reported, not fatal: the stream-issued numbers stand
        torch.cuda.synchronize()
        return "graph capture failed: %s" % str(e).splitlines()[0][:200]
    t = []
    with torch.cuda.stream(st):  # replay and its events on one stream
        g.replay()
        torch.cuda.synchronize()
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(st)
            g.replay()
            b.record(st)
            torch.cuda.synchronize()
            t.append(a.elapsed_time(b) / calls)
    return round(statistics.median(t), 5)


def per_call_ms(runner, calls, first_step):
    """Median and minimum device time of single calls, one event pair per call, taken after
    (and apart from) the timed region so that its events do not perturb the contract's number."""
    st = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(ev):
        a.record(st)
        runner.step(first_step + i)
        b.record(st)
    torch.cuda.synchronize()
    t = sorted(a.elapsed_time(b) for a, b in ev)
    return {"median": round(statistics.median(t), 5), "min": round(t[0], 5), "calls": calls}


def dominant_kernel(w):
    """The kernel that carries a call (mirrors the library's dispatch: the warp-per-cell kernel up
    to V = 2055; the streaming kernel, in one or two launches, plus its fix-up pass when 4k <= V;
    the staged cluster kernel otherwise; the greedy kernel)."""
    if not hasattr(w, "top_ratio"):
        return "k_greedy_lse"
    if w.V <= 2055:
        return "k_sample_warp"
    import vocab_wide_logit_gb300 as pkg
    k = pkg.top_k(w.top_ratio, w.V)
    return "k_sample_stream (+ fix-up k_sample_cluster in the same timed step)" \
        if 4 * k <= w.V else "k_sample_cluster"


def oracle_cpu_rate(inp, max_seconds=10.0, iteration=0):
    """Run the CPU oracle (single thread) on a bounded sample of the workload's cells.
    Returns (cells per second, sample description, cells, oracle outputs on those cells)."""
    import oracle
    from vocab_wide_logit_gb300 import workloads as wl
    cb = wl.bf16_bits(inp.c_logits)
    ub = wl.bf16_bits(inp.u_logits) if inp.u_logits is not None else None
    n = inp.cells
    # calibrate on a small strided sample, then size the timed sample to about max_seconds
    cal = np.arange(0, n, max(1, n // 200), dtype=np.int64)
    t0 = time.perf_counter()
    oracle.sample_cells(inp.request_ids, cb, ub, inp.seq_lens, inp.C, inp.P, inp.V, inp.guidance,
                        inp.temperature, inp.top_ratio, inp.seed, iteration, cal)
    per = (time.perf_counter() - t0) / len(cal)
    want = int(min(n, max(len(cal), max_seconds / max(per, 1e-9))))
    cells = np.unique(np.linspace(0, n - 1, want).astype(np.int64))
    t0 = time.perf_counter()
    ref = oracle.sample_cells(inp.request_ids, cb, ub, inp.seq_lens, inp.C, inp.P, inp.V, inp.guidance,
                              inp.temperature, inp.top_ratio, inp.seed, iteration, cells)
    dt = time.perf_counter() - t0
    return len(cells) / dt, "%d of %d cells (evenly spaced), iteration %d" % (len(cells), n, iteration), cells, ref


def oracle_cpu_rate_greedy(g, max_seconds=10.0):
    import oracle
    from vocab_wide_logit_gb300 import workloads as wl
    bits = wl.bf16_bits(g.logits)
    t0 = time.perf_counter()
    oracle.greedy_rows(bits, g.n, g.V, np.arange(min(4, g.n), dtype=np.int64))
    per = (time.perf_counter() - t0) / min(4, g.n)
    want = int(min(g.n, max(1, max_seconds / max(per, 1e-9))))
    rows = np.arange(want, dtype=np.int64)
    t0 = time.perf_counter()
    ref = oracle.greedy_rows(bits, g.n, g.V, rows)
    dt = time.perf_counter() - t0
    return want / dt, "%d of %d rows" % (want, g.n), rows, ref


NEAR_TIE_REL = 1e-5


def sample_parity(runner, iteration, cells, ref):
    """GPU output of one call at `iteration` against the oracle on the sampled cells: tokens
    bit-exact except near-ties (the two best perturbed scores, oracle side, within 1e-5 relative),
    |delta logprob| on the matching cells."""
    runner.step(iteration)
    torch.cuda.synchronize()
    tok = runner.tok.cpu().numpy().reshape(-1)[cells]
    lp = runner.lp.cpu().numpy().reshape(-1)[cells].astype(np.float64)
    with np.errstate(invalid="ignore"):
        near = np.abs(ref["top1"] - ref["top2"]) < NEAR_TIE_REL * np.maximum(np.abs(ref["top1"]), 1.0)
    match = tok == ref["tokens"]
    fin = match & np.isfinite(ref["logprobs"])
    dl = np.abs(lp[fin] - ref["logprobs"][fin])
    return {"cells": int(len(cells)), "token_mismatches": int((~match & ~near).sum()),
            "near_ties": int(near.sum()), "near_tie_mismatches": int((~match & near).sum()),
            "max_dlogprob": float(dl.max()) if dl.size else 0.0}


def greedy_parity(runner, rows, ref):
    runner.step(0)
    torch.cuda.synchronize()
    mx = runner.mx.cpu().numpy()[rows]
    am = runner.am.cpu().numpy()[rows]
    lse = runner.lse.cpu().numpy()[rows].astype(np.float64)
    return {"rows": int(len(rows)), "max_mismatches": int((mx != ref["max"]).sum()),
            "argmax_mismatches": int((am != ref["argmax"]).sum()),
            "max_dlse": float(np.abs(lse - ref["lse"]).max())}


def cpu_model():
    """The host CPU's model name (lscpu), for the baseline's record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return None


def baseline_entry(value, unit, sample):
    return {"value": round(value, 2), "unit": unit, "cores": 1, "kind": "oracle", "sample": sample,
            "host_cpus": os.cpu_count(), "cpu_model": cpu_model()}


def e2e_rate(inp, dev, steps):
    """Through the public API from pinned host memory: every step copies c (and u) host->device,
    samples, and copies (tokens, logprobs) back; steps are pipelined two deep (the next step's copy
    runs while this one samples). Host wall clock over K steps, device synchronised on both sides."""
    from vocab_wide_logit_gb300.api import HostSampler
    hs = HostSampler(torch.from_numpy(inp.request_ids), torch.from_numpy(inp.seq_lens.astype(np.int32)),
                     torch.from_numpy(inp.guidance), torch.from_numpy(inp.temperature), inp.C, inp.P, inp.P_u,
                     inp.V, device=dev, depth=2)
    c_h = inp.c_logits.pin_memory()
    u_h = inp.u_logits.pin_memory() if inp.u_logits is not None else None
    for i in range(3):
        hs(c_h, u_h, inp.top_ratio, inp.seed, i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    slots = [hs.submit(c_h, u_h, inp.top_ratio, inp.seed, i % 32) for i in range(steps)]
    for s in slots[-hs.depth:]:
        hs.result(s)
    torch.cuda.synchronize()
    ms = (time.perf_counter() - t0) * 1e3 / steps
    return inp.cells / (ms / 1e3), hs.h2d_bytes(), hs.d2h_bytes(), ms


def roofline(bytes_per_step, ms, workload, kernel=None):
    """achieved = algorithmic bytes of one call / its device time (CUDA events around the
    call's launches, averaged over the timed steps)."""
    peak, src = hbm_peak()
    ach = bytes_per_step / (ms / 1e3) / 1e9
    return {"bound": "hbm", "kernel": kernel, "achieved": round(ach, 1), "peak": peak, "peak_source": src,
            "unit": "GB/s", "frac": round(ach / peak, 4), "frac_of_8000": round(ach / 8000.0, 4),
            "traffic": committed_traffic(workload) if workload in KERNEL_SOURCES else None,
            "algorithmic_bytes_per_launch": bytes_per_step}


def metric_name(is_greedy):
    return ("greedy rows/s (max/LSE/argmax, V=248320)" if is_greedy else
            "sampled positions/s (fused CFG + top-ratio + Gumbel, HBM roofline fraction alongside)")


def run_config(w, is_greedy, world):
    """The workload description both arms report (the reference arm times the same workload)."""
    return {"workload": w.name, "units_per_gpu_step": w.n if is_greedy else w.cells,
            "bytes_per_gpu_step": w.algorithmic_bytes(),
            "l2": "4 rotating input buffers, 508 MB total > L2" if is_greedy else
                  ("inputs larger than L2 (no flush)" if w.algorithmic_bytes() > 129e6 else
                   "inputs smaller than L2 (a latency-bound call: L2-resident after the first step)"),
            "parallelism": "dp%d (independent cells per rank)" % world}


def config_entry(name, dev, steps, warmup, cpu_seconds):
    """Device time, roofline, the oracle timed on a bounded sample, and parity on that sample,
    for one configuration (rank 0, N = 1)."""
    w = make_workload(name)
    is_greedy = name == "cfg4"
    runner = GreedyRunner(w, dev) if is_greedy else SampleRunner(w, dev)
    ms = time_steps(runner, steps, warmup, 1)
    unit = "rows/s" if is_greedy else "sampled positions/s"
    e = {"workload": w.name, "ms_per_step": round(ms, 5), "us_per_step": round(ms * 1e3, 2),
         "ms_per_call": per_call_ms(runner, 64, warmup + steps),
         "us_per_call_graph": round(1e3 * graph_call_ms(runner), 2),
         "units_per_s": round(runner.units / (ms / 1e3), 1), "unit": unit,
         "roofline": roofline(runner.bytes_per_step, ms, name, dominant_kernel(w))}
    if is_greedy:
        cv, sample, rows, ref = oracle_cpu_rate_greedy(w, cpu_seconds)
        e["parity"] = greedy_parity(runner, rows, ref)
    else:
        cv, sample, cells, ref = oracle_cpu_rate(w, cpu_seconds)
        e["parity"] = sample_parity(runner, 0, cells, ref)
    e["cpu_baseline"] = baseline_entry(cv, unit, sample)
    return e, runner


# ------------------------------------------------------------------------------------- arms
def run_ours(args):
    rank, world, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import vocab_wide_logit_gb300 as pkg
    pkg.load()
    wname = args.workload
    w = make_workload(wname)
    is_greedy = wname == "cfg4"
    runner = GreedyRunner(w, dev) if is_greedy else SampleRunner(w, dev)
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(dev.index)).split(",")[dev.index]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES") else dev.index
    with ClockSampler(gpu_index) as clk:
        ms = time_steps(runner, args.steps, args.warmup, world, counter=pkg.launch_count)
    clocks = clk.summary()
    units = runner.units * world
    value = units / (ms / 1e3)
    unit = "rows/s" if is_greedy else "sampled positions/s"
    line = {
        "metric": metric_name(is_greedy),
        "value": round(value, 1), "unit": unit, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (seeded, bf16 inputs)",
        "config": run_config(w, is_greedy, world),
        "roofline": roofline(runner.bytes_per_step, ms, wname, dominant_kernel(w)),
        "gpu_launches": runner.timed_launches,
        "clocks": clocks,
    }
    if rank == 0 and not is_greedy:
        line["logit_elements_per_s"] = round(value * w.V, 1)
    if rank == 0:
        line["ms_per_call"] = per_call_ms(runner, 64, args.warmup + args.steps)
        # end to end through the public API, from pinned host memory
        if not is_greedy:
            ev, hb, db, ems = e2e_rate(w, dev, max(4, min(args.steps, 12)))
            line["e2e"] = {"value": round(ev * world, 1), "unit": unit, "h2d_bytes_per_step": hb,
                           "d2h_bytes_per_step": db, "ms_per_step": round(ems, 4),
                           "pipeline": "2 deep: next step's host->device copy overlaps this step's sampling"}
        # the oracle on this host, bounded sample, and parity on that sample (N = 1 only)
        if world == 1:
            if is_greedy:
                cv, sample, rows, ref = oracle_cpu_rate_greedy(w, args.cpu_seconds)
                line["parity"] = greedy_parity(runner, rows, ref)
            else:
                cv, sample, cells, ref = oracle_cpu_rate(w, args.cpu_seconds)
                line["parity"] = sample_parity(runner, 0, cells, ref)
            line["cpu_baseline"] = baseline_entry(cv, unit, sample)
        if not args.no_extra and wname == "cfg3" and world == 1:
            extra = {}
            nsteps = max(10, min(args.steps, 500))
            # the next rows built on the path, on the resident config-3 buffers
            nxt = {
                "f2_per_request": next_row_entry(
                    PerRequestRunner(runner, dev), nsteps, args.warmup,
                    "cfg3 via ds_sample_ex: per-request ratios in {0.05, 0.1, 0.2} and iterations",
                    "same kernels as the main line; inputs larger than L2"),
                "f1_reveal": next_row_entry(
                    RevealRunner(runner, dev), nsteps, args.warmup,
                    "ds_reveal on one cfg3 step: 64 requests, C = 8, each commits 10% of its cells",
                    "L2-resident scores: latency-bound"),
            }
            del runner
            torch.cuda.empty_cache()
            for other in ("cfg1", "cfg2", "cfg5", "cfg4"):
                osteps = max(10, min(args.steps, 1500))
                extra[other], orunner = config_entry(other, dev, osteps, args.warmup, args.cpu_seconds_other)
                if other == "cfg4":
                    for dt, nm in ((torch.float32, "f4_log_softmax_f32"), (torch.bfloat16, "f4_log_softmax_bf16")):
                        nxt[nm] = next_row_entry(
                            LogSoftmaxRunner(orunner, dt), nsteps, args.warmup,
                            "ds_log_softmax on the cfg4 rows (256 x 248320), %s out" % str(dt).split(".")[-1],
                            "one read of the logits and one dense write; 4 rotating inputs")
                    nxt["f3_merge_triples"] = next_row_entry(
                        MergeRunner(orunner.pkg, dev), nsteps, args.warmup,
                        "ds_merge_triples: 16384 tokens x 8 shards", "1.6 MB, L2-resident: launch-bound")
                del orunner
                torch.cuda.empty_cache()
            extra["next_rows"] = nxt
            line["also"] = extra
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_reference(args):
    """The CPU oracle, as it stands, on this host's cores: each step samples a bounded slice of
    the same workload; rank 0 alone under torchrun."""
    rank, world, local = dist_env()
    if rank != 0:
        return
    wname = args.workload
    w = make_workload(wname)
    is_greedy = wname == "cfg4"
    unit = "rows/s" if is_greedy else "sampled positions/s"
    budget = max(1.0, args.ref_seconds_per_step)
    rates = []
    sample = ""
    for i in range(args.warmup + args.steps):
        if is_greedy:
            r, sample, _, _ = oracle_cpu_rate_greedy(w, budget)
        else:
            r, sample, _, _ = oracle_cpu_rate(w, budget, iteration=i % 32)
        if i >= args.warmup:
            rates.append(r)
    value = statistics.median(rates)
    line = {"impl": "reference", "metric": metric_name(is_greedy),
            "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic (seeded, bf16 inputs)",
            "config": run_config(w, is_greedy, world),
            "cpu_baseline": baseline_entry(value, unit, sample + " per step"),
            "e2e": {"value": round(value, 2), "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)


class _SleepStep:
    """Launcher self-test step: 2 ms x (rank + 1) of wall time (no GPU work)."""

    def __init__(self, rank):
        self.rank = rank

    def step(self, i):
        time.sleep(0.002 * (self.rank + 1))

    units = 1


def run_selftest(args):
    """The launch, timing and reporting path on CPU ranks (gloo), with a sleep for a step."""
    rank, world, local = dist_env()
    if world > 1:
        torch.distributed.init_process_group("gloo")
    r = _SleepStep(rank)
    ms = time_steps(r, args.steps, args.warmup, world, timer=HostTimer(), device="cpu")
    if rank == 0:
        print(json.dumps({"selftest": True, "metric": "launcher self-test (sleep steps, no GPU work)",
                          "value": round(world * r.units / (ms / 1e3), 3), "unit": "steps/s", "n_gpus": world,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4)}), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def spawn_command(args, argv):
    """Re-run this script under torch.distributed.run with one rank per GPU on this node."""
    import socket
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    return [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(args.gpus),
            "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + argv


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["cfg3", "cfg5", "cfg4", "cfg1", "cfg2"], default="cfg3")
    ap.add_argument("--no-extra", action="store_true", help="skip the other configurations under 'also'")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle budget for the headline workload")
    ap.add_argument("--cpu-seconds-other", type=float, default=4.0, help="oracle budget per other configuration")
    ap.add_argument("--ref-seconds-per-step", type=float, default=3.0)
    ap.add_argument("--launch-selftest", action="store_true", help="multi-rank plumbing on CPU (gloo), no GPU work")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(subprocess.call(spawn_command(args, sys.argv[1:])))
    if args.launch_selftest:
        run_selftest(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
