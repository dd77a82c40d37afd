"""Benchmark of the MXFP8 decode projection with its mailbox publish/consume.

One step = one call of the whole path on the N=7168, K=16384, m=8, S=4
workload: the publishing GEMM followed by the PDL consumer (generation
handed over, slots polled, copied out and reset).  The headline is the
weight-stream bandwidth: (N*K + N*K/32) bytes per call / time per call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Timed region: exactly W untimed steps, then exactly K steps, replayed from
CUDA graphs of chained calls that rotate through enough weight copies (more
than 12 x the 129 MB L2) that every call streams its weight from HBM; CUDA
events on the launching stream, barrier + synchronize on both sides, max
over ranks.  nvidia-smi samples the clocks from the timed region through at
least two seconds of the same calls right after it, while the CPU baseline
(the oracle on the host cores) runs.  The same line reports the GEMM alone
(the roofline), the end-to-end figure from pinned host buffers, and the
other workloads of the path (N=7168 K=8192 m=8 S=2, N=4096 K=4096 m=4 S=1,
N=256 K=256 m=1 S=1), each with its own weight rotation.
Under torchrun every rank runs an independent replica on its own GPU (the
path does not shard); ``value`` is the weight bytes all ranks streamed / the
slowest rank's time.  The reference arm times the CPU oracle on a bounded
sample of the workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from pathlib import Path

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

METRIC = "us/call and weight-stream HBM GB/s (% of GB300 peak), MXFP8 GEMM m<=8"
UNIT = "GB/s"
L2_BYTES = 129 * 2**20
# Weight bytes the timed loops rotate through, in L2 sizes.  Three copies of
# the N=7168, K=16384 weight (2.8 x L2) let 8-10 % of each call's weight
# bytes come from L2 (ncu over a whole graph replay: lines the GEMM warms in
# L2 with normal priority outlive the evict-first stream until their copy
# comes round again); six (5.6 x L2) still 5 %; fifteen (14 x L2) none.
ROTATION_L2_MULTIPLE = 12
WORKLOAD_CHOICES = {"headline": "HEADLINE", "graph": "GRAPH_8192", "chain": "CHAIN_4096",
                    "tiny": "TINY"}
_WORKLOAD = "headline"
GRAPH_STEPS = 30  # calls per captured graph (a multiple of every weight-copy count)
SOAK_SECONDS = 2.0  # least time the clocks are sampled under the chain's load
GATE_CYCLES = 100_000  # the spin before a timed region: about 50 us at 2 GHz
WORKLOAD_CALLS = 6000  # timed calls of each other workload in the headline's line
E2E_GRAPH_STEPS = 480  # end-to-end steps per captured graph (likewise)
E2E_BATCH = 30         # end-to-end steps per wait on the input copies (divides E2E_GRAPH_STEPS)
FALLBACK_HBM_GBS = 6800.0
KERNEL_SOURCES = ("mxfp8_gemm_mailbox_gb300/csrc/publish_gemm_kernel.cuh",
                  "mxfp8_gemm_mailbox_gb300/csrc/publish_gemm.cu",
                  "mxfp8_gemm_mailbox_gb300/csrc/publish_gemm_fold.cu",
                  "mxfp8_gemm_mailbox_gb300/csrc/publish_gemm_k256.cu",
                  "mxfp8_gemm_mailbox_gb300/csrc/ptx.cuh",
                  "mxfp8_gemm_mailbox_gb300/csrc/abi.cu")
TRAFFIC_FILE = ROOT / "profiles" / "publish_gemm_headline_traffic.json"
CLOCK_QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=60000)
    p.add_argument("--warmup", type=int, default=300)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="budget of the oracle CPU-baseline sample (0: skip it)")
    p.add_argument("--no-workloads", action="store_true",
                   help="leave the other workloads out of the headline's line")
    p.add_argument("--workload", choices=tuple(WORKLOAD_CHOICES), default="headline",
                   help="the chain's workload: headline N=7168 K=16384 m=8 S=4 (default), "
                        "graph N=7168 K=8192 m=8 S=2, chain N=4096 K=4096 m=4 S=1, "
                        "tiny N=256 K=256 m=1 S=1")
    p.add_argument("--profile-graph", action="store_true",
                   help="after the timed region, replay the chain's graph once more between "
                        "cudaProfilerStart and cudaProfilerStop (for ncu's graph profiling)")
    p.add_argument("--cta-k", type=int, default=0, choices=(0, 128, 256),
                   help="sweep: the tactic's K per pipeline stage (0: the library's choice)")
    p.add_argument("--sweep-k", type=str, default="",
                   help="sweep: comma-separated K values to run (default: every K of the sweep)")
    p.add_argument("--path", choices=("chain", "protocols", "sweep"), default="chain",
                   help="chain: the headline (default); protocols: the output hand-off "
                        "protocols on their own (sentinel mailbox, tagged pairs, all-gather); "
                        "sweep: the chain on every m x N x K x S case of the sweep")
    return p.parse_args(argv)


# ----------------------------------------------------------------- ranks
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(seconds: float, units: float, group_initialised: bool):
    """(max seconds over ranks, sum of units over ranks)."""
    if not group_initialised:
        return seconds, units
    import torch
    import torch.distributed as dist

    backend = dist.get_backend()
    dev = torch.device("cuda") if backend == "nccl" else torch.device("cpu")
    t = torch.tensor([seconds], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(group_initialised: bool):
    if group_initialised:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples every 200 ms while the timed region runs."""

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={CLOCK_QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names[1:], f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- helpers
def measured_peak():
    f = ROOT / "MEASURED_PEAKS.json"
    if f.exists():
        try:
            return float(json.loads(f.read_text())["hbm_gbs"]), "measured"
        except (KeyError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def _code_lines(text: str):
    """The lines of a C++ source with // comments and blank lines dropped, so
    that editing a comment or the layout does not mark the kernel as changed."""
    for line in text.splitlines():
        code = line.split("//", 1)[0].rstrip()
        if code:
            yield code


def kernel_source_hash() -> str:
    """A hash of the kernel sources' code, comments and whitespace dropped:
    the key of the recorded DRAM traffic."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        for line in _code_lines((ROOT / rel).read_text()):
            h.update("".join(line.split()).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch of the GEMM from the committed ncu summary, if it
    was taken on the kernel as it is now (the headline workload only)."""
    if _WORKLOAD != "headline" or not TRAFFIC_FILE.exists():
        return None
    try:
        rec = json.loads(TRAFFIC_FILE.read_text())
    except ValueError:
        return None
    if rec.get("kernel_source_sha256_16") != kernel_source_hash():
        return None
    return rec.get("dram_bytes_per_launch")


def workload():
    import synthetic

    return getattr(synthetic, WORKLOAD_CHOICES[_WORKLOAD])


def weight_copies(weight_bytes: int) -> int:
    """Weight copies the timed loops rotate through: enough that their bytes
    exceed ROTATION_L2_MULTIPLE x the L2, so no call finds another call's
    weight in L2 (at most 30), and a divisor of both graph lengths so every
    replay rotates the same way."""
    need = max(3, -(-ROTATION_L2_MULTIPLE * L2_BYTES // weight_bytes))
    for c in (3, 5, 6, 10, 15, 30):
        if c >= need:
            return c
    return 30


def rotation_note(copies: int, weight_bytes: int) -> str:
    """What the rotation does to L2, for the JSON line."""
    total = copies * weight_bytes
    head = (f"{copies} rotating weight copies ({total >> 20} MiB, "
            f"{total / L2_BYTES:.1f} x the 129 MB L2)")
    if total >= ROTATION_L2_MULTIPLE * L2_BYTES:
        return head + ": no call finds another call's weight in L2; every call reads its " \
                      "weight from HBM"
    if total >= 2 * L2_BYTES:
        return head + ": weights stream from HBM, though lines warmed in L2 can outlive a " \
                      "rotation"
    return head + ": the weights stay in L2; a latency figure, not a bandwidth one"


# ------------------------------------------------------------ CPU oracle
class OracleSample:
    """The oracle's whole chain (FP64 GEMM, publish, consume) on the first
    ``columns`` output columns and the first ``k`` of K (all m rows)."""

    def __init__(self, columns: int, k: int | None = None):
        import oracle
        import synthetic

        wl = workload()
        columns = min(columns, wl.n)
        self.columns = columns
        self.k = k or wl.k
        sub = synthetic.Workload(wl.name, columns, self.k, wl.m, wl.split_k, wl.capacity,
                                 wl.exp_lo, wl.exp_hi, wl.x_zero_fraction, wl.signed_pairs,
                                 wl.seed)
        self.weight_bytes = sub.weight_bytes
        self.w, self.ws = synthetic.make_weights(sub)
        self.x, self.xs = synthetic.make_activations(sub)
        self.mb = oracle.Mailbox(wl.capacity, columns)
        self.ok = oracle.OK

    def call(self) -> float:
        t0 = time.perf_counter()
        st, _, _ = self.mb.chain(self.w, self.ws, self.x, self.xs, want_c=False)
        t1 = time.perf_counter()
        if st != self.ok:
            raise RuntimeError(f"oracle chain status {st}")
        return t1 - t0

    def describe(self, calls: int) -> str:
        wl = workload()
        return (f"{calls} oracle calls (FP64 GEMM + publish + consume, one thread) on the first "
                f"{self.columns} of {wl.n} output columns and {self.k} of K={wl.k}, m={wl.m}: "
                f"{self.weight_bytes} weight bytes per call")


def oracle_baseline(seconds_budget: float, columns: int = 1024):
    """(GB/s of weight stream, calls, seconds, sample text) of the oracle
    repeated on a column slice until the budget is spent."""
    sample = OracleSample(columns)
    calls, total = 0, 0.0
    while total < seconds_budget or calls == 0:
        total += sample.call()
        calls += 1
    return sample.weight_bytes * calls / total / 1e9, calls, total, sample.describe(calls)


def oracle_baseline_all_cores(seconds_budget: float, columns: int = 1024):
    """The same oracle chain on every host core at once: one thread per core,
    each repeating the call on its own copy of the column slice (the oracle's
    C routines run with the interpreter lock released).  Returns (GB/s of
    weight stream over all threads, threads, calls, wall seconds)."""
    from concurrent.futures import ThreadPoolExecutor

    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    samples = [OracleSample(columns) for _ in range(threads)]

    def worker(sample):
        calls, start = 0, time.perf_counter()
        while calls == 0 or time.perf_counter() - start < seconds_budget:
            sample.call()
            calls += 1
        return calls

    t0 = time.perf_counter()
    with ThreadPoolExecutor(max_workers=threads) as pool:
        counts = list(pool.map(worker, samples))
    wall = time.perf_counter() - t0
    calls = sum(counts)
    return samples[0].weight_bytes * calls / wall / 1e9, threads, calls, wall


# -------------------------------------------------------------- our arm
class Chain:
    """The chained calls of one workload (publishing GEMM, then the PDL
    consumer), rotating through enough weight copies that every call streams
    its weight from HBM: the copies, one handle each, one mailbox, and CUDA
    graphs of GRAPH_STEPS chained calls (plus graphs of fewer calls, captured
    on demand, so any step count can be issued exactly)."""

    def __init__(self, wl, device, stream):
        import torch

        import mxfp8_gemm_mailbox_gb300 as mx
        import synthetic

        self.wl, self.device, self.stream = wl, device, stream
        w, ws = synthetic.make_weights(wl)
        x, xs = synthetic.make_activations(wl)
        self.host_x, self.host_xs = x, xs
        W0 = torch.from_numpy(w).to(device)
        WS = torch.from_numpy(ws).to(device)
        self.X = torch.from_numpy(x).to(device)
        self.XS = torch.from_numpy(xs).to(device)
        self.copies = weight_copies(wl.weight_bytes)
        weights = [W0] + [W0.clone() for _ in range(self.copies - 1)]
        self.mb = mx.Mailbox(wl.capacity, wl.n, device=device)
        self.gemms = [mx.PublishGemm(Wc, WS, self.mb, split_k=wl.split_k) for Wc in weights]
        self.cfg = self.gemms[0].config()
        for g in self.gemms:
            g.precompile(wl.m)
        self.out = torch.empty((wl.m, wl.n), dtype=torch.bfloat16, device=device)
        with torch.cuda.stream(stream):
            for i in range(self.copies):  # eager: every handle's first run before capture
                self.gemms[i].run(self.X, self.XS)
                self.mb.consume(wl.m, self.out)
        stream.synchronize()
        self._graphs = {}

    def graph(self, steps: int):
        """The captured graph of `steps` chained calls (steps <= GRAPH_STEPS)."""
        import torch

        if steps not in self._graphs:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.stream(self.stream):
                with torch.cuda.graph(graph, stream=self.stream):
                    for i in range(steps):
                        self.gemms[i % self.copies].run(self.X, self.XS)
                        self.mb.consume(self.wl.m, self.out)
            self._graphs[steps] = graph
        return self._graphs[steps]

    def prepare(self, *step_counts):
        """Captures every graph that issue() will need for these counts and
        replays each once, so no graph's first launch (which uploads it to
        the device) falls inside a timed region."""
        import torch

        counts = {GRAPH_STEPS} | {n % GRAPH_STEPS for n in step_counts if n % GRAPH_STEPS}
        with torch.cuda.stream(self.stream):
            for n in sorted(counts):
                self.graph(n).replay()
        self.stream.synchronize()

    def issue(self, steps: int):
        """Exactly `steps` chained calls on the stream, from the graphs."""
        import torch

        whole, rest = divmod(steps, GRAPH_STEPS)
        with torch.cuda.stream(self.stream):
            for _ in range(whole):
                self.graph(GRAPH_STEPS).replay()
            if rest:
                self.graph(rest).replay()

    def timed(self, steps: int) -> float:
        """Seconds of `steps` chained calls between CUDA events on the stream.
        A short spin kernel (about 50 us) holds the stream before the start
        event, so the host has queued the first graph by the time the event
        is reached: the device-side time then holds the calls' own work, not
        the host's launch of the first graph onto an idle stream."""
        import torch

        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            torch.cuda._sleep(GATE_CYCLES)
        e0.record(self.stream)
        self.issue(steps)
        e1.record(self.stream)
        self.stream.synchronize()
        return e0.elapsed_time(e1) / 1e3

    def soak(self, min_seconds: float, until=None):
        """Whole graphs back to back for at least `min_seconds` and until
        `until()` is false, at most 64 replays in flight.  Returns (calls,
        seconds) between CUDA events."""
        import torch

        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        marks = []
        replays = 0
        t0 = time.perf_counter()
        e0.record(self.stream)
        with torch.cuda.stream(self.stream):
            while (time.perf_counter() - t0 < min_seconds or (until is not None and until())
                   or replays == 0):
                self.graph(GRAPH_STEPS).replay()
                replays += 1
                ev = torch.cuda.Event()
                ev.record(self.stream)
                marks.append(ev)
                if len(marks) > 64:
                    marks.pop(0).synchronize()
        e1.record(self.stream)
        self.stream.synchronize()
        return replays * GRAPH_STEPS, e0.elapsed_time(e1) / 1e3

    def gemm_back_to_back_us(self, launches: int, warm: int = 3) -> float:
        """The publishing GEMM alone (publish off: the same kernel, no consume
        needed), GRAPH_STEPS launches per graph over the rotating weights."""
        import torch

        cbuf = torch.empty((self.wl.m, self.wl.n), dtype=torch.bfloat16, device=self.device)
        graph = torch.cuda.CUDAGraph()
        replays = max(1, launches // GRAPH_STEPS)
        with torch.cuda.stream(self.stream):
            with torch.cuda.graph(graph, stream=self.stream):
                for i in range(GRAPH_STEPS):
                    self.gemms[i % self.copies].run_unfused(self.X, self.XS, cbuf)
            for _ in range(warm):
                graph.replay()
            g0 = torch.cuda.Event(enable_timing=True)
            g1 = torch.cuda.Event(enable_timing=True)
            g0.record(self.stream)
            for _ in range(replays):
                graph.replay()
            g1.record(self.stream)
        self.stream.synchronize()
        return g0.elapsed_time(g1) * 1e3 / (replays * GRAPH_STEPS)

    def isolated_us(self, launches: int) -> float:
        """The GEMM launched alone: CUDA events around each launch, so launch
        and ramp-up are included; each followed by its consume."""
        import torch

        starts = [torch.cuda.Event(enable_timing=True) for _ in range(launches)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(launches)]
        with torch.cuda.stream(self.stream):
            for i in range(launches):
                starts[i].record(self.stream)
                self.gemms[i % self.copies].run(self.X, self.XS)
                ends[i].record(self.stream)
                self.mb.consume(self.wl.m, self.out)
        self.stream.synchronize()
        return statistics.mean(a.elapsed_time(b) * 1e3 for a, b in zip(starts, ends))

    def check(self):
        import mxfp8_gemm_mailbox_gb300 as mx

        status, words = self.mb.status(self.stream)
        if status != mx.OK:
            raise RuntimeError(f"mailbox status {status} after the run: state {words}")

    def close(self):
        for g in self.gemms:
            g.close()
        self.gemms = []
        self._graphs = {}


def end_to_end(chain, steps: int):
    """The same chain through the public API from pinned host buffers: every
    step copies its own x and x scales in (one stream) and its output out
    (another stream).  An event edge inside the chain of kernels cuts the
    programmatic launch between a consumer and the next GEMM (about 6 us per
    step, measured), so the compute stream waits on the input copies once per
    batch of E2E_BATCH steps: batch j+1's inputs land while batch j computes,
    and each step's output copy forks off right after its consumer.  The
    per-step host work (about twenty launches and stream operations) would
    dominate, so E2E_GRAPH_STEPS steps are captured once and replayed; every
    replay still copies every step's inputs in and its output back.  Returns
    (seconds, steps, h2d bytes per step, d2h bytes per step)."""
    import torch

    wl, device, stream = chain.wl, chain.device, chain.stream
    hx = torch.from_numpy(chain.host_x).pin_memory()
    hxs = torch.from_numpy(chain.host_xs).pin_memory()
    nbuf = 2 * E2E_BATCH
    houts = [torch.empty((wl.m, wl.n), dtype=torch.bfloat16).pin_memory() for _ in range(nbuf)]
    dXs = [torch.empty_like(chain.X) for _ in range(nbuf)]
    dXSs = [torch.empty_like(chain.XS) for _ in range(nbuf)]
    outs = [torch.empty_like(chain.out) for _ in range(nbuf)]
    h2d_stream = torch.cuda.Stream(device=device)
    d2h_stream = torch.cuda.Stream(device=device)
    gemms, copies, mb = chain.gemms, chain.copies, chain.mb

    def e2e_steps(count):
        k = E2E_BATCH
        nbatch = (count + k - 1) // k
        loaded = [torch.cuda.Event() for _ in range(nbatch)]
        computed = [torch.cuda.Event() for _ in range(nbatch)]
        read = [torch.cuda.Event() for _ in range(nbatch)]
        step_done = [torch.cuda.Event() for _ in range(count)]

        def load(j):  # the inputs of batch j, one copy pair per step
            with torch.cuda.stream(h2d_stream):
                if j >= 2:
                    h2d_stream.wait_event(computed[j - 2])  # batch j-2 no longer reads them
                for i in range(j * k, min(count, (j + 1) * k)):
                    dXs[i % nbuf].copy_(hx, non_blocking=True)
                    dXSs[i % nbuf].copy_(hxs, non_blocking=True)
                loaded[j].record(h2d_stream)

        load(0)
        for j in range(nbatch):
            if j + 1 < nbatch:
                load(j + 1)
            with torch.cuda.stream(stream):
                stream.wait_event(loaded[j])
                if j >= 2:
                    stream.wait_event(read[j - 2])  # batch j-2's outputs have left the device
            for i in range(j * k, min(count, (j + 1) * k)):
                b = i % nbuf
                with torch.cuda.stream(stream):
                    gemms[i % copies].run(dXs[b], dXSs[b])
                    mb.consume(wl.m, outs[b])
                    step_done[i].record(stream)
                with torch.cuda.stream(d2h_stream):
                    d2h_stream.wait_event(step_done[i])
                    houts[b].copy_(outs[b], non_blocking=True)
            with torch.cuda.stream(stream):
                computed[j].record(stream)
            with torch.cuda.stream(d2h_stream):
                read[j].record(d2h_stream)

    e2e_steps(4)
    torch.cuda.synchronize(device)
    e2e_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(e2e_graph, stream=stream):
        h2d_stream.wait_stream(stream)
        d2h_stream.wait_stream(stream)
        e2e_steps(E2E_GRAPH_STEPS)
        stream.wait_stream(h2d_stream)
        stream.wait_stream(d2h_stream)
    replays = max(1, steps // E2E_GRAPH_STEPS)
    with torch.cuda.stream(stream):
        for _ in range(2):
            e2e_graph.replay()
    stream.synchronize()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        f0.record(stream)
        for _ in range(replays):
            e2e_graph.replay()
        f1.record(stream)
    stream.synchronize()
    last = (E2E_GRAPH_STEPS - 1) % nbuf
    if not torch.equal(houts[last], outs[last].cpu()):
        raise RuntimeError("the end-to-end output read back differs from the device copy")
    h2d = int(chain.X.numel() + chain.XS.numel())
    d2h = int(chain.out.numel() * chain.out.element_size())
    return f0.elapsed_time(f1) / 1e3, replays * E2E_GRAPH_STEPS, h2d, d2h


def workload_entry(wl, device, stream, peak: float, calls: int = WORKLOAD_CALLS) -> dict:
    """µs per call, weight-stream GB/s and roofline fraction of one workload's
    chain, with its own weight rotation, plus the GEMM alone back to back."""
    import torch

    chain = Chain(wl, device, stream)
    try:
        chain.prepare(calls)
        chain.issue(10 * GRAPH_STEPS)  # warm-up
        seconds = chain.timed(calls)
        gemm_us = chain.gemm_back_to_back_us(calls)
        chain.check()
        us = seconds / calls * 1e6
        gbs = wl.weight_bytes / (us * 1e-6) / 1e9
        gemm_gbs = wl.weight_bytes / (gemm_us * 1e-6) / 1e9
        cfg = chain.cfg
        return {
            "workload": f"N={wl.n} K={wl.k} m={wl.m} S={wl.split_k}",
            "us_per_call": round(us, 3),
            "gbs": round(gbs, 1),
            "frac": round(gbs / peak, 4),
            "gemm_us": round(gemm_us, 3),
            "gemm_gbs": round(gemm_gbs, 1),
            "gemm_frac": round(gemm_gbs / peak, 4),
            "calls": calls,
            "weight_bytes_per_call": wl.weight_bytes,
            "weight_copies": chain.copies,
            "l2": rotation_note(chain.copies, wl.weight_bytes),
            "tactic": {k: cfg[k] for k in ("split_k", "fold", "stages", "pipes", "grid_ctas",
                                           "smem_bytes")},
        }
    finally:
        chain.close()
        del chain
        torch.cuda.synchronize(device)
        torch.cuda.empty_cache()


def run_ours(args):
    import threading

    import torch

    world, rank, local = dist_env()
    group = False
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
        group = True
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)

    wl = workload()
    stream = torch.cuda.Stream(device=device)
    chain = Chain(wl, device, stream)
    cfg = chain.cfg
    steps, warmup = max(1, args.steps), max(3, args.warmup)
    chain.prepare(steps, warmup)

    # Exactly `warmup` untimed steps, then exactly `steps` timed ones.
    chain.issue(warmup)
    stream.synchronize()
    barrier(group)
    torch.cuda.synchronize(device)
    with ClockSampler(local) as clocks:
        local_s = chain.timed(steps)
        barrier(group)
        torch.cuda.synchronize(device)
        # The clocks: the same graphs replayed for at least SOAK_SECONDS right
        # after the timed region, while the CPU baseline (rank 0, one GPU)
        # runs on the host cores, so the sampler sees the GPU under this load.
        cpu = {}
        worker = None
        if rank == 0 and world == 1 and args.cpu_seconds > 0:
            worker = threading.Thread(target=lambda: cpu.update(cpu_baseline(args.cpu_seconds)))
            worker.start()
        soak_calls, soak_s = chain.soak(SOAK_SECONDS,
                                        until=(worker.is_alive if worker is not None else None))
        if worker is not None:
            worker.join()
    if args.profile_graph:
        # One more replay of the timed graph between the CUDA profiler's start
        # and stop, for `ncu --profile-from-start off --graph-profiling graph`:
        # the DRAM bytes of GRAPH_STEPS whole chained calls.
        torch.cuda.profiler.start()
        chain.issue(GRAPH_STEPS)
        stream.synchronize()
        torch.cuda.profiler.stop()
    seconds, bytes_all = aggregate(local_s, float(steps * wl.weight_bytes), group)
    us_per_call = seconds / steps * 1e6
    value = bytes_all / seconds / 1e9

    # The dominant kernel, the publishing GEMM, back to back and alone.
    gemm_us = chain.gemm_back_to_back_us(max(steps, 3000))
    iso_us = chain.isolated_us(min(300, max(steps, 30)))
    peak, peak_kind = measured_peak()
    achieved = wl.weight_bytes / (gemm_us * 1e-6) / 1e9

    e2e_s, n_e2e, h2d, d2h = end_to_end(chain, min(3000, max(steps, E2E_GRAPH_STEPS)))
    e2e_s, e2e_bytes = aggregate(e2e_s, float(n_e2e * wl.weight_bytes), group)
    chain.check()
    chain.close()
    del chain
    torch.cuda.synchronize(device)
    torch.cuda.empty_cache()

    # The other workloads of the path, each with its own rotation.
    workloads = {}
    if _WORKLOAD == "headline" and not args.no_workloads:
        import synthetic

        for name in ("graph", "chain", "tiny"):
            workloads[name] = workload_entry(getattr(synthetic, WORKLOAD_CHOICES[name]), device,
                                             stream, peak)

    if rank == 0:
        traffic = recorded_traffic()
        clock = clocks.summary()
        clock["window"] = (f"the timed region and {soak_s:.2f} s of the same chained calls right "
                           f"after it ({soak_calls} calls, "
                           f"{soak_s / soak_calls * 1e6:.3f} us per call)")
        line = {
            "metric": METRIC,
            "value": round(value, 1),
            "unit": UNIT,
            "n_gpus": world,
            "steps": steps,
            "warmup": warmup,
            "ms_per_step": round(us_per_call / 1e3, 6),
            "us_per_call": round(us_per_call, 3),
            "pct_of_peak": round(100 * (value / world) / peak, 1),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "e4m3",
            "data": "synthetic (seeded N(0,1) E4M3, E8M0 block-32 scales, 1% zero x)",
            "config": {
                "workload": f"decode projection N={wl.n} K={wl.k} m={wl.m} S={wl.split_k} "
                            "+ mailbox publish/consume",
                "n": wl.n, "k": wl.k, "m": wl.m, "split_k": cfg["split_k"],
                "stages": cfg["stages"], "grid_ctas": cfg["grid_ctas"],
                "smem_bytes": cfg["smem_bytes"],
                "weight_bytes_per_call": wl.weight_bytes,
                "l2": rotation_note(weight_copies(wl.weight_bytes), wl.weight_bytes),
                "timing": f"CUDA graphs of {GRAPH_STEPS} chained calls (GEMM -> PDL consumer), "
                          "fewer for a remainder, exactly the steps asked",
                "parallelism": "replicas" if world > 1 else "single GPU",
            },
            "roofline": {
                "bound": "hbm",
                "kernel": f"publish_gemm_kernel<{wl.split_k}, 0, {cfg['fold']}, "
                          f"{(cfg.get('cta_k') or 128) // 128}>",
                "achieved": round(achieved, 1),
                "peak": peak,
                "peak_kind": peak_kind,
                "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": traffic,
                "algorithmic_bytes_per_launch": wl.weight_bytes,
                "launch_us": round(gemm_us, 3),
                "launch_timing": f"{GRAPH_STEPS} back-to-back launches per CUDA graph, publish off",
                "isolated_launch_us": round(iso_us, 3),
            },
            "cpu_baseline": cpu or None,
            "e2e": {
                "value": round(e2e_bytes / e2e_s / 1e9, 1),
                "unit": UNIT,
                "us_per_call": round(e2e_s / n_e2e * 1e6, 3),
                "steps": n_e2e,
                "h2d_bytes_per_step": h2d,
                "pipelining": f"every step copies its inputs in (one stream) and its output "
                              f"out (another); the compute waits on the input copies once "
                              f"per {E2E_BATCH} steps, the next batch's inputs landing "
                              f"while the current one computes; {E2E_GRAPH_STEPS} steps per "
                              "captured CUDA graph",
                "d2h_bytes_per_step": d2h,
            },
            "gpu_launches": 2 * steps,
            "tactic": {k: cfg[k] for k in ("split_k", "fold", "stages", "acc_blocks", "w_layout",
                                            "l2_prefetch", "l2_prefetch_early", "pipes",
                                            "tmem_columns")},
            "clocks": clock,
            "workloads": workloads,
        }
        print(json.dumps(line), flush=True)
    if group:
        import torch.distributed as dist

        dist.destroy_process_group()


def cpu_baseline(seconds: float) -> dict:
    """The oracle on the host cores: one thread for `seconds`, then one
    thread per core for half as long."""
    gbs, calls, secs, sample = oracle_baseline(seconds)
    out = {"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": sample, "seconds": round(secs, 2)}
    agbs, threads, acalls, asecs = oracle_baseline_all_cores(seconds / 2)
    out["all_cores"] = {"value": round(agbs, 4), "unit": UNIT, "cores": threads,
                        "sample": f"{acalls} calls of the same chain on the same slice, "
                                  f"one thread per core, over {asecs:.1f} s"}
    return out


# -------------------------------------------------------- reference arm
def run_reference(args):
    """The oracle as the reference arm: each step one oracle call of the
    whole chain on a column slice of the workload, the slice sized so all
    warm-up and timed steps fit in about two minutes."""
    world, rank, _ = dist_env()
    if rank != 0:
        return  # rank 0 alone runs the oracle; the others exit without work
    steps, warm = max(1, args.steps), max(0, args.warmup)
    per_step = min(3.0, 120.0 / (steps + warm))
    wl = workload()
    k = wl.k
    while True:  # shrink K until an 8-column call fits the per-step budget
        probe = OracleSample(8, k)
        t8 = min(probe.call() for _ in range(3))
        if t8 <= per_step or k <= 128:
            break
        k //= 2
    columns = int(max(8, min(1024, 8 * int(per_step / max(t8, 1e-6)))))
    sample = OracleSample(columns, k)
    for _ in range(warm):
        sample.call()
    total = sum(sample.call() for _ in range(steps))
    gbs = sample.weight_bytes * steps / total / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(gbs, 6),
        "unit": UNIT,
        "n_gpus": world,
        "steps": steps,
        "warmup": warm,
        "ms_per_step": round(total / steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) E4M3, E8M0 block-32 scales, 1% zero x)",
        "config": {
            "workload": f"decode projection N={wl.n} K={wl.k} m={wl.m} S={wl.split_k} "
                        "+ mailbox publish/consume",
            "n": wl.n, "k": wl.k, "m": wl.m, "split_k": wl.split_k,
            "sample_columns": columns, "sample_k": k,
            "weight_bytes_per_step": sample.weight_bytes,
        },
        "cpu_baseline": {"value": round(gbs, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample.describe(steps)},
        "e2e": {"value": round(gbs, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------- protocol rows
def run_protocols(args):
    """Each hand-off protocol on its own, at the headline's output size
    (m = 8 rows x N = 7168 BF16 columns), timed from CUDA graphs of
    GRAPH_STEPS calls between CUDA events: the sentinel mailbox (publish +
    consume), the tagged-pair mailbox (publish + consume), and the one-rank
    Lamport all-gather at payloads up to a few hundred kilobytes."""
    import numpy as np
    import torch

    import mxfp8_gemm_mailbox_gb300 as mx

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    wl = workload()
    rng = np.random.default_rng(5)
    c = torch.from_numpy(rng.integers(-2**15, 2**15, size=(wl.m, wl.n)).astype(np.int16)).to(device)
    stream = torch.cuda.Stream(device=device)

    def per_call_us(fn, calls_per_step=1):
        with torch.cuda.stream(stream):
            for _ in range(3):
                fn()
            stream.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                for _ in range(GRAPH_STEPS):
                    fn()
            for _ in range(3):
                graph.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            replays = max(1, args.steps // GRAPH_STEPS)
            e0.record(stream)
            for _ in range(replays):
                graph.replay()
            e1.record(stream)
        stream.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (replays * GRAPH_STEPS * calls_per_step)

    results = {}
    mb = mx.Mailbox(wl.capacity, wl.n, device=device)
    out = torch.empty((wl.m, wl.n), dtype=torch.bfloat16, device=device)

    def sentinel():
        mb.publish(c)
        mb.consume(wl.m, out)
    results["sentinel_mailbox_us"] = round(per_call_us(sentinel), 3)
    status, words = mb.status(stream)
    if status != mx.OK:
        raise RuntimeError(f"sentinel mailbox status {status}: {words}")
    tm = mx.TaggedMailbox(wl.capacity, wl.n, device=device)

    def tagged():
        tm.publish(c, 7)
        tm.consume(wl.m, 7, out)
    results["tagged_pairs_us"] = round(per_call_us(tagged), 3)
    gather_us = {}
    for nbytes in (16, 65536, 262144):
        g = mx.LamportGather(262144, device=device)
        src = torch.zeros(nbytes // 4, dtype=torch.int32, device=device)
        dst = torch.empty_like(src)
        gather_us[str(nbytes)] = round(per_call_us(lambda: g(src, dst)), 3)
        status, words = g.status(stream)
        if status != mx.OK:
            raise RuntimeError(f"gather status {status}: {words}")
    results["lamport_all_gather_us"] = gather_us
    payload = wl.m * wl.n * 2
    line = {
        "metric": "us/call of the output hand-off protocols (one GPU)",
        "value": results["sentinel_mailbox_us"],
        "unit": "us",
        "n_gpus": 1,
        "steps": max(1, args.steps // GRAPH_STEPS) * GRAPH_STEPS,
        "higher_is_better": False,
        "dtype": "bf16 bits",
        "data": "synthetic",
        "config": {"workload": f"hand-off of m={wl.m} x N={wl.n} BF16 ({payload} bytes)",
                   "timing": f"CUDA graphs of {GRAPH_STEPS} calls"},
        "results": results,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------- sweep table


def run_sweep(args):
    """The chain (publishing GEMM + PDL consumer) on every case of the sweep,
    m 1..8 x N {2048, 4096, 7168} x K {2048, 4096, 8192, 16384} x S {1, 2, 4},
    with the default tactic for each (N, K, S).  Each (N, K, S) gets enough
    handles (each with its own tiled weight copy) that the copies rotated
    through exceed twice the L2, so every call streams its weight from HBM;
    per case one CUDA graph of at least GRAPH_STEPS calls is replayed between
    CUDA events.  Prints one JSON line with a row per case."""
    import math

    import torch

    import mxfp8_gemm_mailbox_gb300 as mx
    import synthetic

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    peak, peak_kind = measured_peak()
    stream = torch.cuda.Stream(device=device)
    rows = []
    calls_target = max(GRAPH_STEPS, args.steps)
    ks = [int(v) for v in args.sweep_k.split(",") if v] or list(synthetic.SWEEP_K)
    for n in synthetic.SWEEP_N:
        for k in ks:
            base = synthetic.sweep_workload(8, n, k, 1)
            w, ws = synthetic.make_weights(base)
            W = torch.from_numpy(w).to(device)
            WS = torch.from_numpy(ws).to(device)
            weight_bytes = n * k + n * k // 32
            copies = min(64, max(3, -(-ROTATION_L2_MULTIPLE * L2_BYTES // weight_bytes)))
            for s in synthetic.SWEEP_S:
                mb = mx.Mailbox(8, n, device=device)
                gemms = [mx.PublishGemm(W, WS, mb, split_k=s, cta_k=args.cta_k, stream=stream)
                         for _ in range(copies)]
                cfg = gemms[0].config()
                out = torch.empty((8, n), dtype=torch.bfloat16, device=device)
                calls = copies * math.ceil(GRAPH_STEPS / copies)
                for m in synthetic.SWEEP_M:
                    wl = synthetic.sweep_workload(m, n, k, s)
                    x, xs = synthetic.make_activations(wl)
                    X = torch.from_numpy(x).to(device)
                    XS = torch.from_numpy(xs).to(device)
                    for g in gemms:
                        g.precompile(m)
                    with torch.cuda.stream(stream):
                        for i in range(calls):
                            gemms[i % copies].run(X, XS)
                            mb.consume(m, out)
                        stream.synchronize()
                        graph = torch.cuda.CUDAGraph()
                        with torch.cuda.graph(graph, stream=stream):
                            for i in range(calls):
                                gemms[i % copies].run(X, XS)
                                mb.consume(m, out)
                        for _ in range(max(3, args.warmup // calls)):
                            graph.replay()
                        replays = max(1, calls_target // calls)
                        e0 = torch.cuda.Event(enable_timing=True)
                        e1 = torch.cuda.Event(enable_timing=True)
                        e0.record(stream)
                        for _ in range(replays):
                            graph.replay()
                        e1.record(stream)
                    stream.synchronize()
                    status, words = mb.status(stream)
                    if status != mx.OK:
                        raise RuntimeError(f"mailbox status {status} ({words}) at m={m} N={n} "
                                           f"K={k} S={s}")
                    us = e0.elapsed_time(e1) * 1e3 / (replays * calls)
                    gbs = weight_bytes / (us * 1e-6) / 1e9
                    rows.append({"m": m, "n": n, "k": k, "split_k": s, "us_per_call": round(us, 3),
                                 "gbs": round(gbs, 1), "frac": round(gbs / peak, 4),
                                 "stages": cfg["stages"], "fold": cfg["fold"],
                                 "cta_k": cfg["cta_k"], "pipes": cfg["pipes"],
                                 "grid_ctas": cfg["grid_ctas"], "copies": copies})
                    del graph
                for g in gemms:
                    g.close()
                del gemms
                torch.cuda.synchronize(device)
                torch.cuda.empty_cache()
    best = max(rows, key=lambda r: r["gbs"])
    line = {
        "metric": "us/call and weight-stream HBM GB/s of the chain, every sweep case",
        "value": best["gbs"],
        "unit": UNIT,
        "n_gpus": 1,
        "higher_is_better": True,
        "dtype": "e4m3",
        "data": "synthetic (sweep recipe: signed x row pairs, duplicated and zero W rows, "
                "scale exponents in [-6, 3])",
        "config": {"workload": "sweep m 1..8 x N {2048, 4096, 7168} x K "
                               + "{" + ", ".join(map(str, ks)) + "} x S {1, 2, 4}",
                   "cta_k": args.cta_k or "library's choice",
                   "timing": "one CUDA graph of >= 30 chained calls per case, rotating "
                             f"min(64, {ROTATION_L2_MULTIPLE} x L2 / weight bytes) weight "
                             "copies (rows give the count)"},
        "peak": peak, "peak_kind": peak_kind,
        "rows": rows,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)


def main(argv=None):
    global _WORKLOAD
    args = parse_args(argv)
    _WORKLOAD = args.workload
    if args.impl == "reference":
        run_reference(args)
    elif args.path == "protocols":
        run_protocols(args)
    elif args.path == "sweep":
        run_sweep(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
