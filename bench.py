"""Benchmark of the Q4 verify matmul on GB300.

Default workload: the attention input projection of the 27B-class hybrid
(K = 5120 -> N = 14336, Q4 group-64 weights), verify rows swept M = 1, 2, 4, 8,
16.  One step = for each M, `reps` calls of q4_matmul, each on a different copy
of the weights from a rotating pool larger than L2, captured once into a CUDA
graph and replayed.  value = algorithmic HBM bytes of the step / device time,
bytes per call = N*K*0.5625 + M*K*2 + M*N*4 (weights once, x once, y once).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload attn_sweep|attn_wide|lm_head|mlp_gdn|full_pass|draft_edges]

full_pass: one step = the whole 27B-shaped verify pass through q4_decode_step
(64 layers x [in-proj, out-proj, gate/up, down] + the LM head twice, M = 16,
glue between layers), captured once in a CUDA graph; value = 15,149,629,440
weight bytes + activations and outputs per step / device time.

draft_edges: one step = `reps` calls of q4_draft_select_edges (4 lanes x 7 draft
positions, 16 x 16 edges each, rank 256, two 248,320 x 256 bf16 codebooks),
each timed alone after an L2 flush; value = algorithmic bytes (the 32 gathered
codebook rows, hidden, ids and scores of every row) / device time.

Under torchrun each rank runs its own replica (the path needs no exchange);
rank 0 prints one JSON line with the max-over-ranks time.
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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Q4 verify-matmul HBM GB/s (% of GB300 peak) at M=1..16; M=16/M=1 time ratio"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", choices=["attn_sweep", "attn_wide", "lm_head", "mlp_gdn", "full_pass", "draft_edges"], default="attn_sweep")
    p.add_argument("--reps", type=int, default=20, help="calls per graph (one graph per M)")
    p.add_argument("--graph-replays", type=int, default=50, help="replays of each M's graph per step")
    p.add_argument("--no-configs", action="store_true", help="attention sweep only (skip the other 27B shapes, "
                   "the LM head and the full pass)")
    p.add_argument("--cpu-seconds", type=float, default=15.0, help="target CPU time of the oracle sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--layers", type=int, default=64, help="full_pass only: the first LAYERS of the 64 layers "
                   "(4 linears each, no LM head; a small case for profiler captures)")
    return p.parse_args()


def workload_spec(name):
    """List of (label, N, K, [M...]) and the workload's description."""
    import synth_inputs as si
    if name == "attn_sweep":
        N, K = si.SHAPES["attn_in"]
        return [("attn_in", N, K, [1, 2, 4, 8, 16])], "attention input projection K=5120->N=14336, M sweep 1,2,4,8,16"
    if name == "attn_wide":
        N, K = si.SHAPES["attn_in"]
        return [("attn_in", N, K, [1, 8, 16, 24, 32])], ("attention input projection K=5120->N=14336, "
                                                          "M = 1, 8, 16, 24, 32 (up to four lanes of eight rows)")
    if name == "lm_head":
        N, K = si.SHAPES["lm_head"]
        return [("lm_head", N, K, [16, 16])], "LM head K=5120->N=248320, M=16, twice per step"
    if name == "full_pass":
        # the distinct linears of a GDN layer, M=16 (the CPU sample's shapes)
        shapes = [(n, *si.SHAPES[n], [16]) for n in ("gdn_in", "gdn_out", "gate_up", "down")]
        return shapes, ("full 27B-shaped verify pass: 64 layers (attention when i%4==3, else GDN) x [in-proj, "
                        "out-proj, gate/up, down] + LM head x2, M=16, chained through q4_decode_step")
    shapes = [(n, *si.SHAPES[n], [1, 16]) for n in ("gate_up", "down", "gdn_in", "gdn_out")]
    return shapes, "MLP + GDN projections (gate/up, down, GDN in, GDN out), M=1 and 16"


def max_over_ranks(value, world, device=None):
    """The maximum of a per-rank float over all ranks (the slowest replica
    sets the job time).  CPU tensor under gloo, device tensor under nccl."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    on = "cpu" if dist.get_backend() == "gloo" else device
    t = torch.tensor([float(value)], dtype=torch.float64, device=on)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step_per_rank, steps, ms_max, world):
    """Whole-job GB/s: the bytes every rank processed over the max-over-ranks time."""
    return world * bytes_per_step_per_rank * steps / (ms_max / 1e3) / 1e9


def call_bytes(M, N, K):
    return N * K * 9 // 16 + M * K * 2 + M * N * 4


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _strip_comments(src: str) -> str:
    """C/C++ source without its comments and blank lines (comment edits do not change a kernel)."""
    import re
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def kernel_source_hash(texts=None):
    """Hash of what the dominant kernel is made of, comments removed: its header,
    the PTX wrappers it uses and the host function that launches it (box, grid,
    split).  `texts` (name -> source) replaces the files on disk."""
    csrc = os.path.join(ROOT, "bit_row_speculative_gb300", "csrc")

    def read(fn):
        if texts is not None:
            return texts[fn]
        with open(os.path.join(csrc, fn)) as fh:
            return fh.read()

    h = hashlib.sha256()
    for fn in ("q4_tm.cuh", "q4_sm100.cuh"):
        h.update(fn.encode())
        h.update(_strip_comments(read(fn)).encode())
    abi = read("q4_abi.cu")
    for start in ("void plan_ranges(", "q4_status launch_tm("):
        i = abi.find(start)
        j = abi.find("\n}\n", i)
        h.update(_strip_comments(abi[i:j] if i >= 0 and j > i else abi).encode())
    return h.hexdigest()[:16]


def read_traffic(workload):
    """Per-launch DRAM bytes of the dominant kernel from the committed ncu
    summary, only if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"traffic_{workload}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as fh:
        for line in fh:
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
    if vals.get("source_hash") != kernel_source_hash():
        return None
    try:
        return float(vals["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.proc = None
        self.out = None
        try:
            self.out = open(os.devnull if gpu_id is None else os.path.join("/tmp", f"q4clk_{os.getpid()}.csv"), "w+")
            cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
            if gpu_id:
                cmd += ["-i", gpu_id]
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.seek(0)
        rows = [r.split(",") for r in self.out.read().strip().splitlines() if r.count(",") >= 7]
        try:
            os.unlink(self.out.name)
        except OSError:
            pass
        sm = [float(r[0]) for r in rows if r[0].strip().replace(".", "").isdigit()]
        mx = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].strip() == "Active"})
        power = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "power_w_max": max(power) if power else None}


CLOCK_REJECT = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clock_rejection(clocks):
    """Why a timed region's clock record voids its number, or None: a hardware or
    thermal slowdown was active, or the median SM clock sat well below its
    maximum with no reason given (a clock lock left by someone else).  A power
    cap alone is kept (it is normal under a long dense load)."""
    reasons = clocks.get("reasons") or []
    bad = [r for r in reasons if r in CLOCK_REJECT]
    if bad:
        return "active: " + ", ".join(bad)
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    if sm and mx and sm < 0.85 * mx and not reasons:
        return f"SM clock {sm:.0f} of {mx:.0f} MHz with no reason given"
    return None


def timed_region(run, gpu_id, world, dev, sync, status, sampler_cls=None, settle=0.3):
    """One timed region under the clock sampler, with a barrier and a device
    synchronize on both sides; `run()` enqueues the timed work and returns its
    CUDA-event measurements.  If the clock record of any rank is rejected
    (`clock_rejection`), the region runs once more and the second record is
    the one returned, marked `remeasured` (and `rejected` if it fails again)."""
    sampler_cls = sampler_cls or ClockSampler
    first = None
    for attempt in range(2):
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        sync()
        sampler = sampler_cls(gpu_id)
        time.sleep(settle)                     # nvidia-smi's first sample
        result = run()
        sync()
        clocks = sampler.stop()
        status()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        why = clock_rejection(clocks)
        any_bad = max_over_ranks(1.0 if why else 0.0, world, dev) > 0.0
        if not any_bad:
            break
        if attempt == 0:
            first = why or "rejected on another rank"
            print(f"[bench] clock record rejected ({first}); measuring once more", file=sys.stderr)
        else:
            clocks["rejected"] = why or "rejected on another rank"
    clocks["remeasured"] = first is not None
    if first is not None:
        clocks["first_rejected"] = first
    return result, clocks


_CPU_INPUTS = {}


def cpu_model():
    """The host CPU's model name from /proc/cpuinfo (on Arm, implementer and part
    numbers when no name is given), and the machine type."""
    import platform
    name, impl, part = None, None, None
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                k, _, v = line.partition(":")
                k, v = k.strip().lower(), v.strip()
                if k in ("model name", "cpu model") and not name:
                    name = v
                elif k == "cpu implementer" and not impl:
                    impl = v
                elif k == "cpu part" and not part:
                    part = v
    except OSError:
        pass
    if not name and impl:
        name = f"Arm CPU implementer {impl} part {part}" + (" (Neoverse V2, as in Grace)" if (impl, part) == ("0x41", "0xd4f") else "")
    return f"{name or 'unknown'} ({platform.machine()}, {os.cpu_count()} logical CPUs)"


def cpu_oracle_sample(spec, seconds, seed=0, single_core=False):
    """Time the CPU oracle on a bounded sample of the workload: every M of the
    sweep over a run of output columns (the whole matrix, repeated, when the
    host is fast enough), about `seconds` of wall time; GB/s with the same byte
    formula as the GPU line.  single_core: also the same on one thread."""
    import numpy as np
    import oracle
    import synth_inputs as si
    oracle.build()
    label, N, K, Ms = spec[0]
    key = (N, K, tuple(Ms))
    if key not in _CPU_INPUTS:                       # inputs made once per process, outside the timing
        _CPU_INPUTS[key] = (si.make_weights(N, K, 424242).numpy(),
                            {M: si.bf16_bits(si.make_x(M, K, 99 + M)).numpy().view(np.uint16) for M in set(Ms)})
    W, xs = _CPU_INPUTS[key]

    def timed(threads, secs):
        # calibrate on a probe of 16 columns per thread
        probe = min(N, 16 * threads)
        t0 = time.perf_counter()
        for M in Ms:
            oracle.matmul(xs[M], W, N, K, cols=np.arange(probe), threads=threads)
        dt = max(time.perf_counter() - t0, 1e-6)
        want = max(probe, int(probe * secs / dt))
        ncols, reps = (want, 1) if want <= N else (N, max(1, round(want / N)))
        cols = np.arange(ncols)
        t0 = time.perf_counter()
        for _ in range(reps):
            for M in Ms:
                oracle.matmul(xs[M], W, N, K, cols=cols, threads=threads)
        el = time.perf_counter() - t0
        nbytes = reps * sum(call_bytes(M, ncols, K) for M in Ms)
        what = f"first {ncols} of {N} output columns" if reps == 1 else f"all {N} output columns, {reps} times"
        return nbytes / el / 1e9, f"{label} K={K}, {what}, M in {Ms}, fp64 oracle on {threads} thread(s), {el:.1f} s wall"

    threads = os.cpu_count() or 1
    value, sample = timed(threads, seconds)
    out = {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample, "cpu": cpu_model()}
    if single_core:
        v1, s1 = timed(1, max(1.0, seconds / 3))
        out["single_core"] = {"value": v1, "unit": "GB/s", "cores": 1, "sample": s1}
    return out


def run_reference(args, rank, world):
    """The oracle as the reference arm, on the host cores (rank 0 only)."""
    if rank != 0:
        return
    if args.workload == "draft_edges":
        run_reference_edges(args, world)
        return
    spec, desc = workload_spec(args.workload)
    per_step = []
    walls = []
    cb = None
    for _ in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        cb = cpu_oracle_sample(spec, max(1.0, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup))))
        walls.append(time.perf_counter() - t0)
        per_step.append(cb["value"])
    vals = per_step[args.warmup:]
    value = statistics.mean(vals)
    label, N, K, Ms = spec[0]
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * statistics.mean(walls[args.warmup:]), 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": desc, "N": N, "K": K, "M": Ms},
            "cpu_baseline": {"kind": "oracle", "cores": cb["cores"], "sample": cb["sample"], "value": value,
                             "unit": "GB/s"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(check_roofline(line)), flush=True)


def run_reference_edges(args, world):
    """The edge-score oracle as the reference arm (host cores, rank 0)."""
    import numpy as np
    import torch
    import synth_inputs as si
    V, R = si.VOCAB, si.EDGE_RANK
    pb = si.make_codebook(V, R, 6001).view(torch.int16).numpy().view(np.uint16)
    sb = si.make_codebook(V, R, 6002).view(torch.int16).numpy().view(np.uint16)
    inputs = [si.make_edge_inputs(4, V, R, 7000 + k) for k in range(4)]
    vals, walls, cb = [], [], None
    for _ in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        cb = cpu_edges_sample(pb, sb, inputs, max(0.5, min(args.cpu_seconds, 60.0 / max(1, args.steps + args.warmup))))
        walls.append(time.perf_counter() - t0)
        vals.append(cb["value"])
    value = statistics.mean(vals[args.warmup:])
    line = {"impl": "reference", "metric": EDGE_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * statistics.mean(walls[args.warmup:]), 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"draft_select_edges: 4 lanes x 7 positions, 16 x 16 edges, rank {R}, "
                                   f"codebooks {V} x {R} bf16"},
            "cpu_baseline": {"kind": "oracle", "cores": cb["cores"], "sample": cb["sample"], "value": value,
                             "unit": "GB/s"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(check_roofline(line)), flush=True)


def check_roofline(line):
    """A measured rate above the peak is a counting error or L2 reuse, not a result:
    flag it in the line and on stderr (a fraction up to 1.05 is allowed, the peak being
    a measured copy, not a bound)."""
    rf = line.get("roofline") or {}
    frac = rf.get("frac")
    if isinstance(frac, (int, float)) and frac > 1.05:
        msg = f"roofline fraction {frac:.3f} above the measured peak: a counting or L2-reuse error"
        line["warning"] = msg
        print("WARNING: " + msg, file=sys.stderr, flush=True)
    return line


def e2e_pipelined(args, spec, pools, xs, ys, stream, dev, world, step_bytes, chunk=10):
    """End to end through q4.matmul with host buffers.  Every call of a step
    copies its own x from pinned host memory to the device and reads its own y
    back to pinned host memory.  The copies run on a second stream, a chunk of
    calls at a time: the inputs of chunk j + 1 are copied and the results of
    chunk j - 1 read back while chunk j's matmuls run, and the matmul stream
    waits once per chunk (so consecutive matmuls stay chained).  The step,
    copies included, is captured once in a CUDA graph and replayed, as a
    serving loop would."""
    import torch
    import bit_row_speculative_gb300 as q4
    calls = [(label, N, K, M, r) for label, N, K, Ms in spec for M in Ms for r in range(args.reps)]
    hx = [xs[(c[0], c[3])].cpu().pin_memory() for c in calls]
    hy = [torch.empty(ys[(c[0], c[3])].shape, dtype=torch.float32).pin_memory() for c in calls]
    dx = [torch.empty_like(xs[(c[0], c[3])]) for c in calls]
    dy = [torch.empty_like(ys[(c[0], c[3])]) for c in calls]
    h2d = sum(t.numel() * 2 for t in hx)
    d2h = sum(t.numel() * 4 for t in hy)
    cs = torch.cuda.Stream(device=dev)
    chunks = [list(range(a, min(a + chunk, len(calls)))) for a in range(0, len(calls), chunk)]

    def step():
        ev_in = [torch.cuda.Event() for _ in chunks]
        ev_mm = [torch.cuda.Event() for _ in chunks]

        def copy_in(j):
            with torch.cuda.stream(cs):
                for k in chunks[j]:
                    dx[k].copy_(hx[k], non_blocking=True)
                ev_in[j].record(cs)

        def read_back(j):
            with torch.cuda.stream(cs):
                cs.wait_event(ev_mm[j])
                for k in chunks[j]:
                    hy[k].copy_(dy[k], non_blocking=True)

        cs.wait_stream(stream)
        copy_in(0)
        for j, ks in enumerate(chunks):
            if j + 1 < len(chunks):
                copy_in(j + 1)
            stream.wait_event(ev_in[j])
            for k in ks:
                label, N, K, M, r = calls[k]
                W = pools[label][(r * 5 + M) % len(pools[label])]
                q4.matmul(dx[k], W, N, K, y=dy[k], stream=stream)
            ev_mm[j].record(stream)
            read_back(j)
        stream.wait_stream(cs)

    how = "graph"
    g = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(g, stream=stream):
            step()
        run = g.replay
    except Exception as exc:                             # report, then measure eagerly
        how = f"eager ({type(exc).__name__} in capture)"
        run = step
    with torch.cuda.stream(stream):
        run()
    stream.synchronize()
    e_steps = max(1, min(args.steps, 5))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e_steps):
            run()
        e1.record(stream)
    stream.synchronize()
    q4.device_status(stream)
    e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, world, dev)
    return {"value": round(job_throughput(step_bytes, 1, e_ms, world), 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e_ms, 4),
            "how": f"{how}: every call's x copied from pinned host memory and its y read back to pinned host "
                   f"memory, on a second stream in chunks of {chunk} calls overlapping the matmuls"}


def run_ours(args, rank, world, local_rank):
    import torch
    import bit_row_speculative_gb300 as q4
    import synth_inputs as si

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2**20)
    spec, desc = workload_spec(args.workload)

    # prediction first: the byte count and the ceiling at the measured peak
    peak, peak_kind = read_peaks()
    replays = max(1, args.graph_replays)
    step_bytes = sum(call_bytes(M, N, K) for _, N, K, Ms in spec for M in Ms) * args.reps * replays
    if rank == 0:
        print(f"prediction: {step_bytes / 1e9:.3f} GB per step at {peak:.0f} GB/s ({peak_kind}) "
              f"-> {step_bytes / peak / 1e6:.3f} ms per step floor", file=sys.stderr, flush=True)

    # rotating pools of distinct weight copies, each pool > 4x L2
    pools = {}
    for label, N, K, Ms in spec:
        nbytes = N * K * 9 // 16
        copies = max(2, -(-4 * l2 // nbytes))
        base = si.make_weights(N, K, si.w_seed(2, 0) + 7 * rank, device=dev)
        pools[label] = [base] + [base.clone() for _ in range(copies - 1)]
    xs = {(label, M): si.make_x(M, K, si.x_seed(2) + M, device=dev) for label, N, K, Ms in spec for M in Ms}
    ys = {(label, M): torch.empty((M, N), dtype=torch.float32, device=dev) for label, N, K, Ms in spec for M in Ms}

    stream = torch.cuda.Stream(device=dev)
    launches_per_call = 1          # the matmul kernel (it builds its own x records)

    def enqueue(label, N, K, M, i):
        W = pools[label][i % len(pools[label])]
        q4.matmul(xs[(label, M)], W, N, K, y=ys[(label, M)])

    # warm-up (eager), then one CUDA graph per (shape, M) holding `reps` calls
    counter = 0
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for label, N, K, Ms in spec:
                for M in Ms:
                    for r in range(args.reps):
                        enqueue(label, N, K, M, counter)
                        counter += 1
    stream.synchronize()
    q4.device_status(stream)

    graphs = []
    for label, N, K, Ms in spec:
        for M in Ms:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for r in range(args.reps):
                    enqueue(label, N, K, M, counter)
                    counter += 1
            graphs.append((label, N, K, M, g))
    with torch.cuda.stream(stream):
        for *_, g in graphs:          # one untimed replay of each graph
            g.replay()
    stream.synchronize()

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in graphs]
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(props.uuid)
    except Exception:
        pass
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)

    def run_steps():
        per_graph = {i: 0.0 for i in range(len(graphs))}
        with torch.cuda.stream(stream):
            t_start.record(stream)
            for _ in range(args.steps):
                for i, (label, N, K, M, g) in enumerate(graphs):
                    evs[i][0].record(stream)
                    for _ in range(replays):
                        g.replay()
                    evs[i][1].record(stream)
                # accumulate per-graph times after each step (events are reused)
                stream.synchronize()
                for i in range(len(graphs)):
                    per_graph[i] += evs[i][0].elapsed_time(evs[i][1])
            t_end.record(stream)
        return per_graph

    per_graph_ms, clocks = timed_region(run_steps, gpu_id, world, dev, torch.cuda.synchronize,
                                        lambda: q4.device_status(stream))

    kernel_ms = sum(per_graph_ms.values())            # device time of the matmul calls only
    total_ms = t_start.elapsed_time(t_end)
    kernel_ms = max_over_ranks(kernel_ms, world, dev)
    value = job_throughput(step_bytes, args.steps, kernel_ms, world)

    per_m = {}
    for i, (label, N, K, M, g) in enumerate(graphs):
        us = per_graph_ms[i] / (args.steps * args.reps * replays) * 1e3
        per_m[f"{label}_M{M}"] = {"us_per_call": round(us, 3),
                                  "GBs": round(call_bytes(M, N, K) / (us * 1e-6) / 1e9, 1)}
    ratio = ratio32 = None
    if args.workload in ("attn_sweep", "attn_wide"):
        ratio = per_m["attn_in_M16"]["us_per_call"] / per_m["attn_in_M1"]["us_per_call"]
    if args.workload == "attn_wide":
        ratio32 = per_m["attn_in_M32"]["us_per_call"] / per_m["attn_in_M1"]["us_per_call"]

    # LM head: the sampling epilogue (top-32, temperature 1, top_p 0.95) on the
    # head's own logits; bytes = the logits read once + the 32 (index, prob) pairs per row
    epilogue = None
    if args.workload == "lm_head":
        label, N, K, Ms = spec[0]
        yl = ys[(label, Ms[0])]
        ei = torch.empty((yl.shape[0], 32), dtype=torch.int32, device=dev)
        ep = torch.empty((yl.shape[0], 32), dtype=torch.float32, device=dev)
        reps = 50
        with torch.cuda.stream(stream):
            for _ in range(5):
                q4.topk_probs(yl, 32, 1.0, 0.95, idx=ei, probs=ep, stream=stream)
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            for _ in range(reps):
                q4.topk_probs(yl, 32, 1.0, 0.95, idx=ei, probs=ep, stream=stream)
            a1.record(stream)
        stream.synchronize()
        q4.device_status(stream)
        us = a0.elapsed_time(a1) / reps * 1e3
        ebytes = yl.numel() * 4 + yl.shape[0] * 32 * 8
        epilogue = {"what": "q4_topk_probs top_k=32 T=1 top_p=0.95 on the head's logits", "M": yl.shape[0],
                    "us_per_call": round(us, 3), "GBs": round(ebytes / (us * 1e-6) / 1e9, 1),
                    "launches_per_call": 1}
        # the head and its epilogue fused (q4_lm_head_topk: logits in the library's scratch,
        # dropped from L2 after the epilogue reads them)
        xl = xs[(label, Ms[0])]
        with torch.cuda.stream(stream):
            for k in range(3):
                q4.lm_head_topk(xl, pools[label][k % len(pools[label])], N, K, 32, 1.0, 0.95, idx=ei, probs=ep,
                                stream=stream)
            f0 = torch.cuda.Event(enable_timing=True)
            f1 = torch.cuda.Event(enable_timing=True)
            freps = 10
            f0.record(stream)
            for k in range(freps):
                q4.lm_head_topk(xl, pools[label][k % len(pools[label])], N, K, 32, 1.0, 0.95, idx=ei, probs=ep,
                                stream=stream)
            f1.record(stream)
        stream.synchronize()
        q4.device_status(stream)
        fus = f0.elapsed_time(f1) / freps * 1e3
        epilogue["fused_head_and_epilogue"] = {"what": "q4_lm_head_topk (matmul + epilogue, logits not stored)",
                                               "us_per_call": round(fus, 3), "launches_per_call": 2}

    # end to end through the public API with host buffers: per call, pinned
    # host x -> device, the matmul, device y -> pinned host
    e2e = e2e_pipelined(args, spec, pools, xs, ys, stream, dev, world, step_bytes // replays)

    if rank != 0:
        return
    n_calls = sum(len(Ms) for _, _, _, Ms in spec) * args.reps * replays
    achieved = step_bytes / (kernel_ms / args.steps / 1e3) / 1e9
    traffic = read_traffic(args.workload)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(kernel_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 x, q4 weights, fp32 accumulate",
        "data": "synthetic (seeded; nibbles uniform 0..15, scale |N(0,1)|*0.01, bias -8*scale+N(0,1e-3), x N(0,1))",
        "config": {"workload": desc, "calls_per_M_per_step": args.reps * replays,
                   "l2": f"rotating pool of {len(next(iter(pools.values())))} weight copies "
                         f"({sum(w.numel() for w in next(iter(pools.values()))) / 1e6:.0f} MB) > L2 "
                         f"({l2 / 2**20:.0f} MiB); one CUDA graph of {args.reps} calls per M, replayed {replays} "
                         f"times per step",
                   "parallelism": f"replicas x{world}"},
        "per_M": per_m, "ratio_M16_over_M1": None if ratio is None else round(ratio, 4),
        "ratio_M32_over_M1": None if ratio32 is None else round(ratio32, 4),
        "sampling_epilogue": epilogue,
        "frac_of_nominal_8TBs": round(value / world / NOMINAL_HBM_GBS, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "traffic": traffic, "algorithmic_bytes_per_launch": step_bytes // n_calls},
        "gpu_launches": n_calls * launches_per_call * args.steps,
        "clocks": clocks, "e2e": e2e, "timed_region_ms": round(total_ms, 3),
    }
    if args.workload == "attn_sweep" and not args.no_configs:
        del pools, graphs
        torch.cuda.empty_cache()
        line["per_shape"] = model_shapes(args, world, dev, l2, peak, peak_kind, stream)
    if not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = cpu_oracle_sample(spec, args.cpu_seconds, single_core=True)
        except Exception as exc:                     # report, do not hide
            line["cpu_baseline"] = {"error": repr(exc)}
    print(json.dumps(check_roofline(line)), flush=True)


def time_calls(enqueue, n_calls, replays, stream, world, dev):
    """Device microseconds per call of `enqueue(i)` (i = 0 .. n_calls-1), captured
    once in a CUDA graph and replayed `replays` times; the max over ranks."""
    import torch
    with torch.cuda.stream(stream):
        for i in range(min(n_calls, 6)):
            enqueue(i)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(n_calls):
            enqueue(i)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
    stream.synchronize()
    return max_over_ranks(e0.elapsed_time(e1) / (replays * n_calls) * 1e3, world, dev)


def model_shapes(args, world, dev, l2, peak, peak_kind, stream):
    """The other shapes of the 27B-class model at full size, each timed on its own
    (the MLP and GDN projections at M = 1 and 16, the LM head at M = 16), then the
    full chained pass at M = 16 with its time split by layer type (the same
    kernels run layer by layer, with events around each launch)."""
    import torch
    import bit_row_speculative_gb300 as q4
    import synth_inputs as si
    out = {}

    def entry(us, M, N, K, what):
        gbs = call_bytes(M, N, K) / (us * 1e-6) / 1e9
        return {"us_per_call": round(us, 3), "GBs": round(gbs, 1), "frac": round(gbs / peak, 4), "what": what}

    # config 3: gate/up, down, GDN in, GDN out; M = 1 and 16; rotating pools > 4x L2
    for name in ("gate_up", "down", "gdn_in", "gdn_out"):
        N, K = si.SHAPES[name]
        copies = max(2, -(-4 * l2 // (N * K * 9 // 16)))
        base = si.make_weights(N, K, si.w_seed(3, list(si.SHAPES).index(name)), device=dev)
        pool = [base] + [base.clone() for _ in range(copies - 1)]
        for M in (1, 16):
            x = si.make_x(M, K, si.x_seed(3) + M, device=dev)
            y = torch.empty((M, N), dtype=torch.float32, device=dev)
            us = time_calls(lambda i: q4.matmul(x, pool[i % copies], N, K, y=y, stream=stream), 20, 10, stream,
                            world, dev)
            out[f"{name}_M{M}"] = entry(us, M, N, K, f"K={K}->N={N}, {copies} weight copies rotating")
        del pool, base
    # config 4: the LM head, twice per step (target verify and draft readout, different x)
    N, K = si.SHAPES["lm_head"]
    heads = [si.make_weights(N, K, si.w_seed(4, t), device=dev) for t in range(2)]
    xh = [si.make_x(16, K, si.x_seed(4) + t, device=dev) for t in range(2)]
    yh = torch.empty((16, N), dtype=torch.float32, device=dev)
    us = time_calls(lambda i: q4.matmul(xh[i % 2], heads[i % 2], N, K, y=yh, stream=stream), 10, 5, stream, world, dev)
    out["lm_head_M16"] = entry(us, 16, N, K, f"K={K}->N={N}, two heads alternating")
    del heads, xh, yh
    torch.cuda.empty_cache()
    # config 5: the full pass, one q4_decode_step; then the same launches layer by layer
    spec = si.full_pass_spec()
    M = 16
    layers = [(si.make_weights(Nn, Kk, si.w_seed(5, t), device=dev), Nn, Kk, g) for t, (Nn, Kk, g) in enumerate(spec)]
    x0 = si.make_x(M, spec[0][1], si.x_seed(5), device=dev)
    y = torch.empty((M, spec[-1][0]), dtype=torch.float32, device=dev)
    ws = torch.empty(q4.decode_step_workspace_bytes(layers, M), dtype=torch.uint8, device=dev)
    step_ms = time_calls(lambda i: q4.decode_step(layers, x0, y_last=y, workspace=ws, stream=stream), 1, 5, stream,
                         world, dev) / 1e3
    step_bytes = sum(call_bytes(M, Nn, Kk) for Nn, Kk, _ in spec)
    types = {}
    ybuf = torch.empty(M * max(Nn for Nn, _, _ in spec), dtype=torch.float32, device=dev)
    xbuf = torch.empty(M * max(Kk for _, Kk, _ in spec), dtype=torch.bfloat16, device=dev)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(2 * len(spec))]

    def kind(t, Nn, Kk):
        i = t // 4
        if t >= 4 * 64:
            return "lm_head"
        return ["attn_in" if i % 4 == 3 else "gdn_in", "attn_out" if i % 4 == 3 else "gdn_out", "gate_up",
                "down"][t % 4]

    for rep in range(3):
        with torch.cuda.stream(stream):
            xj = x0
            for t, (W, Nn, Kk, g) in enumerate(layers):
                yj = y if t + 1 == len(layers) else ybuf[:M * Nn].view(M, Nn)
                evs[2 * t][0].record(stream)
                q4.matmul(xj, W, Nn, Kk, y=yj, stream=stream)
                evs[2 * t][1].record(stream)
                if t + 1 < len(layers):
                    Kn = layers[t + 1][2]
                    xn = xbuf[:M * Kn].view(M, Kn)
                    evs[2 * t + 1][0].record(stream)
                    q4.glue(yj, Kn, g, x_next=xn, stream=stream)
                    evs[2 * t + 1][1].record(stream)
                    xj = xn
        stream.synchronize()
        if rep < 2:
            continue
        for t, (W, Nn, Kk, g) in enumerate(layers):
            k = kind(t, Nn, Kk)
            d = types.setdefault(k, {"layers": 0, "ms": 0.0, "bytes": 0})
            d["layers"] += 1
            d["ms"] += evs[2 * t][0].elapsed_time(evs[2 * t][1])
            d["bytes"] += call_bytes(M, Nn, Kk)
            if t + 1 < len(layers):
                gd = types.setdefault("glue", {"layers": 0, "ms": 0.0, "bytes": 0})
                gd["layers"] += 1
                gd["ms"] += evs[2 * t + 1][0].elapsed_time(evs[2 * t + 1][1])
                gd["bytes"] += M * Nn * 4 + M * layers[t + 1][2] * 2
    total = sum(d["ms"] for d in types.values())
    split = {}
    for k, d in types.items():
        gbs = d["bytes"] / (d["ms"] * 1e-3) / 1e9
        split[k] = {"layers": d["layers"], "ms": round(d["ms"], 4), "share": round(d["ms"] / total, 4),
                    "GBs": round(gbs, 1), "frac": round(gbs / peak, 4)}
    gbs = step_bytes / (step_ms * 1e-3) / 1e9
    out["full_pass_M16"] = {"ms_per_step": round(step_ms, 4), "GBs": round(gbs, 1), "frac": round(gbs / peak, 4),
                            "what": f"{len(spec)} linears + glue in one q4_decode_step (CUDA graph), "
                                    f"{sum(Nn * Kk * 9 // 16 for Nn, Kk, _ in spec) / 1e9:.3f} GB of weights",
                            "by_layer_type": split,
                            "by_layer_type_how": "the same layers run as separate q4_matmul / q4_glue calls with "
                                                 "events around each launch (eager), "
                                                 f"{total:.3f} ms in all"}
    del layers
    torch.cuda.empty_cache()
    out["peak"] = {"GBs": peak, "kind": peak_kind}
    return out


def run_full_pass(args, rank, world, local_rank):
    """The chained 27B-shaped verify pass through q4_decode_step, M = 16."""
    import torch
    import bit_row_speculative_gb300 as q4
    import synth_inputs as si

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2**20)
    M = 16
    spec = si.full_pass_spec()
    _, desc = workload_spec("full_pass")
    if not 1 <= args.layers <= 64:
        raise SystemExit("--layers must be in 1..64")
    if args.layers < 64:
        # a small case of the same kernels: the first layers only, the last linear ending the step
        spec = spec[:4 * args.layers]
        spec[-1] = (spec[-1][0], spec[-1][1], 0)
        desc = (f"the first {args.layers} of the 64 layers of the 27B-shaped verify pass (4 linears each, no LM "
                f"head; a profiling case, not the full pass), M=16, chained through q4_decode_step")
    weight_bytes = sum(N * K * 9 // 16 for N, K, _ in spec)
    n_mm = len(spec)
    # algorithmic bytes of the step: every weight once, each layer's x and y once
    step_bytes = sum(call_bytes(M, N, K) for N, K, _ in spec)
    peak, peak_kind = read_peaks()
    if rank == 0:
        print(f"prediction: {step_bytes / 1e9:.3f} GB per step at {peak:.0f} GB/s ({peak_kind}) "
              f"-> {step_bytes / peak / 1e6:.3f} ms per step floor", file=sys.stderr, flush=True)

    layers = [(si.make_weights(N, K, si.w_seed(5, t) + 7 * rank, device=dev), N, K, g)
              for t, (N, K, g) in enumerate(spec)]
    x0 = si.make_x(M, spec[0][1], si.x_seed(5), device=dev)
    y = torch.empty((M, spec[-1][0]), dtype=torch.float32, device=dev)
    ws = torch.empty(q4.decode_step_workspace_bytes(layers, M), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            q4.decode_step(layers, x0, y_last=y, workspace=ws, stream=stream)
    stream.synchronize()
    q4.device_status(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        q4.decode_step(layers, x0, y_last=y, workspace=ws, stream=stream)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()

    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(props.uuid)
    except Exception:
        pass
    def run_steps():
        with torch.cuda.stream(stream):
            for i in range(args.steps):
                evs[i][0].record(stream)
                g.replay()
                evs[i][1].record(stream)
        stream.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    step_ms, clocks = timed_region(run_steps, gpu_id, world, dev, torch.cuda.synchronize,
                                   lambda: q4.device_status(stream))
    kernel_ms = max_over_ranks(sum(step_ms), world, dev)
    value = job_throughput(step_bytes, args.steps, kernel_ms, world)

    # end to end through the public call: every step copies x0 from pinned host
    # memory and reads y_last back to pinned host memory.  The read-back of step s
    # (15.9 MB) runs on a second stream while step s + 1 computes (y_last double
    # buffered), as a serving loop would overlap them.
    hx = x0.cpu().pin_memory()
    hy = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for _ in range(2)]
    dx = torch.empty_like(x0)
    dy = [torch.empty_like(y) for _ in range(2)]
    cs = torch.cuda.Stream(device=dev)
    e_steps = max(2, min(args.steps, 6))
    ev_done = [torch.cuda.Event() for _ in range(e_steps + 1)]
    ev_read = [torch.cuda.Event() for _ in range(e_steps + 1)]
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for s in range(e_steps + 1):
            if s == 1:
                e0.record(stream)
            if s >= 2:
                stream.wait_event(ev_read[s - 2])          # this y buffer has been read back
            dx.copy_(hx, non_blocking=True)
            q4.decode_step(layers, dx, y_last=dy[s % 2], workspace=ws, stream=stream)
            ev_done[s].record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(ev_done[s])
                hy[s % 2].copy_(dy[s % 2], non_blocking=True)
                ev_read[s].record(cs)
        stream.wait_stream(cs)
        e1.record(stream)
    stream.synchronize()
    q4.device_status(stream)
    e_ms = max_over_ranks(e0.elapsed_time(e1) / e_steps, world, dev)
    e2e = {"value": round(job_throughput(step_bytes, 1, e_ms, world), 1), "unit": "GB/s",
           "h2d_bytes_per_step": hx.numel() * 2, "d2h_bytes_per_step": hy[0].numel() * 4,
           "ms_per_step": round(e_ms, 4),
           "how": "per step: x0 from pinned host memory, the step, y_last read back to pinned host memory on a second "
                  "stream overlapping the next step"}

    if rank != 0:
        return
    ms = kernel_ms / args.steps
    achieved = step_bytes / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 x, q4 weights, fp32 accumulate",
        "data": "synthetic (seeded; nibbles uniform 0..15, scale |N(0,1)|*0.01, bias -8*scale+N(0,1e-3), x N(0,1))",
        "config": {"workload": desc, "M": M, "layers": n_mm, "weight_bytes_per_step": weight_bytes,
                   "l2": f"inputs ({weight_bytes / 1e9:.2f} GB of weights) far larger than L2 "
                         f"({l2 / 2**20:.0f} MiB); one CUDA graph per step",
                   "parallelism": f"replicas x{world}"},
        "step_ms": {"median": round(statistics.median(step_ms), 4), "min": round(min(step_ms), 4),
                    "max": round(max(step_ms), 4)},
        "frac_of_nominal_8TBs": round(value / world / NOMINAL_HBM_GBS, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind, "traffic": None,
                     "algorithmic_bytes_per_launch": step_bytes // n_mm,
                     "note": "whole step (matmul and glue launches) timed; a lower bound for the matmul kernel"},
        # one matmul per layer (the first builds its own x records) and one glue between
        # consecutive layers (writing the next layer's x records)
        "gpu_launches": (n_mm + (n_mm - 1)) * args.steps,
        "clocks": clocks, "e2e": e2e,
    }
    if not args.no_cpu_baseline:
        try:
            line["cpu_baseline"] = cpu_oracle_sample(workload_spec("full_pass")[0], args.cpu_seconds)
        except Exception as exc:                     # report, do not hide
            line["cpu_baseline"] = {"error": repr(exc)}
    print(json.dumps(check_roofline(line)), flush=True)


EDGE_METRIC = "draft_select_edges: algorithmic GB/s of the gathered codebook rows, hidden, ids and scores"


def edge_call_bytes(rows, R):
    return rows * (32 * R * 2 + R * 4 + 2 * 16 * 4 + 256 * 4)


def cpu_edges_sample(P_bits, S_bits, inputs, seconds):
    """The edge-score oracle timed on the host on successive calls of the workload
    until about `seconds` have passed."""
    import numpy as np
    from oracle import edges as E
    calls, byts = 0, 0
    t0 = time.perf_counter()
    while True:
        hidden, pred, cand = inputs[calls % len(inputs)]
        E.edge_scores(P_bits, S_bits, hidden.numpy(), pred.numpy(), cand.numpy())
        calls += 1
        byts += edge_call_bytes(hidden.shape[0], hidden.shape[1])
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": round(byts / dt / 1e9, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{calls} calls of the workload (4 lanes x 7 positions), fp64 oracle, one thread",
            "ms_per_call": round(dt / calls * 1e3, 2)}


def run_edges(args, rank, world, local_rank):
    """The draft selector's edge scores: 4 lanes x 7 positions per call."""
    import numpy as np
    import torch
    import bit_row_speculative_gb300 as q4
    import synth_inputs as si

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2**20)
    V, R, lanes = si.VOCAB, si.EDGE_RANK, 4
    rows = lanes * si.EDGE_POSITIONS
    P = si.make_codebook(V, R, 6001 + 7 * rank, device=dev)
    S = si.make_codebook(V, R, 6002 + 7 * rank, device=dev)
    host_inputs = [si.make_edge_inputs(lanes, V, R, 7000 + k) for k in range(16)]
    dev_inputs = [tuple(t.to(dev) for t in inp) for inp in host_inputs]
    score = torch.empty((rows, 16, 16), dtype=torch.float32, device=dev)
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)       # written between timed calls
    call_b = edge_call_bytes(rows, R)
    peak, peak_kind = read_peaks()
    stream = torch.cuda.Stream(device=dev)

    def call(k):
        h, pr, ca = dev_inputs[k % len(dev_inputs)]
        q4.draft_select_edges(P, S, h, pr, ca, score=score, stream=stream)

    with torch.cuda.stream(stream):
        for k in range(args.warmup * args.reps):
            call(k)
    stream.synchronize()
    q4.device_status(stream)
    n = args.steps * args.reps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    gpu_id = None
    try:
        gpu_id = "GPU-" + str(props.uuid)
    except Exception:
        pass
    def run_calls():
        with torch.cuda.stream(stream):
            for k in range(n):
                flush.fill_(k & 255)
                evs[k][0].record(stream)
                call(k)
                evs[k][1].record(stream)
        stream.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    call_ms, clocks = timed_region(run_calls, gpu_id, world, dev, torch.cuda.synchronize,
                                   lambda: q4.device_status(stream))
    kernel_ms = max_over_ranks(sum(call_ms), world, dev)
    value = job_throughput(call_b * args.reps, args.steps, kernel_ms, world)

    # end to end through the public call: every call copies its hidden and ids
    # from pinned host memory and reads its scores back, on a second stream in
    # chunks of 10 calls overlapping the kernels; captured once in a CUDA graph
    n_e = 50
    hh = [tuple(t.pin_memory() for t in host_inputs[k % len(host_inputs)]) for k in range(n_e)]
    dd = [tuple(torch.empty_like(t, device=dev) for t in hh[k]) for k in range(n_e)]
    hs = [torch.empty(score.shape, dtype=score.dtype).pin_memory() for _ in range(n_e)]
    ds = [torch.empty_like(score) for _ in range(n_e)]
    cs = torch.cuda.Stream(device=dev)
    chunks = [list(range(a, min(a + 10, n_e))) for a in range(0, n_e, 10)]

    def e2e_step():
        ev_in = [torch.cuda.Event() for _ in chunks]
        ev_k = [torch.cuda.Event() for _ in chunks]

        def copy_in(j):
            with torch.cuda.stream(cs):
                for k in chunks[j]:
                    for d_, h_ in zip(dd[k], hh[k]):
                        d_.copy_(h_, non_blocking=True)
                ev_in[j].record(cs)

        cs.wait_stream(stream)
        copy_in(0)
        for j, ks in enumerate(chunks):
            if j + 1 < len(chunks):
                copy_in(j + 1)
            stream.wait_event(ev_in[j])
            for k in ks:
                q4.draft_select_edges(P, S, dd[k][0], dd[k][1], dd[k][2], score=ds[k], stream=stream)
            ev_k[j].record(stream)
            with torch.cuda.stream(cs):
                cs.wait_event(ev_k[j])
                for k in ks:
                    hs[k].copy_(ds[k], non_blocking=True)
        stream.wait_stream(cs)

    how = "graph"
    ge = torch.cuda.CUDAGraph()
    try:
        with torch.cuda.graph(ge, stream=stream):
            e2e_step()
        run = ge.replay
    except Exception as exc:
        how = f"eager ({type(exc).__name__} in capture)"
        run = e2e_step
    with torch.cuda.stream(stream):
        run()
    stream.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(3):
            run()
        e1.record(stream)
    stream.synchronize()
    q4.device_status(stream)
    e_ms = max_over_ranks(e0.elapsed_time(e1) / (3 * n_e), world, dev)
    per_call_in = sum(t.numel() * t.element_size() for t in hh[0])
    e2e = {"value": round(job_throughput(call_b, 1, e_ms, world), 2), "unit": "GB/s",
           "h2d_bytes_per_step": per_call_in * args.reps, "d2h_bytes_per_step": hs[0].numel() * 4 * args.reps,
           "us_per_call": round(e_ms * 1e3, 3),
           "how": f"{how}: every call's hidden and ids copied in and its scores read back, on a second stream in "
                  "chunks of 10 calls overlapping the kernels"}

    if rank != 0:
        return
    us = kernel_ms / n * 1e3
    achieved = call_b / (us * 1e-6) / 1e9
    line = {
        "metric": EDGE_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(kernel_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16 codebooks, fp32 hidden and accumulate",
        "data": "synthetic (seeded; codebooks N(0,1)*0.05 bf16, hidden N(0,1), 16 distinct candidates per position, "
                "predecessors = the previous position's candidates, the anchor at position 0)",
        "config": {"workload": f"draft_select_edges: {lanes} lanes x {si.EDGE_POSITIONS} positions, 16 x 16 edges, "
                               f"rank {R}, codebooks {V} x {R} bf16 (2 x {V * R * 2 / 1e6:.0f} MB)",
                   "calls_per_step": args.reps,
                   "l2": f"L2 flushed ({2 * l2 / 2**20:.0f} MiB written) before every timed call",
                   "parallelism": f"replicas x{world}"},
        "us_per_call": {"mean": round(us, 3), "median": round(statistics.median(call_ms) * 1e3, 3),
                        "min": round(min(call_ms) * 1e3, 3)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 5), "peak_kind": peak_kind, "traffic": None,
                     "algorithmic_bytes_per_launch": call_b,
                     "note": "one CTA per row gathers 32 rows of 512 B: latency-bound at this size"},
        "gpu_launches": n,
        "clocks": clocks, "e2e": e2e,
    }
    if not args.no_cpu_baseline:
        try:
            pb = P.cpu().view(torch.int16).numpy().view(np.uint16)
            sb = S.cpu().view(torch.int16).numpy().view(np.uint16)
            line["cpu_baseline"] = cpu_edges_sample(pb, sb, host_inputs, min(args.cpu_seconds, 10.0))
        except Exception as exc:                     # report, do not hide
            line["cpu_baseline"] = {"error": repr(exc)}
    print(json.dumps(check_roofline(line)), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        if args.workload == "full_pass":
            run_full_pass(args, rank, world, local_rank)
        elif args.workload == "draft_edges":
            run_edges(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
