"""Benchmark of the fused AllReduce + residual-add + RMSNorm epilogue on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload prefill|decode|two_stage|tiny] [--sweep] [--quick]

One JSON line on rank 0.  A step is one ar_rmsnorm call in AUTO mode (the
heuristic picks one- or two-stage) over the whole workload, inputs resident
in HBM.  The headline workload is the prefill shape (n = 8 partials, H =
6144, m = 8192 tokens), where the HBM roofline applies; the decode and
mid-size shapes are reported beside it as a latency-vs-m table measured the
pages' way (2000 calls captured in one CUDA graph, per-call time = the
fastest replay / 2000; ROCm/aiter #3817, Test Plan, Benchmark), hot (same
buffers) and cold (buffer sets rotating over >= 4x L2).

Bytes per call (algorithmic): (n + 3) * m * H * 2 + H * 2 -- n partials and
the residual read, out and residual_out written, the weight read once.

Multi-GPU: each rank runs its own replica on its own device (rows of
different calls are independent; there is no data-path collective on one
GPU), timing is bracketed by a barrier and a device synchronize, the slowest
rank's time counts, and ``value`` aggregates all ranks (weak scaling).

--impl reference times the CPU oracle (the reference arm of this build) on
the host cores, on a bounded sample of the same workload, same metric.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused AR+residual+RMSNorm µs/call and HBM GB/s (% of ~8 TB/s) vs m"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0     # GB300 HBM3e, nominal
L2_BYTES_FALLBACK = 129 * 1024 * 1024


def algo_bytes(n, m, H):
    return (n + 3) * m * H * 2 + H * 2


def actual_bytes(n, m, H, two_stage):
    return algo_bytes(n, m, H) + (2 * m * H * 2 if two_stage else 0)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "of measured"
    except Exception:
        return FALLBACK_HBM_GBS, "of fallback"


# The files a kernel's device code comes from.
KERNEL_SOURCES = {
    "k_stream_epilogue": ("common.cuh", "stream_epilogue.cuh"),
    "k_fused_epilogue": ("common.cuh", "epilogue.cuh"),
    "k_reduce_flat": ("common.cuh", "epilogue.cuh", "reduce_flat.cu"),
}
# The launch-plan fields that decide a launch's instantiation and shape.
PLAN_KEYS = ("kernel", "cluster", "vpt", "threads", "stages", "ctas", "prefetch")


def source_hash(kernel):
    """Hash of the files that define `kernel` (its device code)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "allreduce_sum_residual_gb300", "csrc")
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, workload, plan=None):
    """DRAM bytes per launch recorded by an ncu capture of this kernel, or None
    when none exists, the kernel sources changed since it was taken, or the
    launch plan (instantiation and shape) differs from the captured one."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
        e = d[f"{kernel}@{workload}"]
        if e.get("source_hash") != source_hash(kernel):
            return None
        if plan is not None and any(e["plan"][k] != plan[k] for k in PLAN_KEYS):
            return None
        return float(e["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.idx = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"arn_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9 and parts[1].isdigit():
                        rows.append(parts)
            os.unlink(self.path)
        except Exception:
            pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [int(r[1]) for r in rows]
        smax = int(rows[0][2])
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------- distributed

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = os.environ.get("ARN_DIST_BACKEND", "nccl")
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world, device=None):
    if world > 1:
        import torch.distributed as dist
        if device is not None and dist.get_backend() == "nccl":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


def max_over_ranks(world, x, device=None):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = device if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(world, x, device=None):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = device if (device is not None and dist.get_backend() == "nccl") else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------- our arm

def settle(device=None):
    """Wait for all work queued so far (on every stream) before side-stream
    work starts.  Inputs and outputs are made on the default stream; a
    kernel launched on a side stream is not ordered after that work, and the
    caching allocator may hand it memory a default-stream kernel is still
    reading (a temporary of the input generator), which would corrupt the
    inputs.  Every function here that launches on a side stream settles
    first."""
    import torch
    torch.cuda.synchronize(device)


def launch_shield(stream, cycles=2_000_000):
    """Keep `stream` busy for ~1 ms (a device-side sleep) before a start
    event, so that the host has enqueued the timed work when the event
    fires: the region then times the kernels, not the host's launch of the
    first graph.  No-op where torch has no device sleep."""
    import torch
    sleep = getattr(torch.cuda, "_sleep", None)
    if sleep is None:
        return
    with torch.cuda.stream(stream):
        sleep(int(cycles))


def timed_steps(fn, stream, steps, warmup, world, device, use_graph=True, chunk=100):
    """W warm-up steps, then exactly K steps timed with CUDA events on
    `stream`, bracketed by barrier + synchronize.  With `use_graph` the K
    steps are replayed from CUDA graphs of `chunk` steps (plus one graph for
    the remainder), so host launch overhead stays out of the timed region,
    as in the pages' method.  Returns (total_s, mean step s)."""
    import torch
    settle(device)
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize(device)
    graphs = []
    if use_graph:
        full, rest = divmod(steps, chunk)
        for count in ([chunk] if full else []) + ([rest] if rest else []):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for _ in range(count):
                    fn()
            graphs.append((g, count))
        plan = [graphs[0]] * full + ([graphs[-1]] if rest else []) if full else graphs
        with torch.cuda.stream(stream):
            for g, _ in graphs:   # one untimed replay of each graph
                g.replay()
        torch.cuda.synchronize(device)
    barrier(world, device)
    torch.cuda.synchronize(device)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    launch_shield(stream)
    t0.record(stream)
    if use_graph:
        with torch.cuda.stream(stream):
            for g, _ in plan:
                g.replay()
    else:
        for _ in range(steps):
            fn()
    t1.record(stream)
    torch.cuda.synchronize(device)
    barrier(world, device)
    total = t0.elapsed_time(t1) / 1e3
    del graphs
    return total, total / steps


def graph_per_call(call, stream, calls, replays, warm=None):
    """The pages' timing method for any step: call(c) for c = 0 .. calls-1
    captured in one CUDA graph (after one eager pass of warm(), by default
    call(0)), replayed once untimed, then `replays` timed replays with CUDA
    events on `stream`, each behind a launch shield.  Returns the fastest
    replay / calls, in seconds."""
    import torch
    settle()
    with torch.cuda.stream(stream):
        (warm or (lambda: call(0)))()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for c in range(calls):
            call(c)
    best = float("inf")
    with torch.cuda.stream(stream):
        g.replay()
        for _ in range(replays):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            launch_shield(stream)
            a.record(stream)
            g.replay()
            b.record(stream)
            b.synchronize()
            best = min(best, a.elapsed_time(b) / 1e3)
    del g
    return best / calls


def graph_latency(arn, inps, mode, eps, stream, calls=2000, replays=80, shape=None):
    """The pages' method: `calls` calls in one CUDA graph (cycling over the
    input sets in `inps`), per-call time = min over replays / calls.
    `shape` = (kernel, cluster, vpt[, threads, stages, ctas]), or a dict of
    ar_rmsnorm_ex's plan keywords (kernel, cluster, vpt, threads, stages,
    ctas, prefetch), forces a launch shape."""
    import torch
    outs = [(torch.empty_like(i.residual), torch.empty_like(i.residual)) for i in inps]
    if shape is not None and not isinstance(shape, dict):
        shape = dict(zip(("kernel", "cluster", "vpt", "threads", "stages", "ctas"), shape))

    def one(i, o, r):
        if shape is None:
            arn.ar_rmsnorm(i.partials, i.residual, i.weight, eps, out=o, residual_out=r, mode=mode)
        else:
            arn.ar_rmsnorm_ex(i.partials, i.residual, i.weight, eps, out=o, residual_out=r,
                              mode=mode, **shape)

    def call(c):
        one(inps[c % len(inps)], *outs[c % len(outs)])

    def warm():
        for i, (o, r) in zip(inps, outs):
            one(i, o, r)

    return graph_per_call(call, stream, calls, replays, warm)


def cold_sets(synth, w, m, base, l2_bytes, calls, cap_bytes=8 << 30):
    """Input sets for a cold-cache graph: views into one pool of bf16 data,
    one set per call up to `calls`, so that the calls of one replay touch
    at least ~2.5x the L2 (or every set is already larger than L2).  The
    weight is shared (it is one H-vector).  Values follow the workload's
    distributions (drawn once for the pool)."""
    import torch
    per_set = (w.n + 1) * m * w.H
    set_bytes = per_set * 2
    want = max(2, -(-int(2.5 * l2_bytes) // set_bytes))
    nsets = int(min(calls, want, max(2, cap_bytes // set_bytes)))
    pool = synth.normal_bf16((nsets, w.n + 1, m, w.H), 0.0, w.p_std, w.seed, 7,
                             backend="torch", device="cuda")
    sets = []
    for i in range(nsets):
        parts = [pool[i, k] for k in range(w.n)]
        sets.append(synth.Inputs(parts, pool[i, w.n], base.weight, base.eps))
    return sets


def unfused_torch_us(inp, stream, calls=50, replays=5):
    """Comparator only (never the product path): the same epilogue as
    separate torch ops -- rank-order fp32 sum, bf16 round (what an
    all-reduce returns), residual add, torch RMSNorm -- in one CUDA graph;
    per-call time = fastest replay / calls."""
    import torch
    H = inp.residual.shape[1]
    w = inp.weight.float()

    def call(c):
        s = inp.partials[0].float()
        for p in inp.partials[1:]:
            s = s + p.float()
        r = s.to(torch.bfloat16).float() + inp.residual.float()
        r.to(torch.bfloat16)
        torch.nn.functional.rms_norm(r, (H,), w, eps=inp.eps).to(torch.bfloat16)

    return graph_per_call(call, stream, calls, replays) * 1e6


def allgather_two_stage_us(arn, inp, stream, calls=20, replays=5):
    """Two-stage with the gather done by stores, all ranks on this GPU: for
    rank r = 0 .. n-1, ar_reduce_scatter_store reduces slice r and writes it
    into n temporaries (one per rank), then stage 2 runs on temps[0].  The
    n-copy write is what a real reduce-scatter + all-gather costs in stores
    (here to local memory).  Per-call time = fastest replay / calls."""
    import torch
    n = len(inp.partials)
    temps = [torch.empty_like(inp.residual) for _ in range(n)]
    out = torch.empty_like(inp.residual)
    rout = torch.empty_like(inp.residual)

    def call(c):
        for r in range(n):
            arn.ar_reduce_scatter_store(inp.partials, temps, r)
        arn.ar_load_rmsnorm(temps[0], inp.residual, inp.weight, inp.eps, out=out, residual_out=rout)

    t = graph_per_call(call, stream, calls, replays)
    del temps
    return t * 1e6


def two_shot_all_ranks_us(arn, inp, stream, calls=20, replays=5):
    """The cross-rank two-shot path with every rank on this GPU, run in turn
    so that no kernel waits on a later launch: ranks 1 .. n-1 post their
    flag, store their stage-1 slice into all n temporaries and post again,
    then rank 0's ar_rmsnorm_two_shot (barrier, its slice, barrier -- both
    find every flag set -- and stage 2).  Epochs come from the signal pads,
    so the graph replays with fresh ones.  Returns (per-call µs, status
    word after)."""
    import torch
    n = len(inp.partials)
    temps = [torch.empty_like(inp.residual) for _ in range(n)]
    pads = [torch.zeros(arn.AR_SIGNAL_PAD_BYTES // 4, dtype=torch.int32, device=inp.residual.device)
            for _ in range(n)]
    out = torch.empty_like(inp.residual)
    rout = torch.empty_like(inp.residual)

    def call(c):
        for r in range(1, n):
            arn.ar_signal_post(pads, r)
            arn.ar_reduce_scatter_store(inp.partials, temps, r)
            arn.ar_signal_post(pads, r)
        arn.ar_rmsnorm_two_shot(inp.partials, inp.residual, inp.weight, inp.eps, temps, pads, 0,
                                out=out, residual_out=rout)

    t = graph_per_call(call, stream, calls, replays)
    status = arn.ar_device_status(inp.residual.device.index or 0, reset=True)
    del temps
    return t * 1e6, status


def empty_node_floor_us(stream, calls=2000, replays=20):
    """Per-node time of a graph of back-to-back trivial kernels (a one-element
    fill): the launch-and-complete floor any dependent kernel chain pays."""
    import torch
    x = torch.zeros(1, device="cuda")
    return graph_per_call(lambda c: x.fill_(1.0), stream, calls, replays) * 1e6


def rank_latency(arn, inps, eps, stream, calls, replays, kind):
    """Per-call time of one rank's cross-rank call (rank 0 of n = the number
    of partials) when every peer is already there: the peers' flags in every
    pad are set far ahead of rank 0's epochs, so its barriers never wait.
    `kind` "two_shot": ar_rmsnorm_two_shot -- a barrier, rank 0 reduces
    only its own slice into the n temporaries, a barrier, then stage 2 on
    its temporary (the other slices of its output are not those of this
    call).  "one_shot":
    ar_rmsnorm_one_shot -- barrier, the epilogue over all n partials,
    barrier; "one_shot_no_end_barrier" -- the same without the second
    barrier, as a group alternating between two partial buffers runs it.
    The single-rank critical path of each cross-rank path (a timing
    comparator).  Same method as graph_latency."""
    import torch
    n = len(inps[0].partials)
    like = inps[0].residual
    temps = [torch.empty_like(like) for _ in range(n)] if kind == "two_shot" else None
    pads = [torch.zeros(arn.AR_SIGNAL_PAD_BYTES // 4, dtype=torch.int32, device=like.device)
            for _ in range(n)]
    for p in pads:
        p[1:n] = 1 << 30                     # peers 1 .. n-1: far ahead of rank 0's epochs
    outs = [(torch.empty_like(i.residual), torch.empty_like(i.residual)) for i in inps]

    def one(i, o, r):
        if kind == "two_shot":
            arn.ar_rmsnorm_two_shot(i.partials, i.residual, i.weight, eps, temps, pads, 0, out=o,
                                    residual_out=r)
        else:
            arn.ar_rmsnorm_one_shot(i.partials, i.residual, i.weight, eps, pads, 0, out=o,
                                    residual_out=r, end_barrier=kind == "one_shot")

    def call(c):
        one(inps[c % len(inps)], *outs[c % len(outs)])

    def warm():
        for i, (o, r) in zip(inps, outs):
            one(i, o, r)

    return graph_per_call(call, stream, calls, replays, warm)


def latency_table(arn, synth, stream, l2_bytes, quick):
    import torch
    rows = []
    for w in (synth.DECODE, synth.TWO_STAGE):
        for m in w.ms:
            base = synth.make_inputs(w, m, backend="torch", device="cuda")
            set_bytes = algo_bytes(w.n, m, w.H)
            calls = 2000 if set_bytes < 64 << 20 else 200
            replays = 80 if set_bytes < 64 << 20 else 10
            if quick:
                replays = min(replays, 10)
            cold = cold_sets(synth, w, m, base, l2_bytes, calls)
            entry = {"workload": w.name, "n": w.n, "H": w.H, "m": m}
            plan = arn.ar_get_plan(w.n, m, w.H, 0)
            entry["auto_path"] = "two_stage" if plan["mode"] == 2 else "one_stage"
            for mode in ("auto",) + tuple(x for x in ("one_stage", "two_stage") if x != entry["auto_path"]):
                hot = graph_latency(arn, [base], mode, w.eps, stream, calls, replays)
                cold_t = graph_latency(arn, cold, mode, w.eps, stream, calls, replays)
                entry[mode] = {"us_hot": round(hot * 1e6, 3), "us_cold": round(cold_t * 1e6, 3),
                               "gbs_cold": round(set_bytes / cold_t / 1e9, 1)}
            for kind in ("two_shot", "one_shot", "one_shot_no_end_barrier"):
                hot = rank_latency(arn, [base], w.eps, stream, calls, replays, kind)
                cold_t = rank_latency(arn, cold, w.eps, stream, calls, replays, kind)
                entry[kind + "_one_rank"] = {"us_hot": round(hot * 1e6, 3),
                                             "us_cold": round(cold_t * 1e6, 3)}
            rows.append(entry)
            del cold, base
            torch.cuda.empty_cache()
    return rows


def e2e_measure(arn, inp, mode, stream, steps):
    """Same call through the public API with HOST buffers: every step copies
    the inputs from pinned host memory to the device, runs the epilogue and
    copies out and residual_out back; all inside the timed region."""
    import torch
    m, H = inp.residual.shape
    hp = [p.cpu().pin_memory() for p in inp.partials]
    hr = inp.residual.cpu().pin_memory()
    hw = inp.weight.cpu().pin_memory()
    dp = [torch.empty_like(p) for p in inp.partials]
    dr = torch.empty_like(inp.residual)
    dw = torch.empty_like(inp.weight)
    do = torch.empty_like(inp.residual)
    dro = torch.empty_like(inp.residual)
    ho = torch.empty((m, H), dtype=torch.bfloat16).pin_memory()
    hro = torch.empty((m, H), dtype=torch.bfloat16).pin_memory()

    def step():
        with torch.cuda.stream(stream):
            for d, h in zip(dp, hp):
                d.copy_(h, non_blocking=True)
            dr.copy_(hr, non_blocking=True)
            dw.copy_(hw, non_blocking=True)
            arn.ar_rmsnorm(dp, dr, dw, inp.eps, out=do, residual_out=dro, mode=mode)
            ho.copy_(do, non_blocking=True)
            hro.copy_(dro, non_blocking=True)

    settle()
    step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    b.synchronize()
    t = a.elapsed_time(b) / 1e3 / steps
    h2d = sum(x.numel() * 2 for x in hp) + hr.numel() * 2 + hw.numel() * 2
    d2h = ho.numel() * 2 + hro.numel() * 2
    return t, h2d, d2h


def e2e_mapped(arn, inp, mode, stream, steps):
    """The same step with every buffer in pinned host memory: one
    ar_rmsnorm_mapped call, whose kernels read the partials, residual and
    weight from host memory and write out and residual_out to host memory
    over the host link (NVLink-C2C).  Every step moves the inputs host ->
    device and the outputs device -> host inside the timed region; nothing
    is staged in device memory.  Returns (s per step, h2d bytes, d2h bytes)."""
    import torch
    m, H = inp.residual.shape
    hp = [p.cpu().pin_memory() for p in inp.partials]
    hr = inp.residual.cpu().pin_memory()
    hw = inp.weight.cpu().pin_memory()
    ho = torch.empty((m, H), dtype=torch.bfloat16).pin_memory()
    hro = torch.empty((m, H), dtype=torch.bfloat16).pin_memory()

    def step():
        arn.ar_rmsnorm_mapped(hp, hr, hw, inp.eps, out=ho, residual_out=hro, mode=mode,
                              stream=stream, device=inp.residual.device)

    settle()
    step()
    torch.cuda.synchronize()
    # the outputs of the device path, for a check that the host path wrote them
    ref_r = torch.empty_like(inp.residual)
    ref_o = torch.empty_like(inp.residual)
    arn.ar_rmsnorm(inp.partials, inp.residual, inp.weight, inp.eps, out=ref_o,
                   residual_out=ref_r, mode=mode)
    torch.cuda.synchronize()
    same_rout = bool(torch.equal(hro, ref_r.cpu()))
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        step()
    b.record(stream)
    b.synchronize()
    t = a.elapsed_time(b) / 1e3 / steps
    h2d = sum(x.numel() * 2 for x in hp) + hr.numel() * 2 + hw.numel() * 2
    d2h = ho.numel() * 2 + hro.numel() * 2
    return t, h2d, d2h, same_rout


def e2e_pipelined(arn, inp, mode, steps, chunks=8):
    """The same end-to-end step, pipelined over `chunks` row blocks on three
    streams: the host->device copies of block c+1, the epilogue of block c
    (ar_rmsnorm on row-slice views; rows are independent) and the
    device->host copies of block c-1 overlap.  Events order every reuse of a
    device block (a block is refilled only after its previous epilogue, and
    its outputs are rewritten only after their previous copy back).  Returns
    (s per step, h2d bytes, d2h bytes)."""
    import torch
    m, H = inp.residual.shape
    hp = [p.cpu().pin_memory() for p in inp.partials]
    hr = inp.residual.cpu().pin_memory()
    hw = inp.weight.cpu().pin_memory()
    dp = [torch.empty_like(p) for p in inp.partials]
    dr = torch.empty_like(inp.residual)
    dw = torch.empty_like(inp.weight)
    do = torch.empty_like(inp.residual)
    dro = torch.empty_like(inp.residual)
    ho = torch.empty((m, H), dtype=torch.bfloat16).pin_memory()
    hro = torch.empty((m, H), dtype=torch.bfloat16).pin_memory()
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    bounds = [(m * c // chunks, m * (c + 1) // chunks) for c in range(chunks)]
    e_in = [torch.cuda.Event() for _ in range(chunks)]
    e_cmp = [torch.cuda.Event() for _ in range(chunks)]
    e_out = [torch.cuda.Event() for _ in range(chunks)]

    def step():
        s_in.wait_event(e_cmp[-1])        # the weight is read until the last block's epilogue
        with torch.cuda.stream(s_in):
            dw.copy_(hw, non_blocking=True)
        for c, (r0, r1) in enumerate(bounds):
            s_in.wait_event(e_cmp[c])
            with torch.cuda.stream(s_in):
                for d, h in zip(dp, hp):
                    d[r0:r1].copy_(h[r0:r1], non_blocking=True)
                dr[r0:r1].copy_(hr[r0:r1], non_blocking=True)
                e_in[c].record(s_in)
            s_cmp.wait_event(e_in[c])
            s_cmp.wait_event(e_out[c])
            with torch.cuda.stream(s_cmp):
                arn.ar_rmsnorm([d[r0:r1] for d in dp], dr[r0:r1], dw, inp.eps, out=do[r0:r1],
                               residual_out=dro[r0:r1], mode=mode)
                e_cmp[c].record(s_cmp)
            s_out.wait_event(e_cmp[c])
            with torch.cuda.stream(s_out):
                ho[r0:r1].copy_(do[r0:r1], non_blocking=True)
                hro[r0:r1].copy_(dro[r0:r1], non_blocking=True)
                e_out[c].record(s_out)

    def copy_time(pairs, s):
        best = float("inf")
        for _ in range(3):
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(s)
            with torch.cuda.stream(s):
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
            b.record(s)
            b.synchronize()
            best = min(best, a.elapsed_time(b) / 1e3)
        return best

    settle()
    step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record(s_in)
    for _ in range(steps):
        step()
    s_out.wait_event(e_cmp[-1])
    b.record(s_out)
    b.synchronize()
    t = a.elapsed_time(b) / 1e3 / steps
    h2d = sum(x.numel() * 2 for x in hp) + hr.numel() * 2 + hw.numel() * 2
    d2h = ho.numel() * 2 + hro.numel() * 2
    # the host link alone: the step's copies in each direction, one at a time
    t_h2d = copy_time(list(zip(dp, hp)) + [(dr, hr), (dw, hw)], s_in)
    t_d2h = copy_time([(ho, do), (hro, dro)], s_out)
    link = {"h2d_gbs": round(h2d / t_h2d / 1e9, 1), "d2h_gbs": round(d2h / t_d2h / 1e9, 1),
            "bound_ms": round(max(t_h2d, t_d2h) * 1e3, 3)}
    return t, h2d, d2h, link


def cpu_model():
    """The host CPU's model name (lscpu, else /proc/cpuinfo), for the record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=5).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.split(":")[0].strip().lower()
                if key in ("model name", "model", "hardware", "cpu model"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.machine() or "unknown"


def cpu_baseline(synth_inp, n, H, eps, two_stage, budget_s=10.0):
    """The oracle as it stands, timed on the host cores on the first R rows
    of the workload: once single-threaded and once row-parallel over every
    host thread, each the fastest of 3 timed passes over its sample (R sized
    so that the 6 passes take about `budget_s` in all).  ``value`` is the
    all-threads rate; ``single_thread`` the one-thread rate."""
    import oracle
    import synth
    threads = oracle.host_threads()
    m = synth_inp.residual.shape[0]

    def rows_bits(r):
        return ([synth.bits(p[:r]) for p in synth_inp.partials], synth.bits(synth_inp.residual[:r]),
                synth.bits(synth_inp.weight))

    def leg(nthreads, budget):
        probe = min(m, max(nthreads, 16))
        parts, res, w = rows_bits(probe)
        t = time.perf_counter()
        oracle.ar_rmsnorm(parts, res, w, eps, two_stage=two_stage, threads=nthreads)
        per_row = max(time.perf_counter() - t, 1e-6) / probe
        rows = int(min(m, max(probe, budget / 3 / per_row)))
        rows = max(nthreads, rows // nthreads * nthreads) if rows < m else m
        parts, res, w = rows_bits(rows)
        best = float("inf")
        for _ in range(3):
            t = time.perf_counter()
            oracle.ar_rmsnorm(parts, res, w, eps, two_stage=two_stage, threads=nthreads)
            best = min(best, time.perf_counter() - t)
        gbs = algo_bytes(n, rows, H) / best / 1e9
        return gbs, rows, best

    gbs1, rows1, t1 = leg(1, budget_s * 0.4)
    gbsn, rowsn, tn = leg(threads, budget_s * 0.6)
    model = cpu_model()
    return {"value": round(gbsn, 4), "unit": "GB/s", "cores": threads, "kind": "oracle",
            "cpu_model": model,
            "sample": f"first {rowsn} of {m} rows of the workload, {threads} threads, fastest of "
                      f"3 passes ({tn:.3f} s per pass); {model}",
            "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"first {rows1} of {m} rows, 1 thread, fastest of 3 "
                                        f"passes ({t1:.3f} s per pass)"},
            "speedup_all_threads": round(gbsn / gbs1, 2)}


def run_ours(args):
    import torch
    import allreduce_sum_residual_gb300 as arn
    import synth

    world, rank, local = dist_setup(args)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    w = synth.WORKLOADS[args.workload]
    m = args.m or max(w.ms)
    n, H = w.n, w.H
    step_mode = args.mode
    arn.ar_reserve_workspace(m * H, local)
    inp = synth.make_inputs(w, m, backend="torch", device=device, seed=w.seed + rank)
    out = torch.empty_like(inp.residual)
    rout = torch.empty_like(inp.residual)
    stream = torch.cuda.Stream(device)
    plan = arn.ar_get_plan(n, m, H, step_mode)
    if args.kernel != "auto":
        plan["kernel"] = arn.KERNELS[args.kernel]
    path = "two_stage" if plan["mode"] == 2 else "one_stage"
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", L2_BYTES_FALLBACK) or L2_BYTES_FALLBACK

    def step():
        with torch.cuda.stream(stream):
            if args.kernel == "auto":
                arn.ar_rmsnorm(inp.partials, inp.residual, inp.weight, inp.eps, out=out,
                               residual_out=rout, mode=step_mode)
            else:
                arn.ar_rmsnorm_ex(inp.partials, inp.residual, inp.weight, inp.eps, out=out,
                                  residual_out=rout, mode=step_mode, kernel=args.kernel)

    with ClockSampler(local) as clk:
        total, mean_step = timed_steps(step, stream, args.steps, args.warmup, world, device,
                                       use_graph=not args.eager)
    clocks = clk.summary()
    total_max = max_over_ranks(world, total, device)
    bytes_step = algo_bytes(n, m, H)
    value = sum_over_ranks(world, bytes_step * args.steps, device) / total_max / 1e9

    # the other path on the same shape (both are timed for prefill)
    other = "two_stage" if path == "one_stage" else "one_stage"

    def step_other():
        with torch.cuda.stream(stream):
            arn.ar_rmsnorm(inp.partials, inp.residual, inp.weight, inp.eps, out=out,
                           residual_out=rout, mode=other)

    mean_o = mean_step
    if not args.kernel_only:
        _, mean_o = timed_steps(step_other, stream, max(10, min(args.steps, 500)), 3, 1, device,
                                use_graph=not args.eager)
    modes = {path: {"us": round(mean_step * 1e6, 2), "gbs": round(bytes_step / mean_step / 1e9, 1)},
             other: {"us": round(mean_o * 1e6, 2), "gbs": round(bytes_step / mean_o / 1e9, 1),
                     "gbs_actual_bytes": round(actual_bytes(n, m, H, other == "two_stage")
                                               / mean_o / 1e9, 1)}}

    peak, peak_kind = peaks()
    kernel = ("k_reduce_flat" if path == "two_stage" else
              "k_stream_epilogue" if plan["kernel"] == arn.AR_KERNEL_STREAM else "k_fused_epilogue")
    achieved = bytes_step / mean_step / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "peak_note": "the measured peak is a torch copy_ (1:1 read/write); a read-heavy "
                             "kernel can exceed it, so frac_of_nominal is the ceiling-based figure",
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4), "kernel": kernel,
                "bytes_per_launch": bytes_step,
                "traffic": ncu_traffic(kernel, args.workload, plan) if m == max(w.ms) else None}
    if path == "two_stage":
        roofline["note"] = "two launches per step; achieved uses the step's algorithmic bytes"

    # End to end on host buffers: every rank at once (each GPU has its own
    # host link), the job's bytes over the slowest rank's time.
    e2e_job = None
    if not args.kernel_only:
        barrier(world, device)
        t_rank, h2d_rank, d2h_rank, same_rout = e2e_mapped(arn, inp, step_mode, stream,
                                                           3 if args.quick else 10)
        e2e_job = (max_over_ranks(world, t_rank, device),
                   int(sum_over_ranks(world, h2d_rank, device)),
                   int(sum_over_ranks(world, d2h_rank, device)), h2d_rank, d2h_rank, same_rout)

    result = None
    if rank == 0:
        lat, cpu, e2e = [], None, None
        if not args.kernel_only:
            if not args.no_latency:
                lat = latency_table(arn, synth, stream, l2, args.quick)
                modes["unfused_torch"] = {"us": round(unfused_torch_us(inp, stream), 2),
                                          "note": "comparator: separate torch ops in a graph"}
                modes["unfused_torch"]["gbs"] = round(bytes_step / modes["unfused_torch"]["us"]
                                                      / 1e3, 1)
                floor = empty_node_floor_us(stream)
                t_ag = allgather_two_stage_us(arn, inp, stream)
                ag_bytes = bytes_step + (n + 1) * m * H * 2  # n temp copies written + one read back
                modes["two_stage_allgather_stores"] = {
                    "us": round(t_ag, 2), "gbs": round(bytes_step / t_ag / 1e3, 1),
                    "gbs_actual_bytes": round(ag_bytes / t_ag / 1e3, 1),
                    "note": "n rank slices each stored into n temporaries, then stage 2"}
                t_ts, ts_status = two_shot_all_ranks_us(arn, inp, stream)
                modes["two_shot_all_ranks"] = {
                    "us": round(t_ts, 2), "gbs": round(bytes_step / t_ts / 1e3, 1),
                    "gbs_actual_bytes": round(ag_bytes / t_ts / 1e3, 1),
                    "status": arn.ar_strerror(ts_status),
                    "note": "ar_rmsnorm_two_shot of rank 0 after ranks 1..n-1 posted, ran their "
                            "stage 1 and posted again: flag barrier, slices into n temporaries, "
                            "flag barrier, stage 2"}
                t_os = rank_latency(arn, [inp], inp.eps, stream, 20, 5, "one_shot") * 1e6
                modes["one_shot_one_rank"] = {
                    "us": round(t_os, 2), "gbs": round(bytes_step / t_os / 1e3, 1),
                    "status": arn.ar_strerror(arn.ar_device_status(
                        inp.residual.device.index or 0, reset=True)),
                    "note": "ar_rmsnorm_one_shot of rank 0 with every peer's flags already set: "
                            "barrier, the epilogue over all n partials (plain loads, no L2 "
                            "prefetch), barrier"}
            serial_t, _, _ = e2e_measure(arn, inp, step_mode, stream, 3 if args.quick else 10)
            pipe_t, h2d, d2h, link = e2e_pipelined(arn, inp, step_mode, 3 if args.quick else 10)
            e2e_t, h2d_job, d2h_job, h2d_m, d2h_m, same_rout = e2e_job
            assert (h2d_m, d2h_m) == (h2d, d2h)
            e2e = {"value": round(world * bytes_step / e2e_t / 1e9, 2), "unit": "GB/s",
                   "h2d_bytes_per_step": h2d_job, "d2h_bytes_per_step": d2h_job,
                   "ms_per_step": round(e2e_t * 1e3, 3), "ranks": world,
                   "api": "ar_rmsnorm_mapped on pinned host buffers: the kernels read the "
                          "inputs from host memory and write the outputs to host memory over "
                          "NVLink-C2C, one call per step",
                   "scope": "value and bytes: every rank at once, the job's bytes over the "
                            "slowest rank's time; link figures and copy_engines: rank 0",
                   "residual_out_equals_device_path": same_rout,
                   "h2d_plus_d2h_gbs": round((h2d + d2h) / e2e_t / 1e9, 1),
                   "host_link": link,
                   "frac_of_link_bound": round(link["bound_ms"] / (e2e_t * 1e3), 3),
                   "copy_engines": {
                       "ms_per_step": round(pipe_t * 1e3, 3),
                       "value": round(bytes_step / pipe_t / 1e9, 2),
                       "pipeline": "ar_rmsnorm on device buffers; cudaMemcpyAsync of 8 row "
                                   "blocks on 3 streams (copy in / epilogue / copy out)",
                       "serial_ms_per_step": round(serial_t * 1e3, 3)}}
            if world == 1:   # the oracle's baseline is taken at N = 1 only
                cpu = cpu_baseline(inp, n, H, inp.eps, path == "two_stage",
                                   budget_s=2.0 if args.quick else 10.0)
        else:
            modes.pop(other, None)
        result = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(total_max / args.steps * 1e3, 5),
            "us_per_call": round(total_max / args.steps * 1e6, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": f"{w.name}: n={n} bf16 partials, H={H}, m={m}, "
                                   f"{step_mode.upper()} mode",
                       "n": n, "H": H, "m": m, "eps": w.eps, "io_dtype": "bf16", "path": path,
                       "plan": plan, "l2": f"inputs {bytes_step / 1e9:.2f} GB > L2 "
                                           f"{l2 / 2**20:.0f} MiB; no flush needed",
                       "parallelism": f"replicas x{world}",
                       "timing": ("CUDA events around K steps replayed from CUDA graphs on the launch "
                       "stream" if not args.eager else "CUDA events around K eager steps")
                      + ", a device sleep before the start event, max over ranks",
                       "device": {"name": props.name, "sm_count": props.multi_processor_count,
                                  "l2_bytes": l2, "host_cores": os.cpu_count()}},
            "pct_of_8tbs": round(value / world / 8000.0 * 100, 2),
            "roofline": roofline, "modes": modes,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": args.steps * plan["launches"],
            "clocks": clocks,
            "latency_vs_m": lat,
            "empty_kernel_node_floor_us": round(floor, 3) if lat else None,
            # the device status word after every timed kernel (a bounded wait
            # that gave up would show here)
            "device_status": arn.ar_strerror(arn.ar_device_status(local)),
        }
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        barrier(world, device)
        dist.destroy_process_group()
    return result


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return None
    import oracle
    import synth
    import torch
    w = synth.WORKLOADS[args.workload]
    n, H, m = w.n, w.H, max(w.ms)
    threads = oracle.host_threads()
    budget = 60.0 if not args.quick else 5.0
    # calibrate rows per step so that warm-up + timed steps take ~budget seconds
    probe = synth.make_inputs(w, threads, backend="numpy")
    pb = [synth.bits(p) for p in probe.partials], synth.bits(probe.residual), synth.bits(probe.weight)
    t = time.perf_counter()
    oracle.ar_rmsnorm(*pb, w.eps, threads=threads)
    per_row = (time.perf_counter() - t) / threads
    rows = int(max(1, min(m, budget / max(1, args.steps + args.warmup) / max(per_row, 1e-9))))
    sample = synth.make_inputs(w, rows, backend="numpy")
    sb = [synth.bits(p) for p in sample.partials], synth.bits(sample.residual), synth.bits(sample.weight)
    two = False  # the oracle's one-stage definition; AUTO picks one-stage on this workload
    for _ in range(args.warmup):
        oracle.ar_rmsnorm(*sb, w.eps, two_stage=two, threads=threads)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.ar_rmsnorm(*sb, w.eps, two_stage=two, threads=threads)
    total = time.perf_counter() - t
    del torch
    bytes_step = algo_bytes(n, rows, H)
    value = bytes_step * args.steps / total / 1e9
    res = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
           "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": round(total / args.steps * 1e3, 4),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
           "data": "synthetic",
           "config": {"workload": f"{w.name}: n={n} bf16 partials, H={H}, m={m}, AUTO mode",
                      "n": n, "H": H, "m": m, "eps": w.eps, "io_dtype": "bf16"},
           "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                            "kind": "oracle",
                            "sample": f"{rows} of {m} rows per step (host numpy generator), "
                                      f"{threads} threads"},
           "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(res), flush=True)
    return res


# ---------------------------------------------------------------- sweep

def run_sweep(args):
    """Both paths on every sweep shape (cold buffers, graph method); one JSON
    line per shape.  Feeds the one-/two-stage threshold table."""
    import torch
    import allreduce_sum_residual_gb300 as arn
    import synth
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    props = torch.cuda.get_device_properties(0)
    l2 = getattr(props, "L2_cache_size", L2_BYTES_FALLBACK) or L2_BYTES_FALLBACK
    arn.ar_reserve_workspace(16384 * 8192, 0)
    for w in synth.SWEEP:
        for m in w.ms:
            set_bytes = algo_bytes(w.n, m, w.H)
            calls = 2000 if set_bytes < 32 << 20 else 100
            replays = 40 if set_bytes < 32 << 20 else 5
            base = synth.make_inputs(w, m, backend="torch", device="cuda")
            inps = cold_sets(synth, w, m, base, l2, calls)
            row = {"n": w.n, "H": w.H, "m": m, "bytes": set_bytes, "sets": len(inps)}
            for mode in ("one_stage", "two_stage"):
                t = graph_latency(arn, inps, mode, w.eps, stream, calls, replays)
                row[mode] = {"us": round(t * 1e6, 3), "gbs": round(set_bytes / t / 1e9, 1)}
            print(json.dumps(row), flush=True)
            del inps, base
            torch.cuda.empty_cache()


def run_shapes(args):
    """Register-kernel launch shapes (cluster x packs per thread) on the
    decode and mid-size shapes; graph method, hot and cold; one JSON line
    per (shape, m).  Feeds the launch plan."""
    import torch
    import allreduce_sum_residual_gb300 as arn
    import synth
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    props = torch.cuda.get_device_properties(0)
    l2 = getattr(props, "L2_cache_size", L2_BYTES_FALLBACK) or L2_BYTES_FALLBACK
    cases = [(synth.DECODE, m) for m in synth.DECODE.ms] + [(synth.TWO_STAGE, m) for m in (32, 64, 128, 256)]
    for w, m in cases:
        base = synth.make_inputs(w, m, backend="torch", device="cuda")
        cold = cold_sets(synth, w, m, base, l2, 2000)
        auto = arn.ar_get_plan(w.n, m, w.H, 1)
        P = w.H // 8
        for cluster in (1, 2, 4, 8, 16):
            for vpt in (1, 2, 4):
                if -(-P // cluster) > 1024 or -(-(-(-P // cluster)) // vpt) > 1024 // vpt:
                    continue
                shape = ("register", cluster, vpt)
                hot = graph_latency(arn, [base], "one_stage", w.eps, stream, 2000, 20, shape)
                cold_t = graph_latency(arn, cold, "one_stage", w.eps, stream, 2000, 20, shape)
                print(json.dumps({"n": w.n, "H": w.H, "m": m, "cluster": cluster, "vpt": vpt,
                                  "auto": auto["cluster"] == cluster and auto["vpt"] == vpt
                                  and auto["kernel"] == 1,
                                  "us_hot": round(hot * 1e6, 3), "us_cold": round(cold_t * 1e6, 3)}),
                      flush=True)
        del cold, base
        torch.cuda.empty_cache()


# bench.py --kernels candidates: name -> forced (kernel, cluster, vpt)
KERNEL_CANDIDATES = {"stream": ("stream", 0, 0),
                     **{f"register{v}": ("register", 0, v) for v in (1, 2, 4, 8)},
                     **{f"late{v}": ("register_late", 0, v) for v in (1, 2, 4, 8)}}


def run_kernels(args):
    """Register vs stream kernel for one-stage at many rows, over n and H
    (graph method, cold sets); one JSON line per case."""
    import torch
    import allreduce_sum_residual_gb300 as arn
    import synth
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    props = torch.cuda.get_device_properties(0)
    l2 = getattr(props, "L2_cache_size", L2_BYTES_FALLBACK) or L2_BYTES_FALLBACK
    ints = lambda s: tuple(int(x) for x in s.split(","))
    for n in ints(args.kernel_ns):
        for H in ints(args.kernel_hs):
            for m in ints(args.kernel_ms):
                w = synth.Workload("k", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0)
                set_bytes = algo_bytes(n, m, H)
                calls = 2000 if set_bytes < 32 << 20 else 100
                replays = 20 if set_bytes < 32 << 20 else 5
                base = synth.make_inputs(w, m, backend="torch", device="cuda")
                inps = cold_sets(synth, w, m, base, l2, calls)
                row = {"n": n, "H": H, "m": m, "bytes": set_bytes}
                shapes = [None] + [KERNEL_CANDIDATES[c] for c in args.kernel_cands.split(",")]
                for key, shape in zip(["auto"] + args.kernel_cands.split(","), shapes):
                    try:
                        t = graph_latency(arn, inps, "one_stage", w.eps, stream, calls, replays, shape)
                        row[key] = round(set_bytes / t / 1e9, 1)
                    except arn.ArError:
                        pass
                print(json.dumps(row), flush=True)
                del inps, base
                torch.cuda.empty_cache()


def run_stream_shapes(args):
    """Stream-kernel shapes (tile width, CTAs per SM) against the register
    kernel, one-stage, m = 8192, cold; one JSON line per (n, H)."""
    import torch
    import allreduce_sum_residual_gb300 as arn
    import synth
    torch.cuda.set_device(0)
    stream = torch.cuda.Stream()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    m = 8192
    for n in (3, 4, 8, 16):
        for H in (4096, 6144, 7168):
            w = synth.Workload("s", n=n, H=H, ms=(m,), p_std=0.5, res_std=1.0)
            inp = synth.make_inputs(w, m, backend="torch", device="cuda")
            B = algo_bytes(n, m, H)
            row = {"n": n, "H": H, "m": m}
            shapes = [("register", 0, v) for v in (1, 2, 4)] + [
                ("stream", 0, 0, 32 + tc, 0, c) for tc in (128, 256, 384, 512) for c in (sms, 2 * sms)]
            for sh in shapes:
                key = sh[0] + (f"_v{sh[2]}" if sh[0] == "register" else f"_tc{sh[3] - 32}_g{sh[5]}")
                try:
                    t = graph_latency(arn, [inp], "one_stage", w.eps, stream, 100, 10, sh)
                    row[key] = round(B / t / 1e9, 1)
                except arn.ArError:
                    row[key] = None
            print(json.dumps(row), flush=True)
            del inp
            torch.cuda.empty_cache()


# AR_MODE=auto|one_stage|two_stage (or 0|1|2) forces the path of the bench's
# timed step, as the pages' AITER_AR_1STAGE switch forces theirs (ROCm/aiter
# #3817, Test Plan, Benchmark); the library itself takes the mode as an
# argument.
_ENV_MODES = {"0": "auto", "1": "one_stage", "2": "two_stage",
              "auto": "auto", "one_stage": "one_stage", "two_stage": "two_stage"}


def env_mode():
    v = os.environ.get("AR_MODE", "auto").strip().lower()
    if v not in _ENV_MODES:
        raise SystemExit(f"AR_MODE={v!r}: expected auto, one_stage, two_stage, 0, 1 or 2")
    return _ENV_MODES[v]


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="prefill", choices=("prefill", "decode", "two_stage", "tiny"))
    ap.add_argument("--sweep", action="store_true")
    ap.add_argument("--shapes", action="store_true", help="register-kernel launch-shape sweep")
    ap.add_argument("--kernels", action="store_true", help="register vs stream kernel sweep")
    ap.add_argument("--stream-shapes", action="store_true", help="stream-kernel shape sweep")
    ap.add_argument("--kernel-ns", default="1,2,3,4,8,16", help="--kernels: input counts")
    ap.add_argument("--kernel-hs", default="4096,7168", help="--kernels: hidden sizes")
    ap.add_argument("--kernel-ms", default="304,1024,4096,16384", help="--kernels: token counts")
    ap.add_argument("--kernel-cands", default=",".join(KERNEL_CANDIDATES),
                    help="--kernels: candidates (stream, register1..8, late1..8)")
    ap.add_argument("--quick", action="store_true", help="shorter latency table and baselines")
    ap.add_argument("--no-latency", action="store_true")
    ap.add_argument("--m", type=int, default=0, help="token count (default: the workload's)")
    ap.add_argument("--mode", default=env_mode(), choices=("auto", "one_stage", "two_stage"),
                    help="the path (default: $AR_MODE, else auto)")
    ap.add_argument("--kernel", default="auto", choices=("auto", "register", "register_late", "stream"),
                    help="force the epilogue kernel (profiling)")
    ap.add_argument("--eager", action="store_true",
                    help="launch the timed steps one by one from Python instead of from graphs")
    ap.add_argument("--kernel-only", action="store_true",
                    help="only the timed steps (no latency table, e2e or CPU baseline)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.shapes:
        return run_shapes(args)
    if args.kernels:
        return run_kernels(args)
    if args.stream_shapes:
        return run_stream_shapes(args)
    return run_ours(args)


if __name__ == "__main__":
    main()
