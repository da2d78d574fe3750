"""Benchmark of the virtual-rank ring AllReduce on GB300.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME]

One step = one vrAllReduce of the whole workload (every stage of the ring, all
channels) on inputs already resident in HBM. Prints ONE JSON line (rank 0):
value = whole-job busBW in GB/s (busBW = algBW * 2(N-1)/N, algBW = B / t, B =
bytes per virtual rank), with the roofline of the ring kernel against the
measured HBM copy bandwidth, the end-to-end figure through the public API with
host buffers, the CPU oracle as a baseline, and the SM clocks seen while
timing. Under torchrun (N > 1 GPUs) every GPU runs an independent replica of
the workload (the path has no cross-GPU exchange on this machine: replicas only);
timing is the max over ranks.

--impl reference times the CPU oracle (the plain fold) on the host cores, on
a bounded sample of the same workload.
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
sys.path.insert(0, ROOT)

L2_BYTES = 126 * (1 << 20)
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
# GPU cycles the stream is held before a timed loop, so that the host has
# enqueued every timed call before the GPU reaches the first (~25 ms).
STREAM_HOLD_CYCLES = 50_000_000


def kernel_source_hash():
    """Hash of the CUDA sources: ncu traffic figures are only reported for the
    kernel build they were taken on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ring_allreduce_virtual_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode())
            h.update(f.read())
    return h.hexdigest()[:16]


def hbm_peak():
    try:
        with open(PEAKS_FILE) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload):
    """dram read+write bytes per launch from the committed ncu summary, if it
    was taken on the current kernel sources."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get(workload)
    if not entry or entry.get("source_hash") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for name, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        loaded = [v for v in sm if mx and v > 0.5 * mx] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, ws, dev):
    """The largest of every rank's `x` (a float): the whole job takes as long
    as its slowest replica. `dev` is the rank's CUDA device (NCCL); with the
    gloo backend the reduction runs on the host."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    if dist.get_backend() == "gloo":
        dev = torch.device("cpu")
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(bytes_per_rank, n_ranks, seconds, world_size):
    """Whole-job busBW of `world_size` replicas that each ran the workload in
    `seconds` (already the max over ranks): each replica contributes its own
    busBW."""
    _, bus = bus_bw(bytes_per_rank, n_ranks, seconds)
    return bus * world_size


METRICS = {"allreduce": "virtual-rank AllReduce busBW (GB/s)",
           "reducescatter": "virtual-rank ReduceScatter busBW (GB/s)",
           "allgather": "virtual-rank AllGather busBW (GB/s)"}


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def bus_bw(bytes_per_rank, n_ranks, seconds):
    alg = bytes_per_rank / seconds / 1e9
    return alg, alg * 2 * (n_ranks - 1) / n_ranks


def cpu_oracle_run(w, xs_host, nthreads, channels_sample):
    """One oracle run over `channels_sample` of the workload's channels
    (whole channels, so the chunk structure is the workload's own)."""
    import oracle
    per = oracle.channel_range(w.count, w.n_channels, w.elem_size, 0)[1]
    count = min(w.count, per * channels_sample)
    t0 = time.perf_counter()
    oracle.allreduce([x[:count] for x in xs_host], w.dtype, w.op, channels_sample, w.chunk_bytes,
                     nthreads=nthreads)
    return time.perf_counter() - t0, count


def host_inputs(w, dev):
    """The workload's inputs, drawn on the GPU and copied to the host."""
    from ring_allreduce_virtual_gb300 import synthetic
    xs = synthetic.rank_buffers(w.n_ranks, w.count, w.dtype, w.dist, w.seed, dev)
    out = [synthetic.to_numpy(x) for x in xs]
    del xs
    return out


def cpu_baseline(w, dev, budget_s=12.0):
    """The oracle as it stands on all host cores, on whole channels of the
    workload, repeated until about `budget_s` of CPU time."""
    nthreads = os.cpu_count() or 1
    xs = host_inputs(w, dev)
    per = None
    sample_ch = w.n_channels
    times = []
    t_start = time.perf_counter()
    while True:
        dt, count = cpu_oracle_run(w, xs, nthreads, sample_ch)
        times.append(dt)
        per = count
        if time.perf_counter() - t_start > budget_s or len(times) >= 20:
            break
    t = statistics.median(times)
    alg, bus = bus_bw(per * w.elem_size, w.n_ranks, t)
    # The same oracle on one core, over one channel (best of three runs or
    # about two seconds).
    t1, per1 = None, None
    t_start = time.perf_counter()
    for _ in range(3):
        dt, per1 = cpu_oracle_run(w, xs, 1, 1)
        t1 = dt if t1 is None else min(t1, dt)
        if time.perf_counter() - t_start > 2.0:
            break
    _, bus1 = bus_bw(per1 * w.elem_size, w.n_ranks, t1)
    return {"value": round(bus, 3), "unit": "GB/s busBW", "cores": nthreads, "kind": "oracle",
            "sample": f"{sample_ch} of {w.n_channels} channels ({per} elements per rank), "
                      f"median of {len(times)} runs, {t:.3f} s each",
            "algbw_gbs": round(alg, 3),
            "single_thread": {"value": round(bus1, 3), "unit": "GB/s busBW", "cores": 1,
                              "sample": f"1 of {w.n_channels} channels ({per1} elements per "
                                        f"rank), best run {t1:.3f} s"}}


# Per-rank elements of the halves' sample on the host: the oracle's
# ReduceScatter and AllGather run on one core.
HALF_SAMPLE_ELEMS = 1 << 22


def cpu_half_run(w, xs_host, coll):
    """One oracle ReduceScatter or AllGather over the first HALF_SAMPLE_ELEMS
    elements (whole blocks) of each rank's buffer; returns (seconds, elements
    per rank of the AllReduce-sized buffer the sample stands for)."""
    import oracle
    n = w.n_ranks
    blk = min(w.count, HALF_SAMPLE_ELEMS) // n
    t0 = time.perf_counter()
    if coll == "reducescatter":
        oracle.reduce_scatter([x[: n * blk] for x in xs_host], w.dtype, w.op)
    else:
        oracle.all_gather([x[:blk] for x in xs_host], w.dtype)
    return time.perf_counter() - t0, n * blk


def run_reference(args, w):
    import torch
    ws, rank, local = dist_env()
    if rank != 0:
        return
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    nthreads = os.cpu_count() or 1
    xs = host_inputs(w, dev)
    if args.coll == "allreduce":
        run = lambda: cpu_oracle_run(w, xs, nthreads, w.n_channels)
        sample = f"all {w.n_channels} channels"
    else:
        run = lambda: cpu_half_run(w, xs, args.coll)
        nthreads = 1
        sample = f"the first {min(w.count, HALF_SAMPLE_ELEMS) // w.n_ranks} elements of each block"
    for _ in range(args.warmup):
        run()
    times = []
    for _ in range(args.steps):
        dt, count = run()
        times.append(dt)
    t = statistics.mean(times)
    if args.coll == "allreduce":
        alg, bus = bus_bw(count * w.elem_size, w.n_ranks, t)
    else:
        alg = count * w.elem_size / t / 1e9
        bus = alg * (w.n_ranks - 1) / w.n_ranks
    line = {"impl": "reference", "metric": METRICS[args.coll],
            "value": round(bus, 3), "unit": "GB/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": {"float32": "f32",
            "bfloat16": "bf16", "float16": "f16", "int32": "i32"}.get(w.dtype, w.dtype),
            "data": "synthetic",
            "config": {"workload": w.name, "collective": args.coll, "n_ranks": w.n_ranks,
                       "count": w.count,
                       "proto": w.proto, "channels": w.n_channels, "chunk_bytes": w.chunk_bytes},
            "cpu_baseline": {"value": round(bus, 3), "unit": "GB/s busBW", "cores": nthreads,
                             "kind": "oracle",
                             "sample": f"{sample} ({count} elements per rank)"},
            "e2e": {"value": round(bus, 3), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args, w):
    import torch
    import ring_allreduce_virtual_gb300 as vr
    from ring_allreduce_virtual_gb300 import synthetic

    ws, rank, local = dist_env()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    vr.lib()
    stream = torch.cuda.current_stream()

    # The workload's rank buffers of B bytes. AllReduce: B in, B out per rank.
    # ReduceScatter: B in, B/N out. AllGather: B/N in, B out (NCCL's sizes:
    # algBW = B / t for all three).
    n = w.n_ranks
    xs = synthetic.rank_buffers(n, w.count, w.dtype, w.dist, w.seed, dev)
    if args.coll == "allreduce":
        outs = [torch.empty_like(x) for x in xs]
    elif args.coll == "reducescatter":
        outs = [torch.empty(w.count // n, dtype=xs[0].dtype, device=dev) for _ in xs]
    else:
        xs = [x[: w.count // n].clone() for x in xs]
        outs = [torch.empty(w.count, dtype=xs[0].dtype, device=dev) for _ in xs]
    in_bytes = sum(x.numel() * x.element_size() for x in xs)
    out_bytes = sum(o.numel() * o.element_size() for o in outs)
    total_in = in_bytes
    flush = None
    if in_bytes + out_bytes < 8 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    comm = vr.Communicator(w.n_ranks, w.n_channels, w.proto, w.chunk_bytes)

    def step():
        if args.coll == "allreduce" and args.algo == "tree":
            comm.all_reduce_tree(xs, outs, w.op, stream=stream, dtype=w.dtype)
        elif args.coll == "allreduce":
            comm.all_reduce(xs, outs, w.op, stream=stream, dtype=w.dtype)
        elif args.coll == "reducescatter":
            comm.reduce_scatter(xs, outs, w.op, stream=stream, dtype=w.dtype)
        else:
            comm.all_gather(xs, outs, stream=stream, dtype=w.dtype)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if comm.async_error() != vr.vrSuccess:
        raise RuntimeError("device wait timed out during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        # Hold the stream for a moment so that the host enqueues every timed
        # step before the GPU reaches the first: the events then time the
        # device alone, not the host's launch latency (that is in e2e).
        torch.cuda._sleep(STREAM_HOLD_CYCLES)
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize()
    barrier(ws)
    if comm.async_error() != vr.vrSuccess:
        raise RuntimeError("device wait timed out while timing")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    t_local = sum(step_ms) / len(step_ms) / 1e3
    t = max_over_ranks(t_local, ws, dev)
    if args.coll == "allreduce":
        alg, bus = bus_bw(w.bytes_per_rank, w.n_ranks, t)
        value = job_value(w.bytes_per_rank, w.n_ranks, t, ws)
    else:  # the halves move (N-1)/N of the data over the ring
        alg = w.bytes_per_rank / t / 1e9
        bus = alg * (n - 1) / n
        value = bus * ws
    peak, peak_kind = hbm_peak()
    algorithmic = in_bytes + out_bytes  # every input byte read once, every output written once
    achieved = algorithmic / t / 1e9

    # End to end through the public API: H2D of every rank's input from pinned
    # host memory, the AllReduce, D2H of every rank's output, per step.
    e2e = None
    if not args.no_e2e:
        hx = [torch.empty(x.shape, dtype=x.dtype, pin_memory=True) for x in xs]
        # The host's inputs are written by the CPU, as a host program's data
        # would be (pinned pages last written by the GPU were measured to
        # stream back to it 2.5-4x slower).
        for h, x in zip(hx, xs):
            h.copy_(x.cpu())
        ho = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs]
        e_steps = max(2, min(args.steps, 4))
        es, ee = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        # Inputs come in on one copy stream and results go out on another, so
        # step i's results travel to the host while step i+1's inputs travel
        # to the device (the two directions of the link run at once). Step
        # i+1's inputs wait for step i's call to have read them, and step
        # i+1's call waits for step i's results to have left.
        cin, cout = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

        def e2e_steps(k, start=None):
            called = out_done = None
            for _ in range(k):
                with torch.cuda.stream(cin):
                    if start is not None:
                        cin.wait_event(start)
                    if called is not None:
                        cin.wait_event(called)
                    for h, x in zip(hx, xs):
                        x.copy_(h, non_blocking=True)
                    in_done = torch.cuda.Event()
                    in_done.record(cin)
                stream.wait_event(in_done)
                if out_done is not None:
                    stream.wait_event(out_done)
                step()
                called = torch.cuda.Event()
                called.record(stream)
                with torch.cuda.stream(cout):
                    cout.wait_event(called)
                    for h, o in zip(ho, outs):
                        h.copy_(o, non_blocking=True)
                    out_done = torch.cuda.Event()
                    out_done.record(cout)
            stream.wait_event(out_done)

        e2e_steps(1)
        torch.cuda.synchronize()
        barrier(ws)
        es.record(stream)
        e2e_steps(e_steps, start=es)
        ee.record(stream)
        torch.cuda.synchronize()
        te = max_over_ranks(es.elapsed_time(ee) / 1e3 / e_steps, ws, dev)
        ebus = bus * t / te  # the same metric over the end-to-end time
        e2e = {"value": round(ebus * ws, 3), "unit": "GB/s",
               "h2d_bytes_per_step": in_bytes, "d2h_bytes_per_step": out_bytes,
               "ms_per_step": round(te * 1e3, 3), "steps": e_steps,
               "copies": "H2D of step i+1 overlaps D2H of step i (two copy streams)"}
        del hx, ho

    # Calibration: the ring-walk fold (vrRingWalk) on the same inputs and
    # outputs, timed the same way. Same result bit for bit, least traffic, no
    # ring: the attainable ceiling, reported beside the metric, not in it.
    calib = None
    if args.coll == "allreduce" and not args.no_calibration:
        for _ in range(args.warmup):
            comm.ring_walk(xs, outs, w.op, stream=stream, dtype=w.dtype)
        cs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ce = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        torch.cuda.synchronize()
        torch.cuda._sleep(STREAM_HOLD_CYCLES)
        for i in range(args.steps):
            if flush is not None:
                flush.zero_()
            cs[i].record(stream)
            comm.ring_walk(xs, outs, w.op, stream=stream, dtype=w.dtype)
            ce[i].record(stream)
        torch.cuda.synchronize()
        walk_ms = [a.elapsed_time(b) for a, b in zip(cs, ce)]
        tw = max_over_ranks(sum(walk_ms) / len(walk_ms) / 1e3, ws, dev)
        calib = {"kernel": "vr_ring_walk", "ms_per_step": round(tw * 1e3, 4),
                 "ms_best": round(min(walk_ms), 4),
                 "achieved": round(algorithmic / tw / 1e9, 2),
                 "frac": round(algorithmic / tw / 1e9 / peak, 4),
                 "ring_time_over_walk_time": round(t / tw, 3)}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline and args.coll == "allreduce":
        cpu = cpu_baseline(w, dev)

    info = comm.info()
    comm.destroy()
    if rank == 0:
        line = {
            "metric": METRICS[args.coll] if args.algo == "ring"
            else "virtual-rank double-binary-tree AllReduce busBW (GB/s)",
            "value": round(value, 3), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t * 1e3, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": {"float32": "f32", "bfloat16": "bf16", "float16": "f16",
                      "int32": "i32"}.get(w.dtype, w.dtype),
            "data": "synthetic",
            "config": {"workload": w.name, "collective": args.coll, "algorithm": args.algo,
                       "n_ranks": w.n_ranks, "count": w.count,
                       "bytes_per_rank": w.bytes_per_rank, "dist": w.dist, "op": w.op,
                       "proto": w.proto, "channels": w.n_channels, "chunk_bytes": w.chunk_bytes,
                       "transport": info["transport"], "fifo_slot_bytes": info["slot_bytes"],
                       "fifo_depth": info["depth"],
                       "cache": "L2 flushed between steps" if flush is not None
                       else "inputs larger than L2", "parallelism": f"replicas x{ws}",
                       "algbw_gbs": round(alg, 3), "busbw_gbs_per_gpu": round(bus, 3),
                       "frac_of_nominal_8000": round(achieved / NOMINAL_HBM_GBS, 4)},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                         "peak_kind": peak_kind, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": recorded_traffic(w.name) if args.coll == "allreduce"
                         else None,
                         "algorithmic_bytes_per_launch": algorithmic},
            "timing": {"ms_mean": round(t * 1e3, 4),
                       "ms_median": round(statistics.median(step_ms), 4),
                       "ms_best": round(min(step_ms), 4)},
            "calibration": calib,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clocks.summary(),
            "gpu_launches": args.steps * ws,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# The message-size sweep: 8 ranks, int32 U-int[-2^20, 2^20], 16 channels,
# every per-rank size 2^3 .. 2^28 bytes, sum and max, per protocol (chunk
# 512 KiB for Simple and LL128, 64 KiB for LL); 4 and 16 ranks at a few sizes
# so that the cost model can tell the per-call cost from the per-step cost.
SWEEP_SIZES = [1 << k for k in range(3, 29)]
SWEEP_FEW = [1 << 10, 1 << 16, 1 << 20, 1 << 24, 1 << 28]
SWEEP_CHUNK = {"simple": 512 << 10, "ll": 64 << 10, "ll128": 512 << 10}


def time_calls(fn, steps, warmup, flush, stream):
    """Mean, median and best milliseconds of `fn` over `steps` calls, timed
    with CUDA events on `stream` after `warmup` calls, L2 flushed before each
    timed call when `flush` is given."""
    import torch
    for _ in range(warmup):
        fn()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    torch.cuda._sleep(STREAM_HOLD_CYCLES)
    for i in range(steps):
        if flush is not None:
            flush.zero_()
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    return sum(ms) / len(ms), statistics.median(ms), min(ms)


def run_sweep(args):
    """busBW and roofline fraction vs message size, one JSON line per point,
    then the ring cost model fitted to the points with its predictions."""
    import torch
    import ring_allreduce_virtual_gb300 as vr
    from ring_allreduce_virtual_gb300 import costmodel, synthetic

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    vr.lib()
    stream = torch.cuda.current_stream()
    peak, peak_kind = hbm_peak()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    plan = []
    for proto in ("simple", "ll", "ll128"):
        plan.append((8, proto, SWEEP_SIZES, ("sum", "max")))
        plan.append((4, proto, SWEEP_FEW, ("sum",)))
        plan.append((16, proto, SWEEP_FEW, ("sum",)))
    points = {p: [] for p in ("simple", "ll", "ll128")}
    pass_points = {p: [] for p in ("simple", "ll", "ll128")}
    stage_points = {p: [] for p in ("simple", "ll", "ll128")}
    n8_passes = {p: {} for p in ("simple", "ll", "ll128")}
    n8_stages = {p: {} for p in ("simple", "ll", "ll128")}
    for n, proto, sizes, ops in plan:
        xs = synthetic.rank_buffers(n, max(sizes) // 4, "int32", "int:-1048576:1048576",
                                    synthetic.SEED_BASE + 2, dev)
        outs = [torch.empty_like(x) for x in xs]
        with vr.Communicator(n, 16, proto, SWEEP_CHUNK[proto]) as comm:
            transport = comm.info()["transport"]
            for size in sizes:
                count = size // 4
                sx, so = [x[:count] for x in xs], [o[:count] for o in outs]
                parts, rings = comm.plan(count, "int32")
                n_passes = costmodel.passes(parts, rings)
                n_stages = costmodel.data_stages(count, n, 16, SWEEP_CHUNK[proto], 4)
                big = 2 * n * size >= 4 * L2_BYTES
                fl = None if big else flush
                for op in ops:
                    t, med, best = time_calls(
                        lambda: comm.all_reduce(sx, so, op, stream=stream), args.steps,
                        args.warmup, fl, stream)
                    tw, _, _ = time_calls(lambda: comm.ring_walk(sx, so, op, stream=stream),
                                          args.steps, args.warmup, fl, stream)
                    if comm.async_error() != vr.vrSuccess:
                        raise RuntimeError("device wait timed out in the sweep")
                    alg, bus = bus_bw(size, n, t / 1e3)
                    achieved = 2 * n * size / (t / 1e3) / 1e9
                    print(json.dumps({
                        "sweep": "int32 ring AllReduce", "n_ranks": n, "proto": proto,
                        "op": op, "bytes_per_rank": size, "transport": transport,
                        "ms_per_step": round(t, 5), "ms_median": round(med, 5),
                        "ms_best": round(best, 5),
                        "busbw_gbs": round(bus, 3), "algbw_gbs": round(alg, 3),
                        "roofline_frac": round(achieved / peak, 4) if big else None,
                        "walk_ms_per_step": round(tw, 5), "parts": parts, "rings": rings,
                        "passes": n_passes, "data_stages": n_stages,
                        "cache": "inputs larger than L2" if big else "L2 flushed between steps"}),
                        flush=True)
                    if op == "sum":
                        points[proto].append((size, n, med * 1e3))
                        pass_points[proto].append((size, n, n_passes, med * 1e3))
                        stage_points[proto].append((size, n, parts, rings, n_stages, med * 1e3))
                        if n == 8:
                            n8_passes[proto][size] = n_passes
                            n8_stages[proto][size] = (parts, rings, n_stages)
        del xs, outs
        torch.cuda.empty_cache()
    fits = {p: costmodel.fit(pts) for p, pts in points.items()}
    model = {}
    for p, f in fits.items():
        res = costmodel.residuals(f, points[p])
        model[p] = {"base_us": round(f.base_us, 3), "hop_us": round(f.hop_us, 4),
                    "bus_gbs": round(f.bus_gbs, 2),
                    "discount_fitted": round(f.bus_gbs / fits["simple"].bus_gbs, 3),
                    "discount_pages": round(costmodel.PAGE_DISCOUNT[p], 3),
                    "median_abs_rel_err": round(float(statistics.median(abs(r) for r in res)), 3),
                    "max_abs_rel_err": round(float(max(abs(r) for r in res)), 3)}
    pfits = {p: costmodel.fit_passes(pts) for p, pts in pass_points.items()}
    pmodel = {}
    for p, f in pfits.items():
        res = costmodel.residuals_passes(f, pass_points[p])
        pmodel[p] = {"base_us": round(f.base_us, 3), "stage_us": round(f.stage_us, 4),
                     "bus_gbs": round(f.bus_gbs, 2),
                     "median_abs_rel_err": round(float(statistics.median(abs(r) for r in res)), 3),
                     "max_abs_rel_err": round(float(max(abs(r) for r in res)), 3)}

    sfits = {p: costmodel.fit_steps(pts) for p, pts in stage_points.items()}
    smodel = {}
    for p, f in sfits.items():
        res = costmodel.residuals_steps(f, stage_points[p])
        smodel[p] = {"base_us": round(f.base_us, 3), "step_us": round(f.step_us, 4),
                     "warp_gbs": round(f.warp_gbs(), 3),
                     "median_abs_rel_err": round(float(statistics.median(abs(r) for r in res)), 3),
                     "max_abs_rel_err": round(float(max(abs(r) for r in res)), 3)}

    def stays_below(faster, slower, sizes):
        later = [b for i, b in enumerate(sizes)
                 if all(faster[c] < slower[c] for c in sizes[i:])]
        return later[0] if later else None

    cross, cross_p, cross_s, seen = {}, {}, {}, {}
    t8 = {p: {b: t for b, n, t in pts if n == 8} for p, pts in points.items()}
    sizes = sorted(t8["simple"])
    for small, large in (("ll", "simple"), ("ll", "ll128"), ("ll128", "simple")):
        key = f"{small}_to_{large}"
        x = costmodel.crossover_bytes(fits[small], fits[large], 8)
        cross[key] = None if x is None else int(x)
        # from the pass model, and measured: the smallest size from which
        # `large` stays faster
        pred = {p: {b: costmodel.predict_passes_us(pfits[p], 8, n8_passes[p][b], b)
                    for b in sizes} for p in (small, large)}
        cross_p[key] = stays_below(pred[large], pred[small], sizes)
        spred = {p: {b: costmodel.predict_steps_us(sfits[p], 8, *n8_stages[p][b], b)
                     for b in sizes} for p in (small, large)}
        cross_s[key] = stays_below(spred[large], spred[small], sizes)
        seen[key] = stays_below(t8[large], t8[small], sizes)
    print(json.dumps({"cost_model": model, "crossover_bytes_per_rank_n8": cross,
                      "pass_model": pmodel,
                      "pass_model_formula": "t_us = base + ceil(parts / rings) (2N - 1) stage"
                                            " + B / (1000 * bus * N / (2(N-1)))",
                      "crossover_pass_model_bytes_per_rank_n8": cross_p,
                      "step_model": smodel,
                      "step_model_formula": "t_us = base + ceil(parts / rings) (2 ne - 1)"
                                            " (step + B / (parts N) / (1000 warp_gbs)),"
                                            " ne = chunks of a loop holding data",
                      "crossover_step_model_bytes_per_rank_n8": cross_s,
                      "crossover_measured_bytes_per_rank_n8": seen,
                      "formula": "t_us = base + 2(N-1) hop + B / (1000 * bus * N / (2(N-1)))",
                      "peak": peak, "peak_kind": peak_kind}), flush=True)


def main():
    from ring_allreduce_virtual_gb300 import workloads
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=workloads.HEADLINE.name,
                    choices=sorted(workloads.ALL))
    ap.add_argument("--coll", default="allreduce",
                    choices=["allreduce", "reducescatter", "allgather"])
    ap.add_argument("--algo", default="ring", choices=["ring", "tree"],
                    help="AllReduce algorithm: the ring, or the double binary tree "
                         "(Simple protocol, up to 16 ranks; another reduction order)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-calibration", action="store_true")
    ap.add_argument("--sweep", action="store_true",
                    help="message-size sweep and cost model (JSON line per point)")
    args = ap.parse_args()
    w = workloads.ALL[args.workload]
    if args.sweep:
        run_sweep(args)
    elif args.impl == "reference":
        run_reference(args, w)
    else:
        run_ours(args, w)


if __name__ == "__main__":
    main()
