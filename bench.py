"""Benchmark: fixed-m attention forward on the Wan2.2-DiT-shaped workload.

One step = the whole hot path on one batch of synthetic input:
    fm_bounds (norms, key mean, m, flags over all 75,600 keys)
    fm_attn_chunk (first KV chunk of 37,800 keys, the ring's first step)
    fm_attn_chunk_final (second chunk, folded and normalised into o in the same pass)
at B=1, H=40, S_q=S_k=75,600, D=128, bf16, virtual K-centering on.
TFLOP/s = 4*H*S_q*S_k*D / t (the two contractions), t from CUDA events on the launch stream.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the CPU oracle (plain fp64 C, all host cores) on a bounded sample
of the same workload.  Under torchrun (N > 1) every rank runs an independent replica
(weak scaling; the path needs no collective); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fixed-m attn fwd TFLOP/s (bf16, S=75,600, H=40, D=128) and % of BF16 tensor peak"
WORKLOAD = "wan"
L2_BYTES = 129 * 1000 * 1000  # GB300 L2
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
# DRAM bytes (read + write) per launch of the chunk kernel from one ncu capture of the Wan
# step at 8 heads (dram__bytes_read.sum + dram__bytes_write.sum), averaged over the
# first-chunk and the final-chunk launch, scaled x5 to 40 heads (every term of the traffic
# grows with the head count).
# Valid only for the kernel code it was measured on (comments aside): the bench reports null
# otherwise.
CHUNK_TRAFFIC = {"code_sha256_16": "de3b182134dfb248", "bytes_per_launch": 5 * (620.001e6 + 846.480e6) / 2}


def kernel_code_hash(path: str) -> str:
    """sha256[:16] of a CUDA source with its // comments and blank lines removed, so that a
    comment edit keeps a recorded measurement while any change to the code drops it."""
    import hashlib
    import re

    lines = []
    for ln in open(path, encoding="utf-8").read().splitlines():
        ln = re.sub(r"//.*$", "", ln).rstrip()
        if ln:
            lines.append(ln)
    return hashlib.sha256("\n".join(lines).encode()).hexdigest()[:16]


def chunk_traffic():
    src = os.path.join(ROOT, "fixed_max_softmax_gb300", "csrc", "fm_chunk_tc.cu")
    try:
        h = kernel_code_hash(src)
    except OSError:
        return None
    return CHUNK_TRAFFIC["bytes_per_launch"] if h == CHUNK_TRAFFIC["code_sha256_16"] else None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(t_ms: float, device=None) -> float:
    """The slowest rank's time (all ranks get it); the local time when not distributed."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return t_ms
    tt = torch.tensor([t_ms], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt.item())


def whole_job_tflops(world: int, flops_per_rank_step: float, steps: int, t_ms: float) -> float:
    """Units processed by all ranks (each an independent replica) over the slowest rank's time."""
    return world * flops_per_rank_step * steps / (t_ms * 1e-3) / 1e12


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                self.out = ""

    def summary(self):
        sms, maxs, watts, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                maxs.append(float(parts[2]))
            except ValueError:
                continue
            try:
                watts.append(float(parts[3]))
            except ValueError:
                pass
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "power_w": None}
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": max(maxs), "reasons": sorted(reasons),
                "samples": len(sms), "power_w": statistics.median(watts) if watts else None}


def cpu_oracle_sample(target_s: float = 12.0, max_rows: int = 24576):
    """Time the fp64 CPU oracle on 1 head x R query rows x all 75,600 keys of the workload.

    R grows until one timed call takes about target_s seconds.  Returns (TFLOP/s, dict)."""
    import oracle
    import workloads

    oracle.build()
    w = workloads.WORKLOADS[WORKLOAD]
    q, k, v = workloads.make_inputs(WORKLOAD, device="cpu", heads=[0])
    threads = oracle.num_threads()
    rows = 16
    while True:
        t0 = time.perf_counter()
        oracle.attention(q[0, :, :rows], k[0], v[0], threads=threads)
        dt = time.perf_counter() - t0
        if dt >= target_s or rows >= max_rows:
            break
        rows = min(max_rows, max(rows * 2, int(rows * target_s / max(dt, 1e-3))))
    flops = w.flops(heads=1, rows=rows)
    # the same on one core, on as many rows as that core's share of the sample
    rows1 = max(16, rows // max(threads, 1))
    t0 = time.perf_counter()
    oracle.attention(q[0, :, :rows1], k[0], v[0], threads=1)
    dt1 = time.perf_counter() - t0
    one_core = w.flops(heads=1, rows=rows1) / dt1 / 1e12
    return flops / dt / 1e12, {"rows": rows, "seconds": dt, "threads": threads, "one_core": one_core,
                               "rows_one_core": rows1, "seconds_one_core": dt1}


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle as it stands, timed on a bounded sample per step."""
    if rank != 0:
        return
    import oracle
    import workloads

    oracle.build()
    w = workloads.WORKLOADS[WORKLOAD]
    q, k, v = workloads.make_inputs(WORKLOAD, device="cpu", heads=[0])
    threads = oracle.num_threads()
    rows = args.ref_rows
    for _ in range(args.warmup):
        oracle.attention(q[0, :, :rows], k[0], v[0], threads=threads)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.attention(q[0, :, :rows], k[0], v[0], threads=threads)
        times.append(time.perf_counter() - t0)
    t = sum(times)
    flops = w.flops(heads=1, rows=rows) * args.steps
    value = flops / t / 1e12
    sample = f"1 head x {rows} query rows x all {w.N} keys per step (fp64 oracle, {threads} threads)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * t / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: B={w.B} H={w.H} S={w.Sq} D={w.D} bf16 inputs, sampled rows",
                   "sample": sample},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, rank, world, local_rank):
    import torch

    import fixed_max_softmax_gb300 as fm
    import workloads

    fm.load()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS[args.workload]
    chunks = workloads.chunk_bounds(w)
    H = w.H if args.heads is None else args.heads
    centering = w.centering[0] if args.centering == "auto" else args.centering == "on"
    q, k, v = workloads.make_inputs(w.name, device=dev, heads=range(H))
    fa = fm.FixedMAttention(w.B, H, w.Sq, w.N, w.D, dev, centering=centering, force_online=args.force_online,
                            out_dtype=q.dtype, sink_keys=args.sink_keys, schedule=args.schedule)
    stream = torch.cuda.current_stream(dev)
    step_flops = w.flops(heads=w.B * H)
    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()

    def step(ev=None, bev=None):
        if bev is not None:
            bev.append(torch.cuda.Event(enable_timing=True))
            bev[-1].record(stream)
        fm.fm_bounds(q, k, v, fa.opt, fa.bounds, fa.workspace, stream)
        if bev is not None:
            bev.append(torch.cuda.Event(enable_timing=True))
            bev[-1].record(stream)
        for i, (s, n) in enumerate(chunks):
            if ev is not None:
                ev.append(torch.cuda.Event(enable_timing=True))
                ev[-1].record(stream)
            if i == len(chunks) - 1:  # last chunk: fold and normalise in one pass
                fm.fm_attn_chunk_final(q, k[:, :, s:s + n], v[:, :, s:s + n], fa.bounds, fa.opt, fa.acc_o,
                                       fa.acc_sum, fa.acc_max, i > 0, fa.out, None, stream)
            else:
                fm.fm_attn_chunk(q, k[:, :, s:s + n], v[:, :, s:s + n], fa.bounds, fa.opt, fa.acc_o, fa.acc_sum,
                                 fa.acc_max, i > 0, stream)
            if ev is not None:
                ev.append(torch.cuda.Event(enable_timing=True))
                ev[-1].record(stream)

    # bounds: key sums with the key mean (centering only), norms, finish (with the row shifts);
    # one launch per chunk with the normalise fused into the last; with key sinks the bounds add
    # their selection and the step ends with one pass that folds the sinks back and normalises
    launches_per_step = (3 if centering else 2) + len(chunks) + (2 if args.sink_keys else 0)
    for _ in range(args.warmup):
        step()
    fm.fm_sync_status(stream)
    flags = fa.bounds.flag
    eligible = float(flags.float().mean().item())

    # ---- timed region: inputs resident in HBM.  Where one input tensor is larger than L2 the
    # steps run back to back; otherwise each step is timed on its own, after a write of a
    # buffer twice the size of L2 that leaves none of the step's data in it.  Inside a step
    # nothing but the path's own launches is enqueued: an event recorded between two launches
    # stops the second from starting while the first finishes (programmatic dependent launch),
    # which cost the 4,096-key steps 2-4 %.  The per-kernel durations (roofline, bounds pass)
    # come from as many steps again, run right after with an event around each launch.
    tensor_bytes = q.numel() * q.element_size()
    flush = None
    if tensor_bytes <= L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    chunk_events = []
    bounds_events = []
    step_events = []
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clk:
        start.record(stream)
        for _ in range(args.steps):
            if flush is not None:
                flush.fill_(1)
                step_events.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                step_events[-1][0].record(stream)
            step()
            if flush is not None:
                step_events[-1][1].record(stream)
        end.record(stream)
        torch.cuda.synchronize(dev)
        # the same steps with an event around each launch: the kernels' own durations
        for _ in range(args.steps):
            if flush is not None:
                flush.fill_(1)
            step(chunk_events, bounds_events)
        torch.cuda.synchronize(dev)
    barrier()
    fm.fm_sync_status(stream)
    t_ms = start.elapsed_time(end) if flush is None else sum(a.elapsed_time(b) for a, b in step_events)
    chunk_ms = [chunk_events[i].elapsed_time(chunk_events[i + 1]) for i in range(0, len(chunk_events), 2)]
    bounds_ms = statistics.mean(bounds_events[i].elapsed_time(bounds_events[i + 1])
                                for i in range(0, len(bounds_events), 2))
    # the bounds pass again without centering (no key sums; the same norms and finish): with it,
    # the two kernels' shares of the pass, each against its own bytes
    bounds_off_ms = None
    if centering and not args.sink_keys:
        off = fm.opts(fa.opt.softmax_scale, False, bool(fa.opt.force_online), bool(fa.opt.per_row), 0,
                      int(fa.opt.schedule))
        off_events = []
        for _ in range(args.steps):
            if flush is not None:
                flush.fill_(1)
            off_events.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
            off_events[-1][0].record(stream)
            fm.fm_bounds(q, k, v, off, fa.bounds, fa.workspace, stream)
            off_events[-1][1].record(stream)
        torch.cuda.synchronize(dev)
        fm.fm_sync_status(stream)
        bounds_off_ms = statistics.mean(a.elapsed_time(b) for a, b in off_events)
    t_ms = max_over_ranks(t_ms, dev)
    ms_per_step = t_ms / args.steps
    value = whole_job_tflops(world, step_flops, args.steps, t_ms)

    # ---- the same step with every chunk folded in one launch (fm_attn_chunks): O and the
    # row sums stay on chip across the chunk boundary, as the pages' accumulator stays
    # resident for the whole ring
    def step_one_launch():
        fm.fm_bounds(q, k, v, fa.opt, fa.bounds, fa.workspace, stream)
        fm.fm_attn_chunks(q, [k[:, :, s:s + n] for s, n in chunks], [v[:, :, s:s + n] for s, n in chunks],
                          fa.bounds, fa.opt, fa.acc_o, fa.acc_sum, fa.acc_max, False, fa.out, None, stream)

    for _ in range(2):
        step_one_launch()
    fm.fm_sync_status(stream)
    o0, o1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    one_events = []
    barrier()
    o0.record(stream)
    for _ in range(args.steps):
        if flush is not None:
            flush.fill_(1)
            one_events.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
            one_events[-1][0].record(stream)
        step_one_launch()
        if flush is not None:
            one_events[-1][1].record(stream)
    o1.record(stream)
    torch.cuda.synchronize(dev)
    fm.fm_sync_status(stream)
    t_one = o0.elapsed_time(o1) if flush is None else sum(a.elapsed_time(b) for a, b in one_events)
    t_one = max_over_ranks(t_one, dev)
    one_launch = {"value": whole_job_tflops(world, step_flops, args.steps, t_one), "unit": "TFLOP/s",
                  "ms_per_step": t_one / args.steps,
                  "how": "fm_bounds + fm_attn_chunks (all chunks and the normalise in one launch)"}

    # ---- end to end through the C ABI with host buffers (pinned), copies timed: every step
    # uploads its Q/K/V from pinned host memory and reads its output back; fm_attention_host
    # overlaps step i+1's upload and step i-1's read-back with step i's kernels
    e2e = None
    if args.e2e_steps > 0:
        qh = q.cpu().pin_memory()
        kh = k.cpu().pin_memory()
        vh = v.cpu().pin_memory()
        outs = [torch.empty(fa.out.shape, dtype=fa.out.dtype).pin_memory() for _ in range(2)]
        hp = fm.HostPipeline(fa, q.dtype, dev)
        hp.run([(qh, kh, vh, outs[0])], chunks)  # warm-up
        fm.fm_sync_status(stream)
        barrier()
        torch.cuda.synchronize(dev)
        with ClockSampler(local_rank) as clk_e2e:
            t0 = time.perf_counter()
            hp.run([(qh, kh, vh, outs[i % 2]) for i in range(args.e2e_steps)], chunks)
            torch.cuda.synchronize(dev)
            te = max_over_ranks((time.perf_counter() - t0) * 1e3, dev)
        ce = clk_e2e.summary()
        fm.fm_sync_status(stream)
        # the machine's host link, for reading the figure: one 774 MB pinned copy each way, timed alone
        link = {}
        for name, (dst, src) in {"h2d_gbs": (q, qh), "d2h_gbs": (outs[0], fa.out)}.items():
            dst.copy_(src, non_blocking=True)  # warm-up: the first copy from a buffer pays setup
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            dst.copy_(src, non_blocking=True)
            b.record(stream)
            torch.cuda.synchronize(dev)
            link[name] = src.numel() * src.element_size() / (a.elapsed_time(b) * 1e-3) / 1e9
        # the same upload (Q, K and V of one step) on a second stream beside one step's kernels:
        # does the link keep its rate under load, and does the step keep its time?
        side = torch.cuda.Stream(dev)
        up_dst = [torch.empty_like(t) for t in (q, k, v)]
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c, d = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c.record(side)
        a.record(stream)
        with torch.cuda.stream(side):
            for dst, src in zip(up_dst, (qh, kh, vh)):
                dst.copy_(src, non_blocking=True)
        step()
        b.record(stream)
        d.record(side)
        torch.cuda.synchronize(dev)
        fm.fm_sync_status(stream)
        link["h2d_gbs_beside_step"] = 3 * tensor_bytes / (c.elapsed_time(d) * 1e-3) / 1e9
        link["step_ms_beside_upload"] = a.elapsed_time(b)
        del up_dst
        e2e = {"value": whole_job_tflops(world, step_flops, args.e2e_steps, te), "unit": "TFLOP/s",
               "host_link": {k2: round(v2, 2 if k2.startswith("step") else 1) for k2, v2 in link.items()},
               "clocks": {k2: ce[k2] for k2 in ("sm_mhz", "power_w", "reasons", "samples")},
               "h2d_bytes_per_step": int(3 * q.numel() * q.element_size()),
               "d2h_bytes_per_step": int(fa.out.numel() * fa.out.element_size()),
               "ms_per_step": te / args.e2e_steps, "steps": args.e2e_steps,
               "timing": "host wall clock between device synchronisations",
               "overlap": "upload of step i+1 and read-back of step i-1 run during step i",
               "how": "fm_attention_host (C ABI, host buffers in page-locked memory, three streams)"}

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    chunk_flops = [w.flops(heads=w.B * H, keys=n) for _, n in chunks]
    # algorithmic bytes of a chunk launch: Q, this chunk's K and V, the accumulators written
    # (and read back on every chunk after the first), averaged over the step's launches
    rows = w.B * H * w.Sq
    algo = []
    for i, (_, n) in enumerate(chunks):
        io = q.element_size() * (rows * w.D + 2 * w.B * H * n * w.D)
        acc = 4 * rows * (w.D + 2)
        if i == len(chunks) - 1 and i > 0:  # fused normalise: acc read, o (bf16) written, acc_o not
            algo.append(io + acc + 4 * rows * 2 + fa.out.element_size() * rows * w.D)
        else:
            algo.append(io + acc * (2 if i > 0 else 1))
    algo_bytes = statistics.mean(algo)
    per_launch_flops = statistics.mean(chunk_flops)
    chunk_avg_ms = statistics.mean(chunk_ms)
    achieved = per_launch_flops / (chunk_avg_ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops_sustained"]
    # the schedule the library resolves AUTO to, per chunk launch (the rule of fm_api.cu: the
    # persistent kernel for a call of at most 8 key tiles with at least twice the SMs in items)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    items = w.B * H * math.ceil(math.ceil(w.Sq / 128) / 2)
    persistent = args.schedule == "persistent" or (
        args.schedule == "auto" and all(math.ceil(n / 128) <= 8 for _, n in chunks) and items >= 2 * sms)
    kernel_name = "fm_chunk_tc_persistent_kernel" if persistent else "fm_chunk_tc_kernel"
    traffic = args.traffic if args.traffic is not None else (
        chunk_traffic() if (H == w.H and w.name == WORKLOAD and not args.force_online and not persistent) else None)
    roofline = {"bound": "tensor", "kernel": kernel_name, "achieved": achieved, "peak": peak,
                "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                "traffic_unit": "bytes per launch (dram read + write)",
                "algorithmic_bytes_per_launch": algo_bytes,
                "peak_kind": f"bf16 sustained ({peak_src})",
                "frac_of_burst_peak": achieved / peaks["bf16_tflops"], "launch_ms": chunk_avg_ms,
                "how": "CUDA events around each chunk launch, in as many steps again right after the timed region"}
    # the bounds pass: Q, K and V read once, K once more for the key mean when centering
    bounds_bytes = q.element_size() * w.B * H * w.D * (w.Sq + (3 if centering else 2) * w.N)
    bounds_line = {"ms": bounds_ms, "algorithmic_bytes": bounds_bytes, "achieved": bounds_bytes / (bounds_ms * 1e-3) / 1e9,
                   "unit": "GB/s", "peak": peaks["hbm_gbs"],
                   "frac": bounds_bytes / (bounds_ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
                   "kernels": "key sums with the key mean (centering), norms, finish with the row shifts",
                   "how": "CUDA events around fm_bounds, in as many steps again right after the timed region"}
    if bounds_off_ms is not None:
        kb = k.element_size() * w.B * H * w.N * w.D  # the key sums read K once
        nb = bounds_bytes - kb                          # the norms read Q, K and V once
        ks_ms = bounds_ms - bounds_off_ms
        bounds_line["per_kernel"] = {
            "key_sums": {"ms": ks_ms, "bytes": kb, "achieved": kb / (ks_ms * 1e-3) / 1e9 if ks_ms > 0 else None},
            "norms_and_finish": {"ms": bounds_off_ms, "bytes": nb, "achieved": nb / (bounds_off_ms * 1e-3) / 1e9},
            "unit": "GB/s",
            "how": "the pass timed again without centering (norms and finish only, the same bytes): the key sums "
                   "are the difference"}
    cpu = None
    if world == 1 and not args.no_cpu_baseline and w.name == WORKLOAD:
        cv, info = cpu_oracle_sample(args.cpu_seconds)
        cpu = {"value": cv, "unit": "TFLOP/s", "cores": info["threads"], "kind": "oracle",
               "sample": f"1 head x {info['rows']} query rows x all {w.N} keys, fp64, "
                         f"{info['seconds']:.1f} s",
               "value_one_core": info["one_core"],
               "sample_one_core": f"1 head x {info['rows_one_core']} query rows x all {w.N} keys, "
                                  f"{info['seconds_one_core']:.1f} s"}
    clocks = clk.summary()
    line = {
        "metric": METRIC if w.name == WORKLOAD else f"fixed-m attn fwd TFLOP/s ({w.name})",
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": f"{w.name}: B={w.B} H={H} S_q=S_k={w.Sq} D={w.D} {w.dtype}, "
                               f"{len(chunks)} KV chunks of {chunks[0][1]}, "
                               f"virtual K-centering {'on' if centering else 'off'}"
                               + (", every tile forced onto the online fallback" if args.force_online else "")
                               + (f", {args.sink_keys} key sinks per head" if args.sink_keys else ""),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": (f"inputs larger than L2 ({tensor_bytes / 1e6:.0f} MB per tensor), no flush" if flush is None
                          else f"{tensor_bytes / 1e6:.0f} MB per tensor fits in L2: a {2 * L2_BYTES / 1e6:.0f} MB "
                               "buffer is written before each step, outside its timing"),
                   "schedule": args.schedule + (f" ({'persistent' if persistent else 'grid'})" if args.schedule == "auto" else ""),
                   "fixed_m_tile_fraction": eligible},
        "pct_of_peak": 100.0 * value / peak,
        "roofline": roofline,
        "bounds_pass": bounds_line,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "one_launch": one_launch,
        "clocks": {k2: clocks[k2] for k2 in ("sm_mhz", "sm_max_mhz", "reasons", "power_w")},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-rows", type=int, default=256, help="query rows per reference step")
    ap.add_argument("--heads", type=int, default=None, help="first N heads only (profiling a smaller case)")
    ap.add_argument("--workload", default=WORKLOAD, help="wan (default, the headline), h40_s4096, mix, adversarial, sinks")
    ap.add_argument("--centering", choices=["auto", "on", "off"], default="auto")
    ap.add_argument("--force-online", action="store_true", help="run every tile on the online fallback")
    ap.add_argument("--sink-keys", type=int, default=0, help="leave this many loudest keys per head out of the key max")
    ap.add_argument("--schedule", choices=["auto", "grid", "persistent"], default="auto",
                    help="work schedule of the tensor-core chunk kernel (fm_opts.schedule)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per chunk launch from an ncu capture of the current kernel")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank, world, local_rank = dist_env()
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        dist.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_ours(args, rank, world, local_rank)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
