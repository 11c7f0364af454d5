#!/usr/bin/env python3
"""Throughput of global L2-norm gradient clipping on one GB300.

One step = one clip (norm, decision and scaling) of a whole ANDREA-120M-shaped
fp32 gradient set (124 tensors, 92,248,320 elements, one matrix spiked x50 so
that the clip fires), through the library's C ABI, inputs resident in HBM.

The metric is algorithmic bytes moved per second: 4 B per element read for the
norm, 4 B read + 4 B written for the scaling pass, 12 B/elem = 1.107 GB per
step.  Printed as one JSON line.

Timing: a pool of P distinct copies of the gradient set; each timed run clips
P of them back to back between two CUDA events on the launching stream.  The
sets are larger than L2 (369 MB vs 126 MB) and L2 is flushed before each run.
Between runs, outside the events, every set is restored from a pristine copy
(a clip changes its input in place, and a clipped set no longer clips).

--impl reference times the oracle (the plain C fp64 implementation used by the
tests) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "global-norm clip GB/s and % of HBM roofline, ANDREA-120M fp32 grads"
NOMINAL_HBM_GBS = 7900.0


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=3200)
    p.add_argument("--warmup", type=int, default=64)
    p.add_argument("--impl", choices=["gclip", "reference"], default="gclip")
    p.add_argument("--variant", choices=["split", "persistent", "split_tma", "persistent_tma", "split_wave",
                                         "three_kernel"],
                   default="split")
    p.add_argument("--workload", default="andrea120m",
                   help="tiny, andrea14m, andrea120m (default), andrea120m_noclip, andrea120m_fp16, "
                        "andrea120m_fp16_inf, andrea120m_bf16, andrea1p2b")
    p.add_argument("--pool", type=int, default=32,
                   help="distinct gradient sets per timed run (at most steps / 4, so that "
                        "every run gives at least four timed runs)")
    p.add_argument("--l2-keep-mb", type=float, default=None,
                   help="MB of the norm pass kept in L2 for the scaling pass "
                        "(default: the library's choice)")
    p.add_argument("--warm", action="store_true",
                   help="one set, no L2 flush (only for workloads that write nothing)")
    p.add_argument("--graph", action="store_true",
                   help="replay each run of clips as one captured CUDA graph")
    p.add_argument("--per-tensor", action="store_true",
                   help="clip each tensor by its own norm (clip_grad_norm_per_tensor)")
    p.add_argument("--accumulate", action="store_true",
                   help="add the last microbatch's gradients, then clip (clip_grad_norm_accumulate)")
    p.add_argument("--to-f32", action="store_true",
                   help="clip out of place into fp32 buffers (clip_grad_norm_to_f32)")
    p.add_argument("--adamw", action="store_true",
                   help="time the fused clip + AdamW step instead of the clip alone")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-all-cores", action="store_true",
                   help="skip the all-cores replica timing of the oracle")
    p.add_argument("--cpu-seconds", type=float, default=10.0,
                   help="budget of the CPU-baseline leg on rank 0")
    return p.parse_args(argv)


# ---------------------------------------------------------------------------
# helpers shared by both arms (host logic; covered by the CPU tests)

def algorithmic_bytes(numel: int, elem_bytes: int, decision: str) -> int:
    """Bytes a clip must move: one read for the norm; a read and a write more
    when elements are rewritten (clip, or an unscale that is not 1)."""
    if decision == "write":
        return 3 * numel * elem_bytes
    return numel * elem_bytes


def pool_size(pool: int, steps: int) -> int:
    """Distinct sets per timed run: at most steps / 4, so that a short run
    still gives four or more timed runs (and a real p10 / p50 / p90)."""
    return max(1, min(pool, steps // 4))


def rank_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def make_reduce_max(world: int, device):
    """The max of a float over the ranks of the default process group (a
    tensor on `device`: the GPU under NCCL, the CPU under gloo)."""
    def reduce_max(x: float) -> float:
        if world == 1:
            return x
        import torch
        import torch.distributed as dist
        t = torch.tensor([x], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return reduce_max


def aggregate(elapsed_ms: float, units: float, world: int, reduce_max=None):
    """Whole-job throughput: units processed by all ranks over the slowest
    rank's time.  reduce_max maps a local float to its max over ranks."""
    t = reduce_max(elapsed_ms) if reduce_max else elapsed_ms
    return units * world / (t / 1e3), t


def strip_comments(text: str) -> str:
    """C/C++ source without its comments and with whitespace collapsed, so
    that a change of wording alone leaves the digest of the code unchanged.
    String and character literals are kept as they are."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        elif c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_digest(read=None) -> str:
    """Digest of the library's code: every file under csrc/ and the C ABI
    header (whose constants the kernels are compiled with), comments and
    whitespace left out.  `read(relative_path)` may supply the files' text
    (for another revision); by default they are read from this tree."""
    if read is None:
        def read(rel):
            with open(os.path.join(ROOT, rel), encoding="utf-8") as fh:
                return fh.read()
    h = hashlib.sha256()
    d = os.path.join("global_l2_norm_gb300", "csrc")
    files = [os.path.join(d, f) for f in sorted(os.listdir(os.path.join(ROOT, d)))]
    files.append(os.path.join("include", "gclip.h"))
    for rel in files:
        h.update(os.path.basename(rel).encode() + b"\0" + strip_comments(read(rel)).encode())
    return h.hexdigest()[:16]


def traffic_from_profile(kernel: str, variant: str = "", workload: str = "andrea120m"):
    """DRAM bytes per launch from the committed ncu summary, if that summary
    was taken on the current kernel source and on this workload (an entry
    that names none was taken on andrea120m); else None.  An entry
    "<kernel>@<variant>" (the kernel as that variant runs it) wins over the
    plain kernel name."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    e = d.get(f"{kernel}@{variant}") or d.get(kernel)
    if not e or e.get("source_digest") != source_digest():
        return None
    if e.get("workload", "andrea120m") != workload:
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.index), "-lms", "200"], stdout=self.file,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        return summarize_clocks(self.file.read())


def summarize_clocks(text: str) -> dict:
    sm, smax, reasons, n = [], [], set(), 0
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in text.strip().splitlines():
        parts = [x.strip() for x in line.split(",")]
        if len(parts) < 9:
            continue
        try:
            sm.append(float(parts[1]))
            smax.append(float(parts[2]))
        except ValueError:
            continue
        n += 1
        for name, v in zip(names, parts[5:9]):
            if v.lower() == "active":
                reasons.add(name)
    if not sm:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
            "reasons": sorted(reasons), "samples": n}


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores

def oracle_inputs(gs):
    import numpy as np
    from oracle import OracleTensor
    out = []
    for t in gs.tensors:
        c = t.detach().contiguous().cpu().reshape(-1)
        if gs.workload.dtype == "f32":
            out.append(OracleTensor(c.numpy().copy(), "f32"))
        elif gs.workload.dtype == "f16":
            out.append(OracleTensor(c.numpy().copy(), "f16"))
        else:
            import torch
            out.append(OracleTensor(c.view(torch.int16).numpy().view(np.uint16).copy(), "bf16"))
    return out


def reference_sample(gs, target_elems: int):
    """A run of whole tensors starting at the (first) spiked matrix, about
    target_elems elements long, so that the sample's own clip fires too."""
    names = [s.name for s in gs.workload.layout]
    start = names.index(gs.spiked[0]) if gs.spiked else 0
    idx, n = [], 0
    i = start
    while n < target_elems and len(idx) < len(names):
        idx.append(i)
        n += gs.tensors[i].numel()
        i = (i + 1) % len(names)
    return idx, n


def time_oracle(host, w, reps_budget_s: float):
    import oracle
    t0 = time.perf_counter()
    reps = 0
    while True:
        _, r = oracle.clip(host, w.max_norm, w.inv_scale)
        reps += 1
        if time.perf_counter() - t0 >= reps_budget_s:
            break
    return (time.perf_counter() - t0) / reps, reps, r


def _oracle_replica(workload: str, target: int, seconds: float, barrier, results) -> None:
    """One host core's replica of the oracle (a spawned process): its own
    seeded sample of the workload, clipped back to back for `seconds` once
    every replica is ready."""
    try:
        import torch
        torch.set_num_threads(1)
        import oracle
        from workloads import WORKLOADS, make_gradset
        w = WORKLOADS[workload]
        gs = make_gradset(w, device="cpu")
        idx, n = reference_sample(gs, target)
        host = oracle_inputs(type(gs)(w, [gs.tensors[i] for i in idx], gs.spiked))
        del gs
        oracle.clip(host, w.max_norm, w.inv_scale)      # load and touch everything once
    except Exception as exc:   # reported by the parent; the barrier must still be met
        barrier.wait()
        results.put(("error", repr(exc)))
        return
    barrier.wait()
    t0 = time.perf_counter()
    reps = 0
    while True:
        _, r = oracle.clip(host, w.max_norm, w.inv_scale)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    results.put((time.perf_counter() - t0, reps, n, r.decision_name))


def oracle_all_cores(w, seconds: float, target: int = 8 << 20):
    """Throughput of the unmodified oracle on every host core at once: one
    spawned process per core, each clipping its own copy of a sample of
    whole tensors (about `target` elements, starting at the spiked matrix);
    value = the bytes all replicas moved / the longest replica's time."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(cores)
    results = ctx.Queue()
    procs = [ctx.Process(target=_oracle_replica, args=(w.name, target, seconds, barrier, results))
             for _ in range(cores)]
    for p_ in procs:
        p_.start()
    out = [results.get(timeout=600) for _ in procs]
    for p_ in procs:
        p_.join(timeout=60)
    errors = [o[1] for o in out if o[0] == "error"]
    if errors:
        return {"error": errors[0], "cores": cores}
    longest = max(o[0] for o in out)
    nbytes = sum(algorithmic_bytes(o[2], w.elem_bytes, "write" if o[3] != "skip" else "read") * o[1]
                 for o in out)
    n = out[0][2]
    return {"value": round(nbytes / longest / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{cores} single-threaded replicas of the C fp64 oracle, one per host "
                      f"core, each clipping its own {n}-element sample of the {w.name} set "
                      f"(whole tensors from the spiked matrix) back to back for {seconds:.0f} s"}


def run_reference(args):
    rank, world, _ = rank_env()
    if rank != 0:
        return 0
    import oracle
    import torch
    from workloads import WORKLOADS, make_gradset
    oracle.build()
    w = WORKLOADS[args.workload]
    gs = make_gradset(w, device="cpu")
    # size each step so that warmup + steps take about a minute on one core
    calib_idx, calib_n = reference_sample(gs, 1 << 20)
    sub = oracle_inputs(type(gs)(w, [gs.tensors[i] for i in calib_idx]))
    t0 = time.perf_counter()
    oracle.clip(sub, w.max_norm, w.inv_scale)
    rate = calib_n / max(time.perf_counter() - t0, 1e-6)
    per_step = max(1 << 16, int(rate * 60.0 / max(1, args.steps + args.warmup)))
    per_step = min(per_step, w.numel)
    idx, n = reference_sample(gs, per_step)
    sub_gs = type(gs)(w, [gs.tensors[i] for i in idx], gs.spiked)
    host = oracle_inputs(sub_gs)
    for _ in range(args.warmup):
        oracle.clip(host, w.max_norm, w.inv_scale)
    times = []
    decision = None
    for _ in range(args.steps):
        t0 = time.perf_counter()
        _, r = oracle.clip(host, w.max_norm, w.inv_scale)
        times.append(time.perf_counter() - t0)
        decision = r.decision_name
    writes = decision != "skip"
    nbytes = algorithmic_bytes(n, w.elem_bytes, "write" if writes else "read")
    total = sum(times)
    value = nbytes * len(times) / total / 1e9
    sample = (f"{len(idx)} whole tensors of the {w.name} set starting at the spiked "
              f"matrix, {n} elements per step (decision {decision})")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / len(times) * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "description": w.description,
                   "elements_per_step": n, "bytes_per_step": nbytes},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the library arm

def run_gclip(args):
    import torch
    import torch.distributed as dist

    import global_l2_norm_gb300 as g
    from workloads import WORKLOADS, make_gradset

    rank, world, local = rank_env()
    if world != args.gpus:
        print(json.dumps({"error": f"--gpus {args.gpus} but WORLD_SIZE={world}"}))
        return 2
    if args.per_tensor + args.to_f32 + args.accumulate > 1:
        print(json.dumps({"error": "--per-tensor, --to-f32 and --accumulate exclude one another"}))
        return 2
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    g.build()
    w = WORKLOADS[args.workload]
    stream = torch.cuda.current_stream(dev)

    # one pristine set, P working sets
    pristine = make_gradset(w, device=dev, flat=True)
    P = 1 if args.warm else pool_size(args.pool, args.steps)
    sets = [make_gradset(w, device=dev, flat=True) for _ in range(P)]
    clippers = [g.GradClipper(s.tensors, variant=args.variant) for s in sets]
    if args.to_f32:
        for c, s_ in zip(clippers, sets):
            c.attach_f32_out([torch.empty(t.numel(), device=dev) for t in s_.tensors])
    addends = []
    if args.accumulate:   # the last microbatch's gradients: another seeded set per pool entry
        addends = [make_gradset(w, seed=4321, device=dev, flat=True) for _ in range(P)]
        for c, a_ in zip(clippers, addends):
            c.attach_addend(a_.tensors)
    if args.l2_keep_mb is not None:
        for c in clippers:
            c.set_l2_keep(int(args.l2_keep_mb * (1 << 20)))
    props = torch.cuda.get_device_properties(dev)
    l2 = props.L2_cache_size
    device_info = {"name": props.name, "sms": props.multi_processor_count, "l2_bytes": l2,
                   "hbm_bytes": props.total_memory}
    flush = torch.empty(2 * l2 + (1 << 20), dtype=torch.uint8, device=dev)

    writes = True

    def clip(c):
        if args.per_tensor:
            c.clip_per_tensor_(w.max_norm, w.inv_scale)
        elif args.to_f32:
            c.clip_to_f32_(w.max_norm, w.inv_scale)
        elif args.accumulate:
            c.clip_accumulate_(w.max_norm, w.inv_scale)
        else:
            c.clip_(w.max_norm, w.inv_scale)

    def restore():
        # a clip that wrote changed its input: put the pristine values back
        if writes:
            for s in sets:
                s.flat.copy_(pristine.flat)
        if not args.warm:
            flush.fill_(1)

    # correctness of the step being timed: the decision and a norm that agrees
    # with a float64 torch norm of the same data (a sanity check, not parity)
    restore()
    clip(clippers[0])
    if args.per_tensor:
        recs = clippers[0].per_tensor_results()
        wr = [r["decision"] != g.GCLIP_DECISION_SKIP and not (
            r["coef_hi"] == 1.0 and r["coef_lo"] == 0.0) for r in recs]
        writes = any(wr)
        written = sum(s_.numel for s_, x in zip(w.layout, wr) if x)
        rec = {"decision": g.GCLIP_DECISION_CLIP if writes else g.GCLIP_DECISION_PASS}
    else:
        rec = clippers[0].result()
        ref_sets = pristine.tensors
        if args.accumulate:   # the sums, each rounded by torch's own addition in the format
            ref_sets = [a + b for a, b in zip(pristine.tensors, addends[0].tensors)]
        ref_norm = math.sqrt(sum(float(t.double().square().sum()) for t in ref_sets)
                             ) * w.inv_scale
        del ref_sets
        if math.isfinite(ref_norm):
            assert abs(rec["norm"] - ref_norm) <= 1e-5 * ref_norm, (rec["norm"], ref_norm)
        else:
            assert rec["nonfinite"] == 1, rec
        writes = rec["decision"] != g.GCLIP_DECISION_SKIP and not (
            rec["coef_hi"] == 1.0 and rec["coef_lo"] == 0.0)
        written = w.numel if writes else 0
        if args.to_f32:   # the gradients are only read; the outputs are always written
            writes = False
            written = w.numel if rec["decision"] != g.GCLIP_DECISION_SKIP else 0
        scaled = written
        if args.accumulate:   # the norm pass always writes the sums
            writes = True
    if args.warm and writes:
        print(json.dumps({"error": "--warm needs a workload whose clip writes nothing"}))
        return 2
    decision_name = {0: "pass", 1: "clip", 2: "skip"}[rec["decision"]]
    nbytes = (w.numel * w.elem_bytes + written * (w.elem_bytes + 4) if args.to_f32
              else w.numel * w.elem_bytes + 2 * written * w.elem_bytes)
    if args.accumulate:   # read x and a, write x + a; then the scaling pass if it writes
        nbytes = 3 * w.numel * w.elem_bytes + 2 * scaled * w.elem_bytes

    # warm-up
    restore()
    for i in range(args.warmup):
        if i and i % P == 0:
            restore()
        clip(clippers[i % P])
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    runs = []
    done = 0
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    graphs = {}

    # clips per timed run: one per set of the pool; warm runs re-clip one set
    run_len = args.pool if args.warm else P

    def run_clips(n):
        if not args.graph:
            for i in range(n):
                clip(clippers[i % P])
            return
        if n not in graphs:
            gr = torch.cuda.CUDAGraph()
            with torch.cuda.graph(gr):
                for i in range(n):
                    clip(clippers[i % P])
            graphs[n] = gr
            restore()
            torch.cuda.synchronize()
        graphs[n].replay()

    while done < args.steps:
        n = min(run_len, args.steps - done)
        restore()
        if args.graph and n not in graphs:
            run_clips(n)          # capture (untimed), then restore again
            restore()
        e0.record(stream)
        run_clips(n)
        e1.record(stream)
        e1.synchronize()
        runs.append((e0.elapsed_time(e1), n))
        done += n
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()

    local_ms = sum(t for t, _ in runs)

    reduce_max = make_reduce_max(world, dev)

    value_bps, total_ms = aggregate(local_ms, nbytes * args.steps, world, reduce_max)
    per_step_ms = total_ms / args.steps
    step_us = sorted(t / n * 1e3 for t, n in runs)

    # per-kernel durations for the roofline (events between the launches)
    launches_per_step = 3 if args.per_tensor or (
        args.variant == "three_kernel" and not (args.to_f32 or args.accumulate)) else (
        2 if args.to_f32 or args.accumulate or not args.variant.startswith("persistent") else 1)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in evs:           # torch creates the CUDA event on its first record
        e.record(stream)
    import ctypes
    ev_handles = (ctypes.c_void_p * 4)(*[e.cuda_event for e in evs])
    L = g.load()
    restore()
    seg = [[], [], []]
    for i in range(min(P, 16)):
        g.check("clip_grad_norm_profiled", L.clip_grad_norm_profiled(
            clippers[i]._h, w.max_norm, w.inv_scale, clippers[i].norm.data_ptr(),
            clippers[i].flag.data_ptr(), stream.cuda_stream, ev_handles))
        evs[3].synchronize()
        for k in range(3):
            seg[k].append(evs[k].elapsed_time(evs[k + 1]))
    seg_ms = [statistics.mean(s) for s in seg]
    if args.per_tensor or args.to_f32 or args.accumulate:
        kernel = ("per-tensor clip (3 launches)" if args.per_tensor else
                  "clip into fp32 (2 launches)" if args.to_f32 else
                  "accumulate + clip (2 launches)")
        k_bytes, k_ms = nbytes, per_step_ms
    elif args.variant.startswith("persistent"):
        kernel = "k_clip_persistent_tma" if args.variant.endswith("tma") else "k_clip_persistent"
        k_bytes, k_ms = nbytes, seg_ms[2]
        # the timed region is back-to-back launches of this one kernel
        k_ms = per_step_ms
    elif args.variant == "three_kernel":
        shares = {"k_chunk_sums": (seg_ms[0], w.numel * w.elem_bytes),
                  "k_grad_scale": (seg_ms[2], nbytes - w.numel * w.elem_bytes)}
        kernel = max(shares, key=lambda k: shares[k][0])
        k_ms, k_bytes = shares[kernel]
    else:
        tma = args.variant.endswith("tma")
        # split: one early-loading block per chunk after a clip that wrote,
        # the claiming wave after one that did not (the library's choice)
        scale = ("k_scale_tma" if tma else
                 "k_grad_scale_wave" if args.variant == "split_wave" or not writes else
                 "k_grad_scale_early")
        shares = {("k_norm_tma" if tma else "k_grad_norm_partial"): (seg_ms[0], w.numel * w.elem_bytes),
                  scale: (seg_ms[2], nbytes - w.numel * w.elem_bytes)}
        kernel = max(shares, key=lambda k: shares[k][0])
        k_ms, k_bytes = shares[kernel]
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    peak = peaks.get("hbm_gbs") or 6800.0
    peak_src = "measured" if peaks.get("hbm_gbs") else "fallback"
    achieved = k_bytes / (k_ms / 1e3) / 1e9 if k_ms > 0 else 0.0
    traffic = traffic_from_profile(kernel, args.variant, args.workload)
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic, "kernel": kernel,
                "peak_source": f"{peak_src} copy bandwidth (MEASURED_PEAKS.json hbm_gbs)"
                if peak_src == "measured" else "fallback 6.8 TB/s",
                "algorithmic_bytes_per_launch": k_bytes,
                "launch_ms": round(k_ms, 5)}
    if traffic:
        # The DRAM-level rate of the same launch: the measured DRAM bytes over
        # the same time.  Algorithmic bytes above DRAM bytes (L2 reuse) are what
        # lets `frac` exceed 1.
        roofline["dram_achieved"] = round(traffic / (k_ms / 1e3) / 1e9, 1)
        roofline["dram_frac"] = round(traffic / (k_ms / 1e3) / 1e9 / peak, 4)
    # The split variants' other kernel, the norm pass, the same way (when it is
    # not the dominant one): its algorithmic reads and, with the committed
    # counters, its DRAM bytes (reads plus the previous clip's write-backs it
    # absorbs) over its own event-timed launch.
    norm_pass = None
    if (not (args.per_tensor or args.to_f32 or args.accumulate) and args.variant.startswith("split")
            and kernel != ("k_norm_tma" if args.variant.endswith("tma") else "k_grad_norm_partial")
            and seg_ms[0] > 0):
        nk = "k_norm_tma" if args.variant.endswith("tma") else "k_grad_norm_partial"
        nb = w.numel * w.elem_bytes
        norm_pass = {"kernel": nk, "launch_ms": round(seg_ms[0], 5), "algorithmic_bytes": nb,
                     "achieved": round(nb / (seg_ms[0] / 1e3) / 1e9, 1),
                     "frac": round(nb / (seg_ms[0] / 1e3) / 1e9 / peak, 4)}
        nt = traffic_from_profile(nk, args.variant, args.workload)
        norm_pass["traffic"] = nt
        if nt:
            norm_pass["dram_achieved"] = round(nt / (seg_ms[0] / 1e3) / 1e9, 1)
            norm_pass["dram_frac"] = round(nt / (seg_ms[0] / 1e3) / 1e9 / peak, 4)

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e and not args.per_tensor and not args.to_f32 and not args.accumulate:
        # Every step copies its inputs from pinned host memory into one of
        # the P device sets (a copy stream: the copy of step k+1 overlaps the
        # clip of step k, as a training loop would stage its next batch) and
        # reads its norm and flag back into pinned host memory.
        host = pristine.flat.cpu().pin_memory()
        n_e2e = max(3, min(20, args.steps))
        norm_h = torch.empty(n_e2e, dtype=torch.float32).pin_memory()
        flag_h = torch.empty(n_e2e, dtype=torch.int32).pin_memory()
        copy_stream = torch.cuda.Stream(dev)

        def e2e_steps(n):
            copied, clipped = [], []
            for k in range(n):
                b = k % P
                with torch.cuda.stream(copy_stream):
                    if k >= P:      # the set is free once the clip that used it is done
                        copy_stream.wait_event(clipped[k - P])
                    sets[b].flat.copy_(host, non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(copy_stream)
                    copied.append(ev)
                stream.wait_event(copied[k])
                nt, ft = clippers[b].clip_(w.max_norm, w.inv_scale, stream=stream)
                norm_h[k:k + 1].copy_(nt, non_blocking=True)
                flag_h[k:k + 1].copy_(ft, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(stream)
                clipped.append(ev)

        s0 = torch.cuda.Event(enable_timing=True)
        s1 = torch.cuda.Event(enable_timing=True)
        e2e_steps(min(3, n_e2e))                       # warm-up
        torch.cuda.synchronize()
        s0.record(stream)
        copy_stream.wait_stream(stream)
        e2e_steps(n_e2e)
        s1.record(stream)                              # after every clip, hence every copy
        s1.synchronize()
        for k in range(n_e2e):
            assert abs(float(norm_h[k]) - rec["norm"]) <= 1e-6 * rec["norm"], k
        e2e_ms = reduce_max(s0.elapsed_time(s1) / n_e2e)
        e2e = {"value": round(nbytes * world / (e2e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
               "h2d_bytes_per_step": host.numel() * host.element_size(),
               "d2h_bytes_per_step": norm_h.element_size() + flag_h.element_size(),
               "ms_per_step": round(e2e_ms, 4),
               "steps": n_e2e,
               "d2h": "the norm and the nonfinite flag (8 B); the clipped gradients stay "
                      "in device memory, where the optimizer step reads them",
               "bound": "the host-to-device copy of the 369 MB set from pinned memory; "
                        "the clip itself overlaps it",
               "pipelining": "the H2D copy of step k+1 (copy stream) overlaps the clip of step k"}

    cpu = cpu_all = None
    if rank == 0 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        hostset = oracle_inputs(pristine)
        sec, reps, r = time_oracle(hostset, w, args.cpu_seconds)
        assert r.decision_name == decision_name, (r.decision_name, decision_name)
        cpu = {"value": round(nbytes / sec / 1e9, 4), "unit": "GB/s", "cores": 1,
               "kind": "oracle",
               "sample": f"the whole {w.name} set ({w.numel} elements), {reps} pass(es), "
                         f"{sec:.2f} s per pass, single-threaded C fp64 oracle"}
        if not args.no_cpu_all_cores:
            cpu_all = oracle_all_cores(w, args.cpu_seconds / 2)

    for c in clippers:
        c.close()

    if rank == 0:
        value = value_bps / 1e9
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step_ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {
                "workload": w.name, "description": w.description, "tensors": len(w.layout),
                "elements": w.numel, "bytes_per_step": nbytes, "decision": decision_name,
                "variant": ("per_tensor" if args.per_tensor else "to_f32" if args.to_f32
                            else "accumulate" if args.accumulate
                            else args.variant), "pool": P,
                "l2_keep_mb": args.l2_keep_mb, "written_elements": written, "parallelism": f"replicas x{world}",
                "device": device_info,
                "l2": ("warm: one set re-read from L2, no flush" if args.warm else
                       "inputs larger than L2 (one set per step, pool of distinct sets); "
                       "L2 flushed before each timed run"),
                "graph": bool(args.graph),
                "timing": "CUDA events around each run of back-to-back clips on the "
                          "launching stream; restores between runs outside the events",
            },
            "frac_of_nominal_8tbs": round(value / NOMINAL_HBM_GBS, 4),
            "elements_per_s": round(w.numel * args.steps * world / (total_ms / 1e3), 1),
            "us_per_step_p10_p50_p90": [round(step_us[int(q * (len(step_us) - 1))], 2)
                                         for q in (0.1, 0.5, 0.9)],
            "kernel_ms": ({"norm": round(seg_ms[0], 5), "scale": round(seg_ms[2], 5)}
                          if args.variant.startswith("split") else
                          {"chunk_sums": round(seg_ms[0], 5), "final": round(seg_ms[1], 5),
                           "scale": round(seg_ms[2], 5)}
                          if args.variant == "three_kernel" else
                          {"persistent": round(seg_ms[2], 5)}),
            "kernel_ms_note": "each launch alone between events (no programmatic dependent "
                              "launch), the L2 not flushed between clips; a norm pass that "
                              "follows a writing clip also absorbs that clip's write-backs",
            "roofline": roofline,
            "norm_pass": norm_pass,
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": args.steps * launches_per_step,
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def run_adamw(args):
    """The fused clip + AdamW step (clip_grad_norm_adamw) on the ANDREA set,
    beside two unfused pipelines: this library's clip, then the same AdamW
    kernel alone (clip_adamw_step), and this library's clip, then torch's
    fused AdamW on the same tensors.  One JSON line."""
    import torch

    import global_l2_norm_gb300 as g
    from workloads import WORKLOADS, make_gradset

    dev = torch.device("cuda", 0)
    g.build()
    w = WORKLOADS[args.workload]
    stream = torch.cuda.current_stream(dev)
    P = pool_size(args.pool, args.steps)
    pristine = make_gradset(w, device=dev, flat=True)
    sets = [make_gradset(w, device=dev, flat=True) for _ in range(P)]
    states = []
    for s in sets:
        st = [tuple(torch.zeros(t.numel(), device=dev) for _ in range(3)) for t in s.tensors]
        for (wt, _, _) in st:
            wt.normal_(0.0, 0.02)
        states.append(st)
    clippers = [g.GradClipper(s.tensors) for s in sets]
    for c, st in zip(clippers, states):
        c.attach_adamw(st)
    hp = dict(lr=3e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 + (1 << 20), dtype=torch.uint8, device=dev)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)

    def timed(fn, steps, restore):
        total, done = 0.0, 0
        while done < steps:
            n = min(P, steps - done)
            restore()
            flush.fill_(1)
            e0.record(stream)
            for i in range(n):
                fn(i)
            e1.record(stream)
            e1.synchronize()
            total += e0.elapsed_time(e1)
            done += n
        return total / steps

    step_no = [0]

    def fused(i):
        step_no[0] += 1
        clippers[i].clip_adamw_(w.max_norm, w.inv_scale, step=step_no[0], **hp)

    # correctness of what is timed: the clip fires on this workload
    clippers[0].clip_adamw_(w.max_norm, w.inv_scale, step=1, **hp)
    decision = clippers[0].result()["decision"]
    timed(fused, args.warmup, lambda: None)
    fused_ms = timed(fused, args.steps, lambda: None)

    # unfused: clip (rewrites the gradients), then torch's fused AdamW.  Both
    # pipelines are also captured as one CUDA graph per timed run and
    # replayed, so that the comparison is between kernels, without the
    # optimizer's host-side work.
    params = [[torch.nn.Parameter(st[0].view(t.shape)) for st, t in zip(states[i], sets[i].tensors)]
              for i in range(P)]
    for i in range(P):
        for prm, t in zip(params[i], sets[i].tensors):
            prm.grad = t if t.dtype == torch.float32 else None
    have_torch = all(p_.grad is not None for ps in params for p_ in ps)
    unfused_ms = unfused_graph_ms = fused_graph_ms = None

    def restore_grads():
        for s_ in sets:
            s_.flat.copy_(pristine.flat)

    def graph_of(fn):
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):      # warm-up on a side stream, as capture wants
            for i in range(P):
                fn(i)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gr):
            for i in range(P):
                fn(i)
        torch.cuda.synchronize()
        return gr

    def timed_graph(gr, steps, restore):
        total, done = 0.0, 0
        while done < steps:
            restore()
            flush.fill_(1)
            e0.record(stream)
            gr.replay()
            e1.record(stream)
            e1.synchronize()
            total += e0.elapsed_time(e1)
            done += P
        return total / done

    # unfused within the library: the clip rewrites the gradients, then the
    # AdamW kernel alone reads them (40 B per fp32 element against 32 fused)
    def unfused_lib(i):
        step_no[0] += 1
        clippers[i].clip_(w.max_norm, w.inv_scale)
        clippers[i].adamw_step_(step=step_no[0], **hp)

    timed(unfused_lib, args.warmup, restore_grads)
    unfused_lib_ms = timed(unfused_lib, args.steps, restore_grads)

    fused_graph = graph_of(lambda i: clippers[i].clip_adamw_(w.max_norm, w.inv_scale, step=7, **hp))
    timed_graph(fused_graph, args.warmup, lambda: None)
    fused_graph_ms = timed_graph(fused_graph, args.steps, lambda: None)
    del fused_graph
    if have_torch:
        opts = [torch.optim.AdamW(ps, fused=True, capturable=True,
                                  **{k: v for k, v in hp.items() if k not in ("beta1", "beta2")},
                                  betas=(hp["beta1"], hp["beta2"])) for ps in params]

        def unfused(i):
            clippers[i].clip_(w.max_norm, w.inv_scale)
            opts[i].step()

        timed(unfused, args.warmup, restore_grads)
        unfused_ms = timed(unfused, args.steps, restore_grads)
        unfused_graph = graph_of(unfused)
        timed_graph(unfused_graph, args.warmup, restore_grads)
        unfused_graph_ms = timed_graph(unfused_graph, args.steps, restore_grads)
        del unfused_graph

    es = w.elem_bytes
    fused_bytes = w.numel * (2 * es + 24)        # g read twice; w, m, v read and written
    # clip 3 * es; AdamW reads g, w, m, v and writes w, m, v
    unfused_bytes = w.numel * (3 * es + 4 + 12 + 12) if have_torch else None
    unfused_lib_bytes = w.numel * (3 * es + es + 24)   # AdamW reads g in its own format
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
    except (OSError, ValueError):
        pass
    peak = peaks.get("hbm_gbs") or 6800.0
    value = fused_bytes / (fused_ms / 1e3) / 1e9
    line = {
        "metric": "fused clip + AdamW step GB/s (algorithmic), " + w.name,
        "value": round(value, 2), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(fused_ms, 5), "higher_is_better": True,
        "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": w.name, "decision": {0: "pass", 1: "clip", 2: "skip"}[decision],
                   "bytes_per_step": fused_bytes, "pool": P, "adamw": hp,
                   "l2": "pool of distinct sets, L2 flushed before each timed run"},
        "roofline": {"bound": "hbm", "achieved": round(value, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(value / peak, 4)},
        "fused_graph_ms_per_step": round(fused_graph_ms, 5),
        "unfused_library": {
            "what": "clip_grad_norm (split), then clip_adamw_step (the same AdamW kernel alone, "
                    "multiplier 1)",
            "ms_per_step": round(unfused_lib_ms, 5), "bytes_per_step": unfused_lib_bytes,
            "value": round(unfused_lib_bytes / (unfused_lib_ms / 1e3) / 1e9, 2), "unit": "GB/s",
            "speedup_of_fused": round(unfused_lib_ms / fused_ms, 3)},
        "unfused": None if unfused_ms is None else {
            "what": "clip_grad_norm (split) then torch.optim.AdamW(fused=True, capturable=True)",
            "ms_per_step": round(unfused_ms, 5),
            "ms_per_step_note": "eager: includes torch's host-side optimizer work",
            "graph_ms_per_step": round(unfused_graph_ms, 5),
            "graph_note": "both pipelines captured as one CUDA graph per timed run and "
                          "replayed: kernel time only",
            "bytes_per_step": unfused_bytes,
            "speedup_of_fused": round(unfused_ms / fused_ms, 3),
            "speedup_of_fused_graphs": round(unfused_graph_ms / fused_graph_ms, 3)},
    }
    for c in clippers:
        c.close()
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.adamw:
        return run_adamw(args)
    return run_gclip(args)


if __name__ == "__main__":
    sys.exit(main())
