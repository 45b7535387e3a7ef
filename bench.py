#!/usr/bin/env python3
"""Throughput of the GB300 LSD radix sort on its headline workload.

One step = one whole sort (every digit pass, through the C ABI) of 2^28
uniform uint32 keys, keys only, bits [0, 32), with the keys already resident
in HBM.  Prints ONE JSON line (rank 0):

  value      Gkeys/s over all ranks (each rank sorts its own replica: the sort
             does not shard, so N GPUs run N independent sorts, weak scaling)
  roofline   the dominant kernel's algorithmic bytes per launch / its average
             CUDA-event duration, against the measured HBM copy bandwidth
  e2e        the same metric through rs_sort_host_batches with pinned host
             buffers: every step copies its input in and its result out
             inside the timed region, pipelined across steps (one step's sort
             overlaps the next one's copy in and the previous one's copy
             out); e2e.serial = one rs_sort_host call per step, unpipelined
  cpu_baseline  the CPU oracle (single thread) on a bounded sample

`--impl reference` times the CPU oracle itself as the reference arm.
"""
from __future__ import annotations

import argparse
import ctypes
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

METRIC = "Gkeys/s sorted (32-bit keys, 2^28) on 1 GB300; % of HBM roofline"
DEFAULT_WORKLOAD = "u32_uniform_2p28"
L2_BYTES = 126 * 2**20
FALLBACK_HBM_GBS = 6800.0
KIND_NAMES = {1: "histogram", 2: "onesweep_pass", 3: "upsweep", 4: "spine_scan", 5: "downsweep",
              6: "copy", 7: "cluster_sort"}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--log2n", type=int, default=None, help="override the size (uniform u32 sweep)")
    ap.add_argument("--algo", default="auto", choices=["auto", "onesweep", "reduce_scan", "cluster"])
    ap.add_argument("--radix-bits", type=int, default=0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--lib", default=None,
                    help="path of a variant build of librs.so (python -m lsd_radix_sort_key_gb300._build "
                         "--libdir DIR --flags ...) to run instead of the default one")
    ap.add_argument("--lbvh", action="store_true",
                    help="time the LBVH radix-tree build over the sorted codes of the workload "
                         "(default workload then morton30_index_2p28) instead of the sort")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def dist_setup(args):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if ws > 1:
        import torch.distributed as dist
        import torch
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
        pg = dist
    return ws, rank, local, pg


def barrier(pg):
    if pg is not None:
        pg.barrier()


def max_over_ranks(pg, x: float, device) -> float:
    if pg is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return float(t.item())


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": FALLBACK_HBM_GBS}, "fallback"


def kernel_source_hash() -> str:
    """sha256 (first 16 hex digits) of the code, without comments, of the
    files that define or instantiate device code: the kernels, their shapes
    and the per-key-type translation units.  The host entry layer (argument
    checks, schedule choice) is left out: changing it changes no kernel."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "lsd_radix_sort_key_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        if fn in ("rs_kernels.cuh", "rs_config.h") or (fn.startswith("rs_sort_") and fn.endswith(".cu")):
            with open(os.path.join(csrc, fn), encoding="utf-8") as f:
                h.update(fn.encode())
                h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def code_only(text: str) -> str:
    """C/C++ source without comments and with whitespace collapsed, so that
    the source hash changes with the code and not with its comments."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # string or character literal, kept whole
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def ncu_traffic(kind: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if its kernel
    sources are the ones built now; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        data = json.load(f)
    entry = data.get(f"{kind}:{workload}")
    if not entry or entry.get("source_hash") != kernel_source_hash():
        return None
    return entry.get("dram_bytes_per_launch")


def link_times(host_in, host_out, dev_buf, dev) -> dict:
    """The host link on this machine, for reading e2e: one step's input copied
    in alone, its result copied out alone, and both at once on two streams
    (3 of each, CUDA events; `*_ms` the fastest, `*_slowest_ms` the slowest).
    The pipelined e2e step cannot beat `both_ms`; single copies on these
    hosts now and then stall for tens of milliseconds, which the slowest
    samples show."""
    import torch
    nbytes = host_in.numel() * host_in.element_size()
    d_in = dev_buf[:nbytes].view(host_in.dtype)
    d_out = dev_buf[nbytes:2 * nbytes].view(host_in.dtype)
    side = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]

    def samples(fn):
        ms = []
        for _ in range(3):
            cur = torch.cuda.current_stream(dev)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(cur)
            fn(cur)
            e1.record(cur)
            torch.cuda.synchronize(dev)
            ms.append(e0.elapsed_time(e1))
        return ms

    def both(cur):
        for sd in side:
            sd.wait_stream(cur)
        with torch.cuda.stream(side[0]):
            d_in.copy_(host_in, non_blocking=True)
        with torch.cuda.stream(side[1]):
            host_out.copy_(d_out, non_blocking=True)
        for sd in side:
            cur.wait_stream(sd)
    out = {"bytes": nbytes}
    for name, fn in (("h2d", lambda cur: d_in.copy_(host_in, non_blocking=True)),
                     ("d2h", lambda cur: host_out.copy_(d_out, non_blocking=True)),
                     ("both", both)):
        ms = samples(fn)
        out[f"{name}_ms"] = round(min(ms), 3)
        out[f"{name}_slowest_ms"] = round(max(ms), 3)
    return out


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        mhz, maxes, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                mhz.append(float(parts[1]))
                maxes.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not mhz:
            return None
        return {"sm_mhz": statistics.median(mhz), "sm_max_mhz": max(maxes) if maxes else None,
                "reasons": sorted(reasons), "samples": len(mhz)}


def host_info():
    """This host's CPU: online cores, the C++ runtime's hardware_concurrency(),
    and the model from /proc/cpuinfo (x86 "model name"; on Arm the
    implementer and part codes)."""
    import oracle
    model, impl, part = None, None, None
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                k, v = k.strip().lower(), v.strip()
                if k in ("model name", "hardware") and v and model is None:
                    model = v
                elif k == "cpu implementer" and impl is None:
                    impl = v
                elif k == "cpu part" and part is None:
                    part = v
    except OSError:
        pass
    if model is None and impl is not None:
        model = f"arm implementer {impl} part {part}"
    return {"cores_online": os.cpu_count(), "hardware_concurrency": oracle.hardware_concurrency(),
            "cpu_model": model}


def _timed(fn, budget_s, max_reps=50):
    fn()  # warm (pages, caches)
    reps, t0 = 0, time.perf_counter()
    while True:
        fn()
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= max_reps:
            return reps, el


def cpu_baseline(workload, key_type, begin_bit, end_bit, log2n, budget_s=10.0):
    """The CPU oracle (one thread) on a bounded sample of the same workload, and
    beside it three more CPU sorts: one std::stable_sort of the same problem,
    the one-bit index-formula sort of "Radix sort を実装 & 測定してみた"
    (section 測定 times it on the CPU), both single-threaded on smaller
    samples, and a multi-threaded LSD radix sort on all host threads."""
    import oracle
    import synth
    sample_log2 = min(log2n, 24)
    n = 1 << sample_log2
    keys = workload.keys(n) if log2n is None or workload.log2n == log2n else synth.u32_uniform(n, 1)
    vals = workload.values(n)
    reps, el = _timed(lambda: oracle.sort(key_type, keys, vals, begin_bit, end_bit), budget_s)
    out = {"value": round(n * reps / el / 1e9, 6), "unit": "Gkeys/s", "cores": 1,
           "kind": "oracle",
           "sample": f"{reps} x oracle sort of the first 2^{sample_log2} keys of the workload "
                     f"({el:.1f} s single-threaded C counting-sort LSD, r=8)",
           "host": host_info()}
    others = []
    par_threads = oracle.parallel_threads()
    for kind, log2s, fn, what, cores in (
            ("std::stable_sort", min(sample_log2, 22), oracle.stable_sort_baseline,
             "single-threaded C++ std::stable_sort of (ordered key bits, index) records", 1),
            ("one_bit_split", min(sample_log2, 20), oracle.one_bit_split_sort,
             "single-threaded one-bit index-formula LSD sort, one pass per key bit", 1),
            ("parallel_lsd", sample_log2, oracle.parallel_lsd_sort,
             f"multi-threaded 8-bit LSD radix sort, one block per thread, on {par_threads} host threads",
             par_threads)):
        m = 1 << log2s
        k, v = keys[:m], None if vals is None else vals[:m]
        r, t = _timed(lambda: fn(key_type, k, v, begin_bit, end_bit), budget_s / 2)
        others.append({"kind": kind, "value": round(m * r / t / 1e9, 6), "unit": "Gkeys/s", "cores": cores,
                       "sample": f"{r} x sort of the first 2^{log2s} keys of the workload ({t:.1f} s, {what})"})
    out["others"] = others
    return out


# --------------------------------------------------------------- reference

def run_reference(args):
    ws, rank, local, pg = dist_setup(args)
    if rank != 0:
        return
    import synth
    import oracle
    w = synth.WORKLOADS[args.workload] if args.log2n is None else synth.sweep_workload(args.log2n)
    sample_log2 = min(w.log2n, 22)
    n = 1 << sample_log2
    keys = w.keys(n)
    vals = w.values(n)
    for _ in range(args.warmup):
        oracle.sort(w.key_type, keys, vals, w.begin_bit, w.end_bit)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.sort(w.key_type, keys, vals, w.begin_bit, w.end_bit)
    el = time.perf_counter() - t0
    value = n * args.steps / el / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "Gkeys/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.key_type, "data": "synthetic",
            "config": {"workload": w.name, "n": w.n, "sample_n": n, "key_type": w.key_type,
                       "begin_bit": w.begin_bit, "end_bit": w.end_bit,
                       "values": w.with_values},
            "cpu_baseline": {"value": round(value, 6), "unit": "Gkeys/s", "cores": 1,
                             "kind": "oracle",
                             "sample": f"each step sorts the first 2^{sample_log2} keys of the "
                                       "workload with the single-threaded CPU oracle",
                             "host": host_info()},
            "e2e": {"value": round(value, 6), "unit": "Gkeys/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- lbvh

def run_lbvh(args):
    """Time rs_lbvh_build over the workload's codes, sorted once on the device
    by the library beforehand (outside the timed region).  One line of JSON:
    Gnodes/s (internal nodes built per second) and the kernel against HBM:
    its algorithmic bytes are the codes read once (4 B each) plus the six
    output arrays written once (5 x 4 B per internal node, 4 B per leaf)."""
    import numpy as np
    import torch

    import lsd_radix_sort_key_gb300 as rs
    import synth

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    rs.lib()
    name = args.workload if args.workload != DEFAULT_WORKLOAD else "morton30_index_2p28"
    w = synth.WORKLOADS[name]
    if args.log2n is not None:  # the same codes at another size (a prefix of the same stream)
        import dataclasses
        w = dataclasses.replace(w, log2n=args.log2n)
        name = f"{name}@2p{args.log2n}"
    if w.key_type != "u32":
        raise SystemExit("--lbvh needs a workload of uint32 codes")
    n = w.n
    host = torch.empty(n, dtype=torch.int32).pin_memory()
    w.keys(out=host.numpy().view(np.uint32))
    kin = host.to(dev)
    vin = torch.arange(n, dtype=torch.int32, device=dev)
    codes, _ = rs.sort(kin, vin, key_type="u32", begin_bit=w.begin_bit, end_bit=w.end_bit)
    del kin, vin
    out = {k: torch.empty(n - 1, dtype=torch.int32, device=dev)
           for k in ("left", "right", "first", "last", "node_parent")}
    out["leaf_parent"] = torch.empty(n, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def build():
        st = rs.rs_lbvh_build(codes, n, out["left"], out["right"], out["first"], out["last"],
                              out["leaf_parent"], out["node_parent"], stream)
        assert st == 0, rs.STATUS.get(st)

    for _ in range(max(args.warmup, 3)):
        build()
    torch.cuda.synchronize(dev)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    clocks = ClockSampler(0)
    clocks.start()
    evs[0].record(stream)
    for s in range(args.steps):
        build()
        evs[s + 1].record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    per = [evs[s].elapsed_time(evs[s + 1]) for s in range(args.steps)]
    ms = statistics.mean(per)
    peaks, peak_kind = measured_peaks()
    alg = 4 * n + 20 * (n - 1) + 4 * n
    achieved = alg / (ms * 1e-3) / 1e9
    line = {"metric": f"Gnodes/s (LBVH radix tree over {n} sorted Morton codes) on 1 GB300",
            "value": round((n - 1) / (ms * 1e-3) / 1e9, 3), "unit": "Gnodes/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u32",
            "data": "synthetic", "config": {"workload": name, "n": n, "inputs": "larger than L2, no flush",
                                             "codes": "sorted by rs_sort_pairs_u32 before the timed region"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"],
                         "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / peaks["hbm_gbs"], 4),
                         "algorithmic_bytes_per_launch": alg},
            "gpu_launches": args.steps, "clocks": clk}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------- ours

def run_ours(args):
    import numpy as np
    import torch

    import lsd_radix_sort_key_gb300 as rs
    import synth

    ws, rank, local, pg = dist_setup(args)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    rs.lib()

    w = synth.WORKLOADS[args.workload] if args.log2n is None else synth.sweep_workload(args.log2n)
    kt, n, b, e = w.key_type, w.n, w.begin_bit, w.end_bit
    kbytes = rs.KEY_BYTES[kt]
    tdt = torch.int64 if kbytes == 8 else torch.int32
    # Each rank sorts its own replica (seed offset by rank): no data-path exchange.
    host_k = torch.empty(n, dtype=tdt).pin_memory()
    import dataclasses
    wr = dataclasses.replace(w, seed=w.seed + (rank << 40))
    wr.keys(out=host_k.numpy().view(np.uint64 if kbytes == 8 else np.uint32))
    host_v = None
    if w.with_values:
        host_v = torch.empty(n, dtype=torch.int32).pin_memory()
        synth.iota_u32(n, out=host_v.numpy().view(np.uint32))
    kin = host_k.to(dev)
    vin = host_v.to(dev) if host_v is not None else None
    kout = torch.empty_like(kin)
    vout = torch.empty_like(vin) if vin is not None else None
    tb = rs.rs_temp_bytes(kt, w.with_values, n, b, e)
    temp = torch.empty(tb, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    desc = rs.make_desc(kt, kin, kout, vin, vout, n, b, e, temp, tb, stream, args.algo,
                        args.radix_bits)
    nk = rs.rs_sort_kernel_count(desc)
    events = [torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
    step_events = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
                   for _ in range(args.steps)]

    for _ in range(max(args.warmup, 3)):
        st, kinds = rs.rs_sort_profiled(desc, events)
        assert st == 0, rs.STATUS.get(st)
    torch.cuda.synchronize(dev)
    status = rs.rs_device_status(temp, stream)
    assert status == 0, rs.STATUS.get(status)

    # The timed region: the K sorts, each with CUDA events between its
    # kernels (rs_sort_profiled), captured once into one CUDA graph and
    # replayed.  The whole-sort metric is defined on graph replays; the events
    # inside the graph give every kernel's duration in that same region.
    cap = torch.cuda.Stream(dev)
    desc_g = rs.make_desc(kt, kin, kout, vin, vout, n, b, e, temp, tb, cap, args.algo,
                          args.radix_bits)
    graph = torch.cuda.CUDAGraph()
    torch.cuda.synchronize(dev)
    with torch.cuda.graph(graph, stream=cap, capture_error_mode="thread_local"):
        for s in range(args.steps):
            st, kinds = rs.rs_sort_profiled(desc_g, step_events[s])
            assert st == 0, rs.STATUS.get(st)
    graph.replay()  # warm the instantiated graph once
    torch.cuda.synchronize(dev)
    assert rs.rs_device_status(temp, stream) == 0

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    barrier(pg)
    torch.cuda.synchronize(dev)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    graph.replay()
    end.record()
    torch.cuda.synchronize(dev)
    barrier(pg)
    clk = clocks.stop()
    total_ms = start.elapsed_time(end)
    total_ms = max_over_ranks(pg, total_ms, dev)
    status = rs.rs_device_status(temp, stream)
    assert status == 0, rs.STATUS.get(status)

    # Per-kernel durations inside the timed region.
    per_kind = {}
    for s in range(args.steps):
        ev = step_events[s]
        for i, k in enumerate(kinds):
            per_kind.setdefault(k, []).append(ev[i].elapsed_time(ev[i + 1]))
    ms_per_step = total_ms / args.steps
    value = n * ws / (ms_per_step * 1e-3) / 1e9

    peaks, peak_src = measured_peaks()
    hbm = float(peaks["hbm_gbs"])
    vbytes = 4 if w.with_values else 0
    passes = -(-(e - b) // (args.radix_bits or 8)) if e > b else 0
    # algorithmic bytes per launch of each kernel kind
    algo_bytes = {1: n * kbytes, 2: n * 2 * (kbytes + vbytes), 3: n * kbytes, 4: 0,
                  5: n * (kbytes + 2 * (kbytes + vbytes)) - n * kbytes, 6: n * 2 * (kbytes + vbytes),
                  7: n * 2 * (kbytes + vbytes)}
    dominant = max(per_kind, key=lambda k: sum(per_kind[k]))
    dom_ms = statistics.mean(per_kind[dominant])
    dom_bytes = algo_bytes[dominant]
    achieved = dom_bytes / (dom_ms * 1e-3) / 1e9
    kernels = {KIND_NAMES[k]: {"launches_per_step": len(v) // args.steps,
                               "avg_ms": round(statistics.mean(v), 4),
                               "share": round(sum(v) / sum(sum(x) for x in per_kind.values()), 4)}
               for k, v in per_kind.items()}
    resolved = "cluster" if 7 in per_kind else "onesweep" if 2 in per_kind else "reduce_scan"
    if resolved == "cluster":  # global memory is read once and written once
        scheme_bpk = 2 * (kbytes + vbytes)
    else:
        scheme_bpk = ((kbytes if resolved == "onesweep" else passes * kbytes)
                      + passes * 2 * (kbytes + vbytes))
    ideal_bpk = passes * 2 * (kbytes + vbytes)
    sort_gbs = n * scheme_bpk / (ms_per_step * 1e-3) / 1e9

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "Gkeys/s", "n_gpus": ws,
        "steps": args.steps, "warmup": max(args.warmup, 3), "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": kt,
        "data": "synthetic",
        "config": {"workload": w.name, "n": n, "key_type": kt, "begin_bit": b, "end_bit": e,
                   "values": w.with_values, "algo": resolved, "radix_bits": args.radix_bits or 8,
                   "passes": passes, "parallelism": f"replicas x{ws}",
                   "timed": "one CUDA graph of the K sorts (events between kernels), replayed once",
                   "l2": "inputs larger than L2 (no flush needed)" if n * kbytes > L2_BYTES
                   else "inputs fit in L2 (no flush: L2-resident number)"},
        "roofline": {"bound": "hbm", "kernel": KIND_NAMES[dominant],
                     "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4), "peak_source": peak_src,
                     "traffic": ncu_traffic(KIND_NAMES[dominant], w.name),
                     "algorithmic_bytes_per_launch": dom_bytes,
                     "avg_launch_ms": round(dom_ms, 4)},
        "sort_roofline": {"scheme": resolved, "bytes_per_key": scheme_bpk,
                          "ideal_bytes_per_key": ideal_bpk,
                          "achieved_gbs": round(sort_gbs, 1),
                          "frac_scheme": round(sort_gbs / hbm, 4),
                          "frac_ideal": round(n * ideal_bpk / (ms_per_step * 1e-3) / 1e9 / hbm, 4)},
        "kernels": kernels,
        "gpu_launches": nk * args.steps,
        "clocks": clk,
    }

    # The same K sorts launched from the host one by one (no graph): what a
    # caller that enqueues rs_sort directly sees.
    del graph
    barrier(pg)
    torch.cuda.synchronize(dev)
    l0, l1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0.record(stream)
    for s in range(args.steps):
        st, _ = rs.rs_sort_profiled(desc, step_events[s])
        assert st == 0
    l1.record(stream)
    torch.cuda.synchronize(dev)
    launch_ms = max_over_ranks(pg, l0.elapsed_time(l1), dev) / args.steps
    assert rs.rs_device_status(temp, stream) == 0
    line["launches"] = {"value": round(n * ws / (launch_ms * 1e-3) / 1e9, 3), "unit": "Gkeys/s",
                        "ms_per_step": round(launch_ms, 4),
                        "api": "rs_sort_profiled called per sort from the host (no graph)"}

    # The library's own graph API (rs_graph_*): the same sort without the
    # event nodes, replayed K times.
    rgraph = rs.Graph(desc)
    for _ in range(3):
        rgraph.launch(stream)
    torch.cuda.synchronize(dev)
    barrier(pg)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0.record(stream)
    for _ in range(args.steps):
        rgraph.launch(stream)
    g1.record(stream)
    torch.cuda.synchronize(dev)
    graph_ms = max_over_ranks(pg, g0.elapsed_time(g1), dev) / args.steps
    rgraph.close()
    assert rs.rs_device_status(temp, stream) == 0
    line["graph"] = {"value": round(n * ws / (graph_ms * 1e-3) / 1e9, 3), "unit": "Gkeys/s",
                     "ms_per_step": round(graph_ms, 4),
                     "api": "rs_graph_create / rs_graph_launch (no events inside)"}

    # End to end through the C ABI with host buffers.
    if not args.no_e2e:
        host_ko = torch.empty_like(host_k).pin_memory()
        host_vo = torch.empty_like(host_v).pin_memory() if host_v is not None else None
        del kout, vout, kin, vin
        wb = rs.rs_host_work_bytes(kt, w.with_values, n, b, e)
        del temp
        torch.cuda.empty_cache()
        work = torch.empty(wb, dtype=torch.uint8, device=dev)
        for _ in range(2):
            assert rs.rs_sort_host(kt, host_k, host_ko, host_v, host_vo, n, b, e, work, wb,
                                   stream) == 0
        torch.cuda.synchronize(dev)
        # Up to 40 steps (~0.3 s pipelined): the host link now and then stalls
        # a single copy for tens of milliseconds, and a longer region weighs
        # one such stall less without leaving it out.
        e2e_steps = max(3, min(args.steps, 40))
        barrier(pg)
        s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s0.record(stream)
        for _ in range(e2e_steps):
            assert rs.rs_sort_host(kt, host_k, host_ko, host_v, host_vo, n, b, e, work, wb,
                                   stream) == 0
        s1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(pg, s0.elapsed_time(s1), dev) / e2e_steps
        serial = {"value": round(n * ws / (e2e_ms * 1e-3) / 1e9, 3), "unit": "Gkeys/s",
                  "ms_per_step": round(e2e_ms, 3), "steps": e2e_steps,
                  "api": "rs_sort_host, one call per step (copy in, sort, copy out in sequence)"}
        del work
        torch.cuda.empty_cache()

        # The same steps pipelined through rs_sort_host_batches: step i's
        # sort overlaps step i+1's copy in and step i-1's copy out.  Every
        # step still copies its whole input in and its whole result out
        # inside the timed region.
        wb2 = rs.rs_host_batches_work_bytes(kt, w.with_values, n, b, e)
        work2 = torch.empty(wb2, dtype=torch.uint8, device=dev)
        outs_k = [torch.empty_like(host_k).pin_memory() for _ in range(2)]
        outs_v = [torch.empty_like(host_v).pin_memory() for _ in range(2)] if host_v is not None else None

        def batches(k):
            return ([host_k] * k, [outs_k[i % 2] for i in range(k)],
                    [host_v] * k if host_v is not None else None,
                    [outs_v[i % 2] for i in range(k)] if host_v is not None else None)
        assert rs.rs_sort_host_batches(kt, *batches(2), n, b, e, work2, wb2, stream) == 0
        torch.cuda.synchronize(dev)
        # The host link is sampled right before and right after the timed
        # region: its speed varies over time on a shared host (1 GiB copies
        # measured from 5 ms to 37 ms on one box), and the pipelined step
        # cannot beat the both-directions time of that moment.
        link_before = link_times(host_k, outs_k[0], work2, dev)
        barrier(pg)
        s0.record(stream)
        assert rs.rs_sort_host_batches(kt, *batches(e2e_steps), n, b, e, work2, wb2, stream) == 0
        s1.record(stream)
        torch.cuda.synchronize(dev)
        pipe_ms = max_over_ranks(pg, s0.elapsed_time(s1), dev) / e2e_steps
        # both paths give the same bytes
        assert torch.equal(outs_k[0], host_ko) and torch.equal(outs_k[1], host_ko)
        if host_v is not None:
            assert torch.equal(outs_v[0], host_vo) and torch.equal(outs_v[1], host_vo)
        line["e2e"] = {"value": round(n * ws / (pipe_ms * 1e-3) / 1e9, 3), "unit": "Gkeys/s",
                       "h2d_bytes_per_step": n * (kbytes + vbytes),
                       "d2h_bytes_per_step": n * (kbytes + vbytes),
                       "ms_per_step": round(pipe_ms, 3), "steps": e2e_steps,
                       "api": "rs_sort_host_batches (pinned host buffers, one batch per step, pipelined)",
                       "serial": serial, "link_before": link_before,
                       "link": link_times(host_k, outs_k[0], work2, dev)}
        del work2

    if rank == 0 and not args.no_cpu:
        line["cpu_baseline"] = cpu_baseline(w, kt, b, e, w.log2n)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if pg is not None:
        pg.destroy_process_group()


def main():
    args = parse()
    if args.lib:
        import lsd_radix_sort_key_gb300 as rs
        rs.LIB_PATH = os.path.abspath(args.lib)
    if args.impl == "reference":
        run_reference(args)
    elif args.lbvh:
        run_lbvh(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
