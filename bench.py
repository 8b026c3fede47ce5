"""Benchmark of the KDA chunked forward on GB300 (tokens/s and HBM roofline).

python bench.py [--gpus N] [--steps K] [--warmup W] [--workload fixed] [--impl ours|reference]

One step = one full KDA forward (varlen schedule if any, prep kernel,
recurrence kernel) over the workload's synthetic inputs, which are resident in
HBM before timing starts. Between timed steps L2 is flushed by writing a
256 MiB buffer outside the per-step CUDA events. Under torchrun every rank runs
its own replica of the workload (the (sequence, head) recurrences are
independent, so the work shards with no collective): per-GPU work is fixed and
`value` is the total tokens of all ranks over the slowest rank's time.

Printed on rank 0: one JSON line with the metric, the roofline of the dominant
kernel and of the other one, the end-to-end figure through the public API with
host buffers, the clocks seen during the timed region, and the CPU baseline:
the fp64 oracle timed on this host's cores on a bounded sample.

The timed steps carry CUDA events only before and after the forward, so the
recurrence kernel's launch overlaps the end of the prep kernel as it does for
any caller. The per-kernel times of the rooflines come from as many further
steps, run right after the timed ones, with an event recorded by the library
between the two kernels (which serialises them).
"""
from __future__ import annotations

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

METRIC = "KDA fwd tokens/sec (1xGB300) and achieved HBM GB/s as % of roofline vs oracle"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="fixed",
                    choices=["tiny", "fixed", "varlen", "long", "large_batch"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cp", default="auto",
                    help="context parallelism: auto (the library's plan), off, or a segment count")
    ap.add_argument("--heads", type=int, default=None,
                    help="override the workload's head count (same shapes and distributions otherwise)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override a fixed-length workload's batch size (a smaller case of the same "
                         "shape, e.g. for an ncu capture)")
    return ap.parse_args()


def cp_arg(text):
    """The --cp argument as kda.fwd's context_parallel: None (auto), False (off) or a count."""
    if text == "auto":
        return None
    if text == "off":
        return False
    return int(text)


def workload_of(args):
    from dataclasses import replace
    from chunked_gated_delta_02_gb300.workloads import named
    w = named(args.workload)
    batch = getattr(args, "batch", None)
    if batch:
        if w.is_varlen:
            raise SystemExit("--batch applies to fixed-length workloads")
        w = replace(w, B=batch)
    heads = getattr(args, "heads", None)
    return replace(w, H=heads) if heads else w


# --------------------------------------------------------------------------- helpers
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def algorithmic_bytes(inp, with_state=True) -> int:
    """Bytes the operation must move: read q,k,g,v,beta (+ initial state), write o (+ final state).

    Per token-head that is 3K + V bf16 values and one bf16 beta in, V bf16 values out (1282 B at
    K = V = 128); the state adds V K fp32 values per (sequence, head) for each direction used."""
    B, T, H, K, V, N = (inp[x] for x in ("B", "T", "H", "K", "V", "N"))
    th = B * T * H
    io = th * (3 * K * 2 + V * 2 + 2 + V * 2)
    if not with_state:
        return io
    state = N * H * V * K * 4
    return io + state * (1 if inp["initial_state"] is not None else 0) + state  # final_state written


def max_over_ranks(vals, device=None):
    """Element-wise maximum of a list of floats over all ranks (the list itself with one rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(x) for x in vals]
    t = torch.tensor([float(x) for x in vals], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_rate(units_per_rank, world_size, ms_max):
    """Units per second of the whole job: every rank processes its own replica of the workload, and
    the job takes as long as its slowest rank."""
    return units_per_rank * world_size / (ms_max * 1e-3)


def kernel_algorithmic_bytes(inp):
    """Bytes each kernel must move by itself, per launch.

    The prep kernel (K1) must read q, k, g and beta: 3K bf16 values and one bf16 beta per
    token-head (770 B at K = 128). The recurrence kernel (K2) must read v and write o (2V bf16
    values per token-head, 512 B at V = 128) and read / write the state (V K fp32 values per
    (sequence, head) and direction). The two add up to the whole path's algorithmic bytes; what
    K1 hands K2 through the workspace is not algorithmic and is not credited to either."""
    B, T, H, K, V, N = (inp[x] for x in ("B", "T", "H", "K", "V", "N"))
    th = B * T * H
    state = N * H * V * K * 4
    prep = th * (3 * K * 2 + 2)
    rec = th * (2 * V * 2) + state * (1 if inp["initial_state"] is not None else 0) + state
    assert prep + rec == algorithmic_bytes(inp)
    return {"prep": prep, "recurrence": rec}


def kernel_rooflines(inp, ms_prep, ms_rec, peak, peak_src, workload):
    """HBM roofline of each kernel: its own algorithmic bytes per launch over its measured time,
    with the ncu DRAM traffic of the same kernel when the committed capture matches the current
    sources. The dominant kernel (longer time) comes first."""
    ab = kernel_algorithmic_bytes(inp)
    out = []
    for name, key, ms in (("prep (K1)", "prep", ms_prep), ("recurrence (K2)", "recurrence", ms_rec)):
        gbs = ab[key] / (ms * 1e-3) / 1e9
        tr = ncu_traffic(workload, key)
        out.append({"bound": "hbm", "kernel": name, "achieved": gbs, "peak": peak, "unit": "GB/s",
                    "frac": gbs / peak, "traffic": tr,
                    "traffic_over_algorithmic": (tr / ab[key]) if tr else None,
                    "algorithmic_bytes_per_launch": ab[key], "ms_per_launch": ms, "peak_source": peak_src})
    out.sort(key=lambda r: -r["ms_per_launch"])
    return out


def tokens_of(inp) -> int:
    return inp["B"] * inp["T"]


def workload_desc(name, inp, w=None):
    from chunked_gated_delta_02_gb300.workloads import named
    w = w or named(name)
    return {"workload": f"{name} KDA fwd: {w.describe()}", "B": inp["B"], "T": inp["T"], "H": inp["H"],
            "K": inp["K"], "V": inp["V"], "num_seqs": inp["N"], "lower_bound": inp["lower_bound"],
            "tokens_per_step": tokens_of(inp), "token_heads_per_step": tokens_of(inp) * inp["H"],
            "l2": "flushed between timed steps (256 MiB write outside the per-step events)",
            "parallelism": "replicas (independent (sequence, head) recurrences; no collective)"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

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
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peak():
    try:
        with open(PEAKS_FILE) as fh:
            pk = json.load(fh)
        return float(pk["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, STREAM-style copy)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "chunked_gated_delta_02_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")):
            with open(os.path.join(csrc, name), "rb") as fh:
                h.update(name.encode())
                h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload, kernel):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernels."""
    try:
        with open(TRAFFIC_FILE) as fh:
            tr = json.load(fh)
    except (OSError, ValueError):
        return None
    ent = tr.get(workload, {}).get(kernel)
    if not ent or ent.get("source_hash") != kernel_source_hash():
        return None
    return ent.get("dram_bytes_per_launch")


# --------------------------------------------------------------------------- CPU oracle
def cpu_baseline(inp, target_s=8.0):
    """The fp64 oracle (plain C, all host cores) on a bounded sample of (sequence, head) pairs."""
    from oracle import c_oracle
    H = inp["H"]
    cu = inp["cu_seqlens"]
    lens = [int(cu[i + 1] - cu[i]) for i in range(inp["N"])] if cu is not None else [inp["T"]] * inp["N"]
    pairs_all = [(s, h) for s in range(inp["N"]) for h in range(H)]
    threads = c_oracle.default_threads()
    # calibrate on a few pairs, then size the sample to ~target_s of wall time
    probe = pairs_all[:max(1, min(len(pairs_all), threads))]
    t0 = time.perf_counter()
    c_oracle.kda_fwd_c(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"], inp["dt_bias"],
                       inp["lower_bound"], inp["scale"], inp["initial_state"], cu, pairs=probe,
                       n_threads=threads, full_o=False)
    dt = time.perf_counter() - t0
    rate = sum(lens[s] for s, _ in probe) / max(dt, 1e-6)        # token-heads per second
    want = rate * target_s
    import numpy as np
    perm = np.random.default_rng(0).permutation(len(pairs_all))      # an even spread over sequences/heads
    sample, th = [], 0
    for i in perm:
        sample.append(pairs_all[int(i)])
        th += lens[pairs_all[int(i)][0]]
        if th >= want:
            break
    reps, t0 = 0, time.perf_counter()
    while True:   # repeat the sample until about target_s of wall time has been spent
        c_oracle.kda_fwd_c(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"],
                           inp["dt_bias"], inp["lower_bound"], inp["scale"], inp["initial_state"], cu,
                           pairs=sample, n_threads=threads, full_o=False)
        reps += 1
        if time.perf_counter() - t0 >= target_s or reps >= 1000:
            break
    dt = (time.perf_counter() - t0) / reps
    token_heads = sum(lens[s] for s, _ in sample)
    return {"value": token_heads / H / dt, "unit": UNIT, "cores": threads, "kind": "oracle",
            "sample": (f"{len(sample)} of {len(pairs_all)} (sequence, head) pairs ({token_heads} token-heads), "
                       f"run {reps}x, {dt:.3f} s wall each on {threads} threads; "
                       f"tokens/s = token-heads/s / H"),
            "seconds": dt}


# --------------------------------------------------------------------------- runs
def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from chunked_gated_delta_02_gb300.workloads import make_inputs
    w = workload_of(args)
    inp = make_inputs(w, seed=args.seed)
    vals = []
    per_step = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    last = None
    for i in range(args.warmup + args.steps):
        last = cpu_baseline(inp, target_s=per_step)
        if i >= args.warmup:
            vals.append(last["value"])
    v = statistics.mean(vals) if vals else 0.0
    out = {"metric": METRIC, "value": v, "unit": UNIT, "impl": "reference", "n_gpus": 0,
           "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": tokens_of(inp) / v * 1e3 if v else None, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": workload_desc(args.workload, inp, w),
           "cpu_baseline": {"value": v, "unit": UNIT, "cores": last["cores"], "kind": "oracle",
                            "sample": last["sample"]},
           "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)
    import chunked_gated_delta_02_gb300 as kda
    from chunked_gated_delta_02_gb300.workloads import make_inputs
    w = workload_of(args)
    inp = make_inputs(w, seed=args.seed + rank)
    cp = cp_arg(args.cp)
    d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    B, T, H, K, V, N = (inp[x] for x in ("B", "T", "H", "K", "V", "N"))
    o = torch.empty(B, T, H, V, dtype=torch.bfloat16, device=dev)
    fs = torch.empty(N, H, V, K, dtype=torch.float32, device=dev)
    varlen = inp["cu_seqlens"] is not None
    wsb = torch.empty(kda.workspace_size(B, T, H, K, V, N, varlen, kda.kda._cp_flags(cp)), dtype=torch.uint8,
                      device=dev)
    n_seg, slice_w = kda.plan(B, T, H, K, V, N, varlen, cp)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    split_evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    warm_ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for e in warm_ev + [e for trip in evs + split_evs for e in trip]:
        e.record()
    torch.cuda.synchronize()

    def step(events):
        kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                d["scale"], d["initial_state"], True, d["cu_seqlens"], workspace=wsb, out=o, final_state=fs,
                events=events, context_parallel=cp)

    for _ in range(args.warmup):
        flush.fill_(1)
        step(warm_ev)
        flush.fill_(2)
        step((warm_ev[0], None, warm_ev[2]))
    torch.cuda.synchronize()
    clocks = ClockSampler(torch.cuda.current_device() if ws == 1 else local)
    clocks.start()
    time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    w0 = time.perf_counter()
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        step((evs[i][0], None, evs[i][2]))
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    wall = time.perf_counter() - w0
    # the per-kernel split: the same steps with an event between the kernels
    for i in range(args.steps):
        flush.fill_(i & 0xFF)
        step(split_evs[i])
    torch.cuda.synchronize()
    clk = clocks.stop()
    tot = [evs[i][0].elapsed_time(evs[i][2]) for i in range(args.steps)]
    prep = [split_evs[i][0].elapsed_time(split_evs[i][1]) for i in range(args.steps)]
    rec = [split_evs[i][1].elapsed_time(split_evs[i][2]) for i in range(args.steps)]
    ms = statistics.mean(tot)
    ms_rec = statistics.mean(rec)
    ms_prep = statistics.mean(prep)
    ms, ms_rec, ms_prep = max_over_ranks([ms, ms_rec, ms_prep], dev)
    e2e = None if args.no_e2e else run_e2e(args, inp, dev, kda, o, fs, wsb, cp)
    if rank == 0:
        peak, peak_src = measured_peak()
        abytes = algorithmic_bytes(inp)
        path_gbs = abytes / (ms * 1e-3) / 1e9
        # the committed ncu traffic is per named workload in its default plan
        resized = bool(args.heads or getattr(args, "batch", None))
        traffic_key = args.workload if (not resized and n_seg < 2) else f"{args.workload}-B{B}-H{H}-cp{n_seg}"
        roofs = kernel_rooflines(inp, ms_prep, ms_rec, peak, peak_src, traffic_key)
        if n_seg >= 2:
            roofs = [dict(r, kernel="recurrence (K2: local pass, combine, final pass)")
                     if r["kernel"].startswith("recurrence") else r for r in roofs]
        trs = [r["traffic"] for r in roofs]
        path_traffic = sum(trs) if all(t is not None for t in trs) else None
        kernels_per_step = (2 if n_seg >= 2 else 0) + 2 + (1 if inp["cu_seqlens"] is not None else 0)
        out = {"metric": METRIC, "value": whole_job_rate(tokens_of(inp), ws, ms), "unit": UNIT, "impl": "ours",
               "n_gpus": ws, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
               "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
               "data": "synthetic",
               "config": dict(workload_desc(args.workload, inp, w),
                              recurrence={"context_parallel_segments": n_seg, "v_slice_width": slice_w,
                                          "cp_arg": args.cp}),
               "roofline": roofs[0], "roofline_other_kernel": roofs[1],
               "path_roofline": {"achieved": path_gbs, "frac": path_gbs / peak, "unit": "GB/s",
                                 "peak": peak, "algorithmic_bytes_per_step": abytes,
                                 "traffic": path_traffic,
                                 "traffic_over_algorithmic": (path_traffic / abytes) if path_traffic else None,
                                 "ms_prep": ms_prep, "ms_recurrence": ms_rec,
                                 "split": "per-kernel times from a second run of the same steps with an "
                                          "event between the kernels"},
               "gpu_launches": kernels_per_step * args.steps,
               "wall_s_timed_region": wall, "clocks": clk}
        if e2e is not None:
            out["e2e"] = e2e
        if not args.no_cpu_baseline:
            cb = cpu_baseline(inp)
            cb.pop("seconds", None)
            out["cpu_baseline"] = cb
        print(json.dumps(out), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()


def run_e2e(args, inp, dev, kda, o, fs, wsb, cp=None):
    """The same metric through the public API with host buffers: every step copies all of its inputs
    from pinned host memory to the device and o and final_state back, inside the timed region.

    The steps are pipelined as a server would run them: inputs and outputs are double-buffered on
    the device and three streams carry the host-to-device copies, the forward and the
    device-to-host copies, so that step i's forward overlaps the copies of its neighbours. The
    same steps run back to back on one stream are reported as ``serial_ms_per_step``."""
    import torch
    host = {k: (v.pin_memory() if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}
    dbufs = [{k: (torch.empty_like(v, device=dev) if isinstance(v, torch.Tensor) else v)
              for k, v in host.items()} for _ in range(2)]
    outs = [(o, fs), (torch.empty_like(o), torch.empty_like(fs))]
    o_h = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for _ in range(2)]
    fs_h = [torch.empty(fs.shape, dtype=fs.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(v.numel() * v.element_size() for v in host.values() if isinstance(v, torch.Tensor))
    d2h = o.numel() * o.element_size() + fs.numel() * fs.element_size()
    steps = max(3, min(args.steps, 10))
    s_in, s_fwd, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_fwd = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def fwd(b):
        d = dbufs[b]
        kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                d["scale"], d["initial_state"], True, d["cu_seqlens"], workspace=wsb, out=outs[b][0],
                final_state=outs[b][1], context_parallel=cp)

    def step(i, serial):
        b = 0 if serial else i & 1
        cin, cfwd, cout = (s_fwd, s_fwd, s_fwd) if serial else (s_in, s_fwd, s_out)
        with torch.cuda.stream(cin):
            if i >= 2 and not serial:
                cin.wait_event(ev_fwd[b])          # the forward of step i - 2 has read buffer b
            for k, v in host.items():
                if isinstance(v, torch.Tensor):
                    dbufs[b][k].copy_(v, non_blocking=True)
            ev_in[b].record(cin)
        with torch.cuda.stream(cfwd):
            cfwd.wait_event(ev_in[b])
            if i >= 2 and not serial:
                cfwd.wait_event(ev_out[b])         # the outputs of step i - 2 were copied out
            fwd(b)
            ev_fwd[b].record(cfwd)
        with torch.cuda.stream(cout):
            cout.wait_event(ev_fwd[b])
            o_h[b].copy_(outs[b][0], non_blocking=True)
            fs_h[b].copy_(outs[b][1], non_blocking=True)
            ev_out[b].record(cout)

    def timed(serial):
        for i in range(2):
            step(i, serial)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(s_in if not serial else s_fwd)
        for s_ in (s_fwd, s_out):
            s_.wait_event(e0)
        for i in range(steps):
            step(i, serial)
        for s_ in (s_in, s_fwd):
            s_out.wait_stream(s_)
        e1.record(s_out)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps

    serial_ms = timed(True)
    ms = timed(False)
    return {"value": tokens_of(inp) / (ms * 1e-3), "unit": UNIT, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "pipelining": "double-buffered device inputs and outputs; host-to-device copies, forward and "
                          "device-to-host copies on three streams, so that consecutive steps overlap",
            "serial_ms_per_step": serial_ms}


def main():
    args = parse()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
