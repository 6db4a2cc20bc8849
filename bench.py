#!/usr/bin/env python
"""Benchmark of the FP8 mixed-precision optimizer hot path on GB300.

One step = one pass of the whole path over one batch of synthetic gradients:
``fp8_cast_adamw_step``, i.e. the scaled cast of the BF16 gradient list to
E4M3 (per-tensor just-in-time scale) and the AdamW step (E4M3 first moment,
FP16 second moment, FP16 weights, GradScaler inf/NaN check) in one call.  Default workload: the
6.7B-parameter long-tail list (32 layers, d 4096, ffn 16384, vocab 50304, plus
200 tiny tensors and one all-zero tensor; 589 tensors, 6,658,707,493 params).

Prints one JSON line.  ``value`` is whole-job Gparams/s with inputs resident
in HBM (CUDA events on the launching stream); ``e2e`` is the same metric when
every step also copies its gradients from pinned host memory (double-buffered:
the next step's copy overlaps this step's kernels) and reads found_inf back;
``roofline`` covers the dominant kernel (the fused AdamW
update), timed live with the library's per-kernel events; ``cpu_baseline`` is
the scalar C oracle on a bounded sample of the same workload.

``--impl reference`` times the oracle (the plain CPU implementation) instead.
Under torchrun each rank steps its own copy of the workload (independent
problems, weak scaling, no data-path collective); rank 0 prints.
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

METRIC = ("FP8-state AdamW step Gparams/s and HBM GB/s (% of GB300 peak); "
          "FP8 cast GB/s")
UNIT = "Gparams/s"
# algorithmic HBM bytes per parameter of one step (BF16 gradients in), with
# the cast fused into the step (fp8_cast_adamw_step):
#   gradient amax: read 2
#   encode + the step's first pass: read 2 (BF16) + 1 (m), write 1 (codes)
#   update: read g, m, v, w = 6, write m, v, w = 5
#   O3 adds the weight copy: master read 2, codes write 1 = 3
STEP_BYTES = {"O2": 17, "O3": 20}
UPDATE_BYTES = 11          # the dominant kernel, per parameter


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="o2_6p7b_tail",
                   choices=["o2_6p7b_tail", "o3_1p3b", "o2_350m", "tiny"])
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--no-other-configs", action="store_true",
                   help="skip the cast (124M), O2 350M, O3 1.3B and tiny lines")
    p.add_argument("--n-layer", type=int, default=None,
                   help="override the workload's layer count (profiling cases)")
    p.add_argument("--vocab", type=int, default=None,
                   help="override the workload's vocabulary (profiling cases)")
    p.add_argument("--grad-fmt", default=None, choices=["e4m3", "e5m2"],
                   help="override the workload's gradient code format "
                        "(profiling case)")
    p.add_argument("--max-grad-norm", type=float, default=None,
                   help="clip the headline step to this global gradient norm "
                        "(fp8_cast_adam_step_clipped; profiling case)")
    p.add_argument("--unfused", action="store_true",
                   help="run the headline as two calls (the cast, then the "
                        "step; profiling case)")
    p.add_argument("--sharded", action="store_true",
                   help="under torchrun: the ZeRO-1 sharded data-parallel step "
                        "(each rank casts its own gradients of every tensor, "
                        "FP8 all-to-all, FP8 mean, owners step their tensors, "
                        "weights broadcast) instead of independent replicas")
    p.add_argument("--reduce-only", type=int, default=None, metavar="K",
                   help="time only the local FP8 reduction of K shards of the "
                        "124M list and print its line (profiling case)")
    p.add_argument("--record-traffic", default=None, metavar="CSV",
                   help="write the step_update DRAM traffic record from an ncu "
                        "raw-page CSV of a capture of this workload (no GPU "
                        "needed), then exit")
    p.add_argument("--capture-command", default="",
                   help="with --record-traffic: the command the capture ran")
    p.add_argument("--cast-only", default=None, choices=["e4m3", "e5m2"],
                   help="time only the scaled cast of the 124M list to this "
                        "format and print its line (profiling case)")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def workload_desc(wl):
    return {
        "workload": wl.name,
        "tensors": len(wl.shapes),
        "params": wl.n_params,
        "level": wl.level,
        "grad_dtype": str(wl.grad_dtype).replace("torch.", ""),
        "grad_fmt": wl.grad_fmt,
        "step": (f"fp8_cast_adamw_step ({str(wl.grad_dtype).replace('torch.', '')} "
                 f"grads -> {wl.grad_fmt.upper()}, then the AdamW step)"),
        "bytes_per_param": STEP_BYTES[wl.level],
        "l2": "inputs larger than L2 (no flush needed)" if wl.n_params > 1e8
              else "inputs smaller than L2",
    }


# ------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def _once(self):
        try:
            out = subprocess.run(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev)], capture_output=True, text=True, timeout=20)
            return out.stdout.strip().splitlines()
        except Exception:
            return []

    def start(self):
        self.lines += self._once()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=10)
            except Exception:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines += out.strip().splitlines()
        self.lines += self._once()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for name, val in zip(names, f[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"],
                    "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ oracle leg

def oracle_sample(wl, budget_s: float, parts: int = 1):
    """A bounded sample of ``wl`` as (tensor, elements) entries: small tensors
    first (the tail, norms, biases), then whole matrices, while the estimated
    oracle time (about 5 M params/s for cast + step) stays within budget_s.
    For a sample split over ``parts`` processes no entry is larger than one
    process's share: what budget is left then takes the leading share of the
    next larger tensors, each entry a tensor of its own."""
    order = sorted(range(len(wl.shapes)), key=lambda i: wl.numels[i])
    limit = max(1, int(budget_s * 5e6))
    cap = max(1, limit // parts)
    chosen, total = [], 0
    for i in order:
        n = wl.numels[i]
        if (total + n > limit or n > cap) and chosen:
            continue
        chosen.append((i, n))
        total += n
    if parts > 1:
        taken = {i for i, _ in chosen}
        for i in order:
            if total + cap > limit:
                break
            if i not in taken and wl.numels[i] > cap:
                chosen.append((i, cap))
                total += cap
    return sorted(chosen), total


def _oracle_states(wl, entries):
    """Fresh oracle optimizer state (m = v = 0, the workload's weights) for
    the sample's entries."""
    import numpy as np
    import torch
    import oracle
    fmt = oracle.FMT[wl.grad_fmt]
    states = []
    for i, n in entries:
        w = wl.weight(i).reshape(-1)[:n].contiguous()
        w = w.view(torch.int16).numpy().view(np.uint16)
        states.append(oracle.StepState(np.zeros(n, np.uint8), 1.0,
                                       np.zeros(n, np.uint8), 1.0,
                                       np.zeros(n, np.uint16), w, g_fmt=fmt,
                                       o3=wl.level == "O3"))
    return states


def _oracle_grads(wl, entries, step):
    """The gradients of the sample's entries at ``step`` as the oracle's raw
    arrays."""
    import numpy as np
    import torch
    out = []
    for i, n in entries:
        g = wl.grad(i, step).reshape(-1)[:n].contiguous()
        out.append(g.numpy() if g.dtype == torch.float32 else
                   g.view(torch.int16).numpy().view(np.uint16))
    return out


def _oracle_cast_step(wl, states, srcs, step):
    """One oracle cast + AdamW step of the given tensors (timed work)."""
    import torch
    import oracle
    fmt = oracle.FMT[wl.grad_fmt]
    dt = {torch.float32: oracle.F32, torch.bfloat16: oracle.BF16,
          torch.float16: oracle.F16}[wl.grad_dtype]
    for st, src in zip(states, srcs):
        c, _, sc = oracle.cast_scaled(src, dt, fmt)
        st.g, st.g_scale = c, float(sc)
    oracle.adamw_step(states, wl.lr, wl.beta1, wl.beta2, wl.eps, wl.wd, step,
                      wl.inv_loss_scale)


def oracle_step_time(wl, entries, step):
    """Wall time of one oracle cast + step over the entries (single thread)."""
    states = _oracle_states(wl, entries)
    srcs = _oracle_grads(wl, entries, step)
    t0 = time.perf_counter()
    _oracle_cast_step(wl, states, srcs, step)
    return time.perf_counter() - t0


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _split_by_size(entries, parts: int):
    """The entries dealt to ``parts`` lists, largest first onto the lightest."""
    lists = [[] for _ in range(parts)]
    load = [0] * parts
    for e in sorted(entries, key=lambda e: -e[1]):
        r = load.index(min(load))
        lists[r].append(e)
        load[r] += e[1]
    return [sorted(x) for x in lists if x]


def _oracle_worker(wl, entries, steps, barrier, out):
    """One process of the parallel oracle: its own entries and state, kept
    across steps.  The gradients of step 1 are made once, before the first
    common start, and serve every step (the oracle's work per element does
    not depend on their values)."""
    import torch
    torch.set_num_threads(1)
    states = _oracle_states(wl, entries)
    srcs = _oracle_grads(wl, entries, 1)
    for k in range(steps):
        barrier.wait()
        t0 = time.perf_counter()
        _oracle_cast_step(wl, states, srcs, k + 1)
        out.put((k, t0, time.perf_counter()))
    barrier.wait()


def oracle_parallel_times(wl, entries, steps: int, procs: int):
    """Wall time of each of ``steps`` oracle cast + steps over the entries,
    split over ``procs`` spawned processes that start each step together: the
    step ends when the last process does.  Tensors are independent apart from
    found_inf, which no timed workload sets, so the results equal one
    process's."""
    import multiprocessing as mp
    import queue
    ctx = mp.get_context("spawn")
    parts = _split_by_size(entries, procs)
    barrier = ctx.Barrier(len(parts))
    out = ctx.Queue()
    ps = [ctx.Process(target=_oracle_worker, args=(wl, part, steps, barrier, out),
                      daemon=True) for part in parts]
    for p in ps:
        p.start()
    t0 = [math.inf] * steps
    t1 = [0.0] * steps
    try:
        got = 0
        while got < steps * len(parts):
            try:
                k, a, b = out.get(timeout=1.0)
            except queue.Empty:
                dead = [p.exitcode for p in ps if p.exitcode not in (None, 0)]
                if dead:
                    raise RuntimeError(f"oracle process exited with {dead[0]}")
                continue
            t0[k] = min(t0[k], a)
            t1[k] = max(t1[k], b)
            got += 1
    finally:
        for p in ps:
            p.join(timeout=60)
            if p.is_alive():
                p.terminate()
    return [b - a for a, b in zip(t0, t1)], len(parts)


def _describe(wl, entries, total):
    whole = sum(1 for i, n in entries if n == wl.numels[i])
    return (f"{len(entries)} tensors of {len(wl.shapes)}: {whole} whole, "
            f"{len(entries) - whole} leading slices ({total} params)")


def cpu_baseline(wl, budget_s: float):
    """The oracle on the host cores: one process on a sample of about
    budget_s / 2 of single-thread work, then every core on a sample that
    many times larger."""
    e1, total1 = oracle_sample(wl, budget_s / 2)
    secs1 = oracle_step_time(wl, e1, 1)
    cores = host_cores()
    entries, total = oracle_sample(wl, budget_s / 2 * cores, cores)
    times, used = oracle_parallel_times(wl, entries, 1, cores)
    secs = times[0]
    import platform
    return {"value": total / secs / 1e9, "unit": UNIT, "cores": used,
            "kind": "oracle", "machine": platform.machine(),
            "sample": f"1 cast+step over {_describe(wl, entries, total)}, "
                      f"{secs:.1f} s, split by tensor over {used} processes",
            "single_thread": {"value": total1 / secs1 / 1e9, "unit": UNIT,
                              "cores": 1,
                              "sample": f"1 cast+step over "
                                        f"{_describe(wl, e1, total1)}, "
                                        f"{secs1:.1f} s"}}


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    cores = host_cores()
    per_step = max(1.0, 90.0 / max(1, args.steps + args.warmup))
    entries, total = oracle_sample(wl, per_step * cores, cores)
    times, used = oracle_parallel_times(wl, entries, args.warmup + args.steps,
                                        cores)
    secs = sum(times[args.warmup:])
    value = total * args.steps / secs / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * secs / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_desc(wl),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": used,
                         "kind": "oracle", "machine": __import__("platform").machine(),
                         "sample": f"each step: cast+step over "
                                   f"{_describe(wl, entries, total)}, split by "
                                   f"tensor over {used} processes, the step-1 "
                                   f"gradients in every step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- GPU leg

def build_state(wl, device, **opt_kw):
    import torch
    import bit_optimizer_gb300 as bo
    numels = wl.numels
    params = bo.arena_views(numels, torch.float16, device)
    for i, p in enumerate(params):
        p.copy_(wl.weight(i, device))
    grads, flat = bo.arena_views(numels, wl.grad_dtype, device, return_base=True)
    for i, g in enumerate(grads):
        g.copy_(wl.grad(i, 1, device))
    torch.cuda.synchronize()
    opt = bo.Fp8AdamW(params, lr=wl.lr, betas=(wl.beta1, wl.beta2), eps=wl.eps,
                      weight_decay=wl.wd, level=wl.level, grad_fmt=wl.grad_fmt,
                      **opt_kw)
    return params, grads, flat, opt


# the update kernel and the host code that sizes its grid and chunk table
KERNEL_SOURCES = ("bit_optimizer_gb300/csrc/step_kernels.cu",
                  "bit_optimizer_gb300/csrc/fp8opt_internal.cuh",
                  "bit_optimizer_gb300/csrc/api.cu")
# written by --record-traffic from an ncu capture of step_update
TRAFFIC_RECORD = "profiles/step_update_traffic.json"


def kernel_source_digest():
    """First 16 hex digits of sha256 over the kernel sources with their
    comments and whitespace removed: a comment edit leaves the kernels, and
    so the recorded traffic, unchanged.  (The sources have no comment
    markers inside string literals.)"""
    import hashlib
    import re
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def update_traffic_per_param():
    """DRAM bytes per parameter of one step_update launch from the recorded
    ncu capture, or None when there is none or the kernel source changed
    since it was taken."""
    try:
        with open(os.path.join(ROOT, TRAFFIC_RECORD)) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_digest") != kernel_source_digest():
        return None
    try:
        return float(rec["traffic_bytes_per_param"])
    except (KeyError, TypeError, ValueError):
        return None


NCU_UNITS = {"byte": 1, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9, "Tbyte": 1e12,
             "KB": 1e3, "MB": 1e6, "GB": 1e9, "nsecond": 1e-9, "usecond": 1e-6,
             "msecond": 1e-3, "second": 1.0, "ns": 1e-9, "us": 1e-6,
             "ms": 1e-3}


def ncu_launches(csv_path, kernel="step_update"):
    """The launches of `kernel` in an ncu raw-page CSV (ncu -i REP --page raw
    --csv): per launch, DRAM bytes read and written and the duration in
    seconds, converted from the units row."""
    import csv
    with open(csv_path, newline="") as f:
        rows = [r for r in csv.reader(f) if r]
    head = next(i for i, r in enumerate(rows) if "Kernel Name" in r)
    names, units = rows[head], rows[head + 1]
    col = {n: i for i, n in enumerate(names)}

    def value(r, metric):
        i = col[metric]
        return float(r[i].replace(",", "")) * NCU_UNITS.get(units[i], 1.0)

    out = []
    for r in rows[head + 2:]:
        if len(r) == len(names) and kernel in r[col["Kernel Name"]]:
            out.append({"dram_read": value(r, "dram__bytes_read.sum"),
                        "dram_write": value(r, "dram__bytes_write.sum"),
                        "seconds": value(r, "gpu__time_duration.sum")})
    return out


def record_traffic(csv_path, wl, command):
    """Writes TRAFFIC_RECORD from an ncu capture of step_update on workload
    wl: DRAM bytes (read + write) per launch over wl's parameters, with the
    current source digest."""
    launches = ncu_launches(csv_path)
    if not launches:
        raise SystemExit(f"no step_update launch in {csv_path}")
    rd = sum(x["dram_read"] for x in launches) / len(launches)
    wr = sum(x["dram_write"] for x in launches) / len(launches)
    us = sum(x["seconds"] for x in launches) / len(launches) * 1e6
    rec = {"kernel": "step_update", "workload": wl.name, "params": wl.n_params,
           "launches": len(launches), "dram_bytes_read": rd,
           "dram_bytes_write": wr, "duration_us": us,
           "traffic_bytes_per_param": round((rd + wr) / wl.n_params, 4),
           "algorithmic_bytes_per_param": UPDATE_BYTES,
           "source_digest": kernel_source_digest(), "command": command}
    with open(os.path.join(ROOT, TRAFFIC_RECORD), "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


# ------------------------------------------------------------- host side

def device_host_numa_node(device_index):
    """The host NUMA node closest to the GPU (cudaDevAttrHostNumaId), or
    None when the runtime cannot say."""
    import ctypes
    for name in ("libcudart.so.13", "libcudart.so.12", "libcudart.so"):
        try:
            rt = ctypes.CDLL(name)
            break
        except OSError:
            continue
    else:
        return None
    v = ctypes.c_int(-1)
    if rt.cudaDeviceGetAttribute(ctypes.byref(v), 134, device_index) != 0:
        return None
    return v.value if v.value >= 0 else None


def node_cpus(node):
    """CPUs of a NUMA node that this process may run on (empty if unknown)."""
    try:
        with open(f"/sys/devices/system/node/node{node}/cpulist") as f:
            text = f.read().strip()
    except OSError:
        return set()
    cpus = set()
    for part in filter(None, text.split(",")):
        a, _, b = part.partition("-")
        cpus.update(range(int(a), int(b or a) + 1))
    return cpus & os.sched_getaffinity(0)


def pinned_on_node(shape, dtype, node):
    """A pinned host tensor allocated while this process runs on the CPUs of
    NUMA node `node` (the default memory policy then places its pages
    there), and the pages per node it actually got."""
    import torch
    cpus = node_cpus(node) if node is not None else set()
    saved = os.sched_getaffinity(0)
    if cpus:
        os.sched_setaffinity(0, cpus)
    try:
        t = torch.empty(shape, dtype=dtype, pin_memory=True)
        t.view(torch.uint8).zero_()               # touch every page
    finally:
        os.sched_setaffinity(0, saved)
    return t, pages_by_node(t.data_ptr())


def pages_by_node(addr):
    """{node: pages} of the mapping that holds `addr`, from
    /proc/self/maps and /proc/self/numa_maps (None if unreadable)."""
    try:
        with open("/proc/self/maps") as f:
            start = next(int(a, 16) for a, b in
                         (ln.split()[0].split("-") for ln in f)
                         if int(a, 16) <= addr < int(b, 16))
        with open("/proc/self/numa_maps") as f:
            for ln in f:
                fields = ln.split()
                if int(fields[0], 16) == start:
                    return {int(k[1:]): int(v) for k, v in
                            (x.split("=", 1) for x in fields[2:] if "=" in x)
                            if k.startswith("N") and k[1:].isdigit()}
    except (OSError, StopIteration, ValueError):
        return None
    return None


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def _events_ms(fn, reps):
    """Average device milliseconds of fn() over reps calls (CUDA events on
    the current stream, synchronised on both sides)."""
    import torch
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    torch.cuda.synchronize()
    return a.elapsed_time(b) / reps


def cast_configs(device, peak, fmts=("e4m3", "e5m2")):
    """The scaled cast of the 124M GPT-2 list (BF16 in, per-tensor
    just-in-time scale): amax pass 2 B + encode pass 3 B per element."""
    import torch
    import synth
    import bit_optimizer_gb300 as bo
    out = {}
    wl = synth.gpt2_cast()
    srcs = bo.arena_views(wl.numels, torch.bfloat16, device)
    for i, x in enumerate(srcs):
        x.copy_(wl.grad(i, 1, device))
    codes = bo.arena_views(wl.numels, torch.uint8, device)
    amax = torch.empty(len(srcs), device=device)
    scale = torch.empty(len(srcs), device=device)
    for fmt in fmts:
        plan = bo.CastPlan(srcs, codes, amax, scale, fmt)
        for _ in range(3):
            plan()
        ms = _events_ms(plan, 20)
        gbs = 5 * wl.n_params / (ms * 1e-3) / 1e9
        out[f"cast_gpt2_124m_{fmt}"] = {"ms": ms, "GB/s": gbs, "frac": gbs / peak,
                                        "bytes_per_elem": 5}
    del srcs, codes
    torch.cuda.empty_cache()
    return out


def reduce_configs(device, peak, ranks=(2, 8)):
    """The local FP8 reduction on the 124M GPT-2 list: k shards per tensor
    (each rank's BF16 gradient cast to E4M3 by the library, rows of a
    [k, numel] buffer with 16-byte row stride), reduced to their mean in E4M3;
    2k + 1 bytes per element.  Each k is timed plain and with the norm terms
    of its outputs."""
    import torch
    import synth
    import bit_optimizer_gb300 as bo
    out = {}
    for k in ranks:
        wl = synth.fp8_reduce(ranks=k)
        n_t = len(wl.shapes)
        shards = [torch.empty((k, (n + 15) // 16 * 16), dtype=torch.uint8,
                              device=device)[:, :n] for n in wl.numels]
        scales = torch.empty((n_t, k), device=device)
        amax = torch.empty(n_t, device=device)
        for r in range(k):
            grads = [wl.rank_grad(i, 1, r, device) for i in range(n_t)]
            rs = torch.empty(n_t, device=device)
            bo.CastPlan(grads, [sh[r] for sh in shards], amax, rs, "e4m3")()
            scales[:, r] = rs
            del grads
        codes = bo.arena_views(wl.numels, torch.uint8, device)
        scale = torch.empty(n_t, device=device)
        plan = bo.ReducePlan(shards, scales, codes, amax, scale, "e4m3", "e4m3",
                             1.0 / k)
        for _ in range(3):
            plan()
        ms = _events_ms(plan, 20)
        bpe = 2 * k + 1
        gbs = bpe * wl.n_params / (ms * 1e-3) / 1e9
        out[f"reduce_gpt2_124m_k{k}"] = {"ms": ms, "GB/s": gbs, "frac": gbs / peak,
                                         "bytes_per_elem": bpe, "shards": k}
        # the same with the norm terms of the outputs (the sharded clipped
        # step's reduction): the exact squares ride in the encode pass
        terms = torch.empty(n_t, dtype=torch.float64, device=device)
        found = torch.zeros(1, dtype=torch.int32, device=device)

        def with_norm():
            plan(norm_terms=terms, found=found, inv_loss_scale=1.0)
        for _ in range(3):
            with_norm()
        ms = _events_ms(with_norm, 20)
        gbs = bpe * wl.n_params / (ms * 1e-3) / 1e9
        out[f"reduce_gpt2_124m_k{k}_norm"] = {"ms": ms, "GB/s": gbs,
                                              "frac": gbs / peak,
                                              "bytes_per_elem": bpe, "shards": k}
        del shards, codes
        torch.cuda.empty_cache()
    return out


def other_configs(device, peak):
    """The remaining workloads, each timed on its own after the headline:
    the scaled cast of the 124M GPT-2 list (BF16 -> E4M3 and -> E5M2, 5 B per
    element), the local FP8 reduction of 2 and 8 shards of that list, the O2
    step on the 350M list (the inf cleared; E4M3 and E5M2 gradients), the O3 step on
    the 1.3B list (20 B per param with the cast), the same with the scaled
    second moment, Adam with L2 decay on the 350M list, the 350M step clipped
    to a global gradient norm (and the norm pass alone), and the launch-bound
    tiny list, also as replays of a captured graph of the capturable step."""
    import dataclasses
    import torch
    import synth
    import bit_optimizer_gb300 as bo
    out = cast_configs(device, peak)
    out.update(reduce_configs(device, peak))
    # (name, workload, reps, optimizer options, algorithmic bytes per param)
    runs = (
        ("o2_350m", synth.o2_350m, 20, {}, STEP_BYTES["O2"]),
        # the same list with E5M2 gradient codes
        ("o2_350m_e5m2", synth.o2_350m, 20, {"grad_fmt": "e5m2"}, STEP_BYTES["O2"]),
        ("o3_1p3b", synth.o3_1p3b, 10, {}, STEP_BYTES["O3"]),
        ("o3_1p3b_scaled_v", synth.o3_1p3b, 10, {"scaled_v": True},
         STEP_BYTES["O3"]),
        # Adam with L2 decay: its first pass also reads w; amax 2, the fused
        # encode and first pass 2 + 1 + 2 + 1, update 11
        ("o2_350m_adam_l2", synth.o2_350m, 20, {"l2": True}, 19),
        # clipping to a global norm, one call: gradient amax 2, encode with
        # the exact squares 3, first pass 2, update 11
        ("o2_350m_clip", synth.o2_350m, 20, {"max_grad_norm": 1.0}, 18),
        ("tiny", synth.tiny, 200, {}, STEP_BYTES["O2"]),
    )
    for name, mk, reps, kw, bpp in runs:
        w = dataclasses.replace(mk(), inf_site=None)
        if "grad_fmt" in kw:
            w = dataclasses.replace(w, grad_fmt=kw["grad_fmt"])
        params, grads, _, opt = build_state(
            w, device, **{k: v for k, v in kw.items() if k != "grad_fmt"})
        flag = torch.zeros(1, dtype=torch.int32, device=device)
        fn = lambda: opt.step(grads, w.inv_loss_scale, found_inf_dev=flag, sync=False)
        for _ in range(3):
            fn()
        ms = _events_ms(fn, reps)
        gbs = bpp * w.n_params / (ms * 1e-3) / 1e9
        out[name] = {"ms_per_step": ms, "Gparams/s": w.n_params / (ms * 1e-3) / 1e9,
                     "GB/s": gbs, "frac": gbs / peak, "level": w.level,
                     "params": w.n_params, "bytes_per_param": bpp, **kw}
        if "max_grad_norm" in kw:
            # the norm alone: one byte per parameter (plus its finalisation)
            nd = torch.zeros(1, device=device)
            fn = lambda: opt._plan.grad_norm(w.inv_loss_scale, norm_dev=nd,
                                             sync=False)
            for _ in range(3):
                fn()
            ms = _events_ms(fn, reps)
            gbs = w.n_params / (ms * 1e-3) / 1e9
            out["grad_norm_350m"] = {"ms": ms, "GB/s": gbs, "frac": gbs / peak,
                                     "bytes_per_param": 1}
        del params, grads, opt
        torch.cuda.empty_cache()
    out["tiny_graph"] = tiny_graph(device, peak)
    return out


def tiny_graph(device, peak):
    """The tiny list's fused step as one replay of a captured CUDA graph:
    the capturable optimizer reads lr, inv_loss_scale and the step count on
    the device, so each replay is a real next step.  Shows the launch and
    call overhead a graph removes from a launch-bound step."""
    import dataclasses
    import torch
    import synth
    import bit_optimizer_gb300 as bo
    w = dataclasses.replace(synth.tiny(), inf_site=None)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        params, grads, _, opt = build_state(w, device, capturable=True)
        flag = torch.zeros(1, dtype=torch.int32, device=device)
        for _ in range(3):
            opt.step(grads, found_inf_dev=flag, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        opt.step(grads, found_inf_dev=flag, stream=s)
    for _ in range(3):
        g.replay()
    reps = 500
    before = int(opt.state.step.item())
    ms = _events_ms(g.replay, reps)
    steps = int(opt.state.step.item()) - before
    gbs = STEP_BYTES["O2"] * w.n_params / (ms * 1e-3) / 1e9
    res = {"ms_per_step": ms, "Gparams/s": w.n_params / (ms * 1e-3) / 1e9,
           "GB/s": gbs, "frac": gbs / peak, "level": w.level,
           "params": w.n_params, "bytes_per_param": STEP_BYTES["O2"],
           "steps_counted": steps, "capturable": True}
    del g
    torch.cuda.synchronize()
    bo.release_stream(s)
    return res


def run_ours(args, wl):
    import torch
    import torch.distributed as dist
    import bit_optimizer_gb300 as bo

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=device)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    clip_kw = ({} if args.max_grad_norm is None
               else {"max_grad_norm": args.max_grad_norm})
    params, grads, flat, opt = build_state(wl, device, fused=not args.unfused,
                                           **clip_kw)
    stream = torch.cuda.current_stream()
    flag = torch.zeros(1, dtype=torch.int32, device=device)
    ils = wl.inv_loss_scale

    for _ in range(args.warmup):
        opt.step(grads, ils, found_inf_dev=flag, sync=False)
    barrier()

    sampler = ClockSampler(local)
    sampler.start()
    bo.timing_enable(True)
    barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for _ in range(args.steps):
        opt.step(grads, ils, found_inf_dev=flag, sync=False)
    t1.record(stream)
    barrier()
    bo.timing_enable(False)
    sampler.stop()
    ms = t0.elapsed_time(t1) / args.steps
    if int(flag.item()) != 0:
        raise RuntimeError("found_inf set on a finite workload")
    kern = {k: bo.timing_read(k) for k in bo.KERNELS}
    launches = sum(n for n, _ in kern.values())

    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())

    n_params = wl.n_params
    value = world * n_params / (ms * 1e-3) / 1e9
    # with clipping (fp8_cast_adam_step_clipped): amax 2, encode 3, first
    # pass 2, update 11 (O3: + 3); as two calls the cast (5) and the step's
    # first pass (2) are separate, plus 1 for a norm pass
    extra = (1 if clip_kw else 0) if not args.unfused else (2 if clip_kw else 1)
    bytes_step = (STEP_BYTES[wl.level] + extra) * n_params
    peak, peak_kind = measured_peak()
    upd_n, upd_ms = kern["step_update"]
    upd_avg_ms = upd_ms / max(upd_n, 1)
    achieved = UPDATE_BYTES * n_params / (upd_avg_ms * 1e-3) / 1e9
    tpp = update_traffic_per_param()

    e2e = None
    if not args.no_e2e:
        # Host buffers: every step copies its gradients from pinned host
        # memory (one copy of the flat arena, alignment padding included),
        # runs the cast and the step through the public plans, and reads
        # found_inf back to the host.  Two device gradient arenas alternate:
        # step t+1's copy (on its own stream) overlaps step t's kernels, and
        # waits only until the step that last read its arena has finished.
        numa = device_host_numa_node(local)
        host, pages = pinned_on_node(flat.shape, flat.dtype, numa)
        host.copy_(flat)
        h2d = host.numel() * host.element_size()
        # the link alone: one plain copy of the same pinned buffer into the
        # same device arena, timed with events on a side stream (best of 2)
        link_ms = None
        link_stream = torch.cuda.Stream(device)
        for _ in range(2):
            la = torch.cuda.Event(enable_timing=True)
            lb = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(link_stream):
                la.record(link_stream)
                flat.copy_(host, non_blocking=True)
                lb.record(link_stream)
            link_stream.synchronize()
            t_ms = la.elapsed_time(lb)
            link_ms = t_ms if link_ms is None else min(link_ms, t_ms)
        grads2, flat2 = bo.arena_views(wl.numels, wl.grad_dtype, device,
                                       return_base=True)
        bufs = [(grads, flat), (grads2, flat2)]
        streams = [torch.cuda.Stream(device), torch.cuda.Stream(device)]
        copy_stream = torch.cuda.Stream(device)
        fused = [bo.CastStepPlan(bo.CastPlan(g, opt.g_codes, opt.g_amax,
                                             opt.g_scale, opt.grad_fmt), opt._plan)
                 for g, _ in bufs]
        hp = (opt.lr, opt.beta1, opt.beta2, opt.eps, opt.wd)
        clip = {"max_grad_norm": opt.max_grad_norm} if clip_kw else {}

        def run(k):
            """k steps; returns their milliseconds between CUDA events (the
            first copy's start on the copy stream and the last step's end)
            and each step's copy duration on the copy stream."""
            copied = [torch.cuda.Event(), torch.cuda.Event()]
            done = [torch.cuda.Event(), torch.cuda.Event()]
            c0 = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
            c1 = [torch.cuda.Event(enable_timing=True) for _ in range(k)]
            e1 = torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(copy_stream):
                c0[0].record(copy_stream)
                bufs[0][1].copy_(host, non_blocking=True)
                c1[0].record(copy_stream)
                copied[0].record(copy_stream)
            for t in range(k):
                b, nb = t % 2, (t + 1) % 2
                if t + 1 < k:                 # the next step's gradients
                    with torch.cuda.stream(copy_stream):
                        if t >= 1:
                            copy_stream.wait_event(done[nb])
                        c0[t + 1].record(copy_stream)
                        bufs[nb][1].copy_(host, non_blocking=True)
                        c1[t + 1].record(copy_stream)
                        copied[nb].record(copy_stream)
                s = streams[b]
                s.wait_event(copied[b])
                if t >= 1:
                    s.wait_event(done[nb])    # the previous step (shared state)
                opt.step_count += 1
                found = fused[b](*hp, opt.step_count, ils, sync=True, stream=s,
                                 l2=opt.l2, **clip)
                done[b].record(s)
                if found != 0:
                    raise RuntimeError("found_inf set on a finite workload")
            e1.record(streams[(k - 1) % 2])
            torch.cuda.synchronize()
            return (c0[0].elapsed_time(e1),
                    [c0[t].elapsed_time(c1[t]) for t in range(k)])

        # warm-up: as many steps as the headline's (at least 2, so that both
        # arenas have been copied into and stepped)
        run(max(2, args.warmup))
        barrier()
        k = max(1, args.e2e_steps)
        e2e_clocks = ClockSampler(local)
        e2e_clocks.start()
        total_ms, copies_ms = run(k)
        ems = total_ms / k
        barrier()
        e2e_clocks.stop()
        if world > 1:
            t = torch.tensor([ems], dtype=torch.float64, device=device)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            ems = float(t.item())
        e2e = {"value": world * n_params / (ems * 1e-3) / 1e9, "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": 4,
               "ms_per_step": ems, "steps": k,
               # the host link measured alone in this run, and the bound it
               # sets: the copy plus the device step (the overlapped loop
               # can only approach the larger of the two)
               "link_gbs": h2d / (link_ms * 1e-3) / 1e9, "link_copy_ms": link_ms,
               "copy_plus_step_ms": link_ms + ms,
               # the same copies inside the loop: a shared host link shows
               # here as copies far slower than link_copy_ms
               "loop_copy_ms": {"median": statistics.median(copies_ms),
                                "min": min(copies_ms), "max": max(copies_ms)},
               "clocks": e2e_clocks.summary(),
               "host_buffer": {"device_host_numa_node": numa,
                               "pages_by_node": pages}}
        del host

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_seconds)
    others = None
    if rank == 0 and world == 1 and not args.no_other_configs:
        del params, grads, flat, opt
        torch.cuda.empty_cache()
        try:
            others = other_configs(device, peak)
        except Exception as e:   # the headline line is printed regardless
            others = {"error": f"{type(e).__name__}: {e}"[:300]}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic", "config": workload_desc(wl),
            "hbm_gbs": world * bytes_step / (ms * 1e-3) / 1e9,
            "hbm_frac_of_peak": bytes_step / (ms * 1e-3) / 1e9 / peak,
            "roofline": {"bound": "hbm", "kernel": "step_update",
                         "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak,
                         "traffic": (None if tpp is None else tpp * n_params),
                         "peak_source": f"{peak_kind} hbm_gbs",
                         "bytes_per_launch": UPDATE_BYTES * n_params,
                         "avg_launch_ms": upd_avg_ms},
            "kernels_ms_per_launch": {k: (v[1] / v[0] if v[0] else None)
                                      for k, v in kern.items()},
            "gpu_launches": launches,
            "clocks": sampler.summary(),
            "e2e": e2e,
            "cpu_baseline": cpu,
            "other_configs": others,
        }
        if clip_kw or args.unfused:
            line["config"]["step"] = (
                ("fp8_cast_scaled, then " if args.unfused else "") +
                ("fp8_adam_step_clipped" if args.unfused else
                 "fp8_cast_adam_step_clipped" if clip_kw else "fp8_adamw_step") +
                (f" (global norm {args.max_grad_norm})" if clip_kw else ""))
            line["config"]["bytes_per_param"] = bytes_step // n_params
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_sharded(args, wl):
    """The data-parallel step of one model over the ranks of a torchrun job
    (NCCL): every rank holds its own BF16 gradients of every tensor; one step
    casts them, sends each tensor's codes to its owner, reduces the ranks'
    shards to their mean, steps the owned tensors and broadcasts the new
    weights.  value = the model's parameters stepped per second (the model is
    fixed: strong scaling)."""
    import torch
    import torch.distributed as dist
    import bit_optimizer_gb300 as bo
    from bit_optimizer_gb300.sharded import ShardedFp8AdamW, TorchDistComm

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist.init_process_group("nccl", device_id=device)
    weights = [wl.weight(i, device) for i in range(len(wl.shapes))]
    opt = ShardedFp8AdamW(weights, TorchDistComm(), lr=wl.lr,
                          betas=(wl.beta1, wl.beta2), eps=wl.eps,
                          weight_decay=wl.wd, level=wl.level,
                          grad_fmt=wl.grad_fmt, max_grad_norm=args.max_grad_norm)
    del weights
    grads, _ = bo.arena_views(wl.numels, wl.grad_dtype, device, return_base=True)
    for i, g in enumerate(grads):
        g.copy_(wl.rank_grad(i, 1, rank, device))
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        if opt.step(grads, wl.inv_loss_scale) != 0:
            raise RuntimeError("found_inf set on a finite workload")
    dist.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for _ in range(args.steps):
        opt.step(grads, wl.inv_loss_scale)
    t1.record()
    dist.barrier()
    torch.cuda.synchronize()
    sampler.stop()
    t = torch.tensor([t0.elapsed_time(t1) / args.steps], dtype=torch.float64,
                     device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms = float(t.item())
    if rank == 0:
        desc = workload_desc(wl)
        desc["step"] = ("sharded data-parallel step: FP8 cast of each rank's "
                        "gradients, FP8 all-to-all, FP8 mean, owners' step "
                        "over equal element ranges (tensors cut across ranks), "
                        "weight all-gather (NCCL); one rank: the fused cast "
                        "and step")
        loads = [sum(b - a for _, a, b in p) for p in opt.layout_pieces]
        line = {
            "metric": METRIC, "value": wl.n_params / (ms * 1e-3) / 1e9,
            "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
            "scaling": "strong", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": desc,
            "shard_elements": {"per_rank_max": max(loads),
                               "per_rank_mean": sum(loads) / world,
                               "tensors_cut": sum(1 for t in range(len(wl.numels))
                                                  if sum(1 for p in opt.layout_pieces
                                                         for x in p if x[0] == t) > 1)},
            "clocks": sampler.summary(),
        }
        print(json.dumps(line), flush=True)
    dist.destroy_process_group()


def main():
    args = parse()
    if args.reduce_only is not None:
        import torch
        peak, _ = measured_peak()
        print(json.dumps(reduce_configs(torch.device("cuda", 0), peak,
                                        ranks=(args.reduce_only,))), flush=True)
        return
    if args.cast_only is not None:
        import torch
        peak, _ = measured_peak()
        print(json.dumps(cast_configs(torch.device("cuda", 0), peak,
                                      fmts=(args.cast_only,))), flush=True)
        return
    import dataclasses
    import synth
    over = {k: v for k, v in (("n_layer", args.n_layer), ("vocab", args.vocab))
            if v is not None}
    wl = synth.WORKLOADS[args.workload](**over)
    # a timed step must be a full update: a workload that seeds an inf (the
    # GradScaler skip case) is timed with that element cleared
    wl = dataclasses.replace(wl, inf_site=None)
    if args.grad_fmt is not None:
        wl = dataclasses.replace(wl, grad_fmt=args.grad_fmt)
    if args.record_traffic is not None:
        print(json.dumps(record_traffic(args.record_traffic, wl,
                                        args.capture_command)), flush=True)
        return
    if args.impl == "reference":
        run_reference(args, wl)
    elif args.sharded:
        run_sharded(args, wl)
    else:
        run_ours(args, wl)


if __name__ == "__main__":
    main()
